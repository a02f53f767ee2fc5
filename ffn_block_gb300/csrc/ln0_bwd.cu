// Backward of norm0 with the inverse token mix folded into its loads.
//
// Page "Subgraph-fusion-based Mega-kernel Generation", section "Exact
// computation": s1 = token_mixer(norm0(x)) + x, so with ds1 the gradient at
// s1 (norm1's backward), dx = ds1 + LN0_backward(da0), where da0 is ds1
// mixed back (the mix swaps the two T axes of [T, T, C] and is its own
// inverse): da0[j, i*C + c] = ds1[i, j*C + c].  LN0_backward is the usual
// LayerNorm backward: with xh = (x - mean) * rstd, g = gamma0 * da0,
//   out = rstd * (g - mean(g) - xh * mean(g * xh)),
//   dgamma0 += da0 * xh, dbeta0 += da0 (column partial sums).
//
// CTA (q, sample group) owns rows j = 8q ... 8q + 7 of a few consecutive
// samples.  Row j of da0 takes, from every row i of ds1, the C columns
// j*C ... j*C + C - 1, so for its eight rows the CTA stages one column stripe
// of ds1 (T rows of 8*C elements: one TMA box of a rank-2 map over ds1, the
// box a few columns wider so that its rows land an odd number of 16-byte
// units apart) next to its own rows of ds1 and x (bulk copies).  Thread v owns the 16-byte vector of columns d = v*E ... v*E + E - 1
// of all eight rows: it gathers da0[j, d] = stripe[i][(j - 8q)*C + c] with
// d = i*C + c, takes the sixteen row sums of its columns, one block reduction
// per sample gives their totals, and the column partials stay in registers
// across the samples.  Nothing token-mixed goes through HBM.  Every wait is
// bounded.

#include "common.cuh"
#include "pairs.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {
namespace {

constexpr int kRowsPerCta = 8;
// Threads per CTA at most (one per 16-byte vector of a row), chosen so that
// three CTAs of that size share an SM with the registers a thread needs.
constexpr int kLn0MaxThreads = 160;

struct Ln0GatherArgs {
  const void* ds1;     // [N, D] gradient at norm1's input
  const void* x;       // [N, D] the block's input (norm0's input)
  const float* mu;     // [N] norm0's row statistics from the forward
  const float* rs;
  const void* gamma;   // [D]
  void* dx;            // [N, D]
  float* pg;           // [P0, D] column partials of dgamma0, P0 = ceil(B/spc) * T/8
  float* pb;           // [P0, D] column partials of dbeta0
  unsigned int* err;
  int B, T, D, C, spc;
};

struct Ln0Geom {
  int piece;         // bytes of one stripe piece (8 * C * e)
  int stripe_pitch;  // piece padded to an odd number of 16-byte units (the TMA box width)
  int row_bytes;     // D * e
  size_t off_ownd, off_ownx, off_red, off_means, off_st, off_bar, smem;
};

__host__ __device__ inline size_t r16(size_t v) { return (v + 15) & ~(size_t)15; }

__host__ __device__ inline Ln0Geom ln0_geom(int Tn, int D, int esize) {
  Ln0Geom g;
  const int C = D / Tn;
  g.piece = kRowsPerCta * C * esize;
  g.stripe_pitch = (int)r16((size_t)g.piece);
  if ((g.stripe_pitch / 16) % 2 == 0) g.stripe_pitch += 16;
  g.row_bytes = D * esize;
  g.off_ownd = (size_t)Tn * g.stripe_pitch;
  g.off_ownx = g.off_ownd + (size_t)kRowsPerCta * g.row_bytes;
  g.off_red = g.off_ownx + (size_t)kRowsPerCta * g.row_bytes;
  g.off_means = g.off_red + 16 * 32 * sizeof(float);
  g.off_st = g.off_means + 16 * sizeof(float);
  g.off_bar = g.off_st + 2 * kRowsPerCta * sizeof(float2);
  g.smem = g.off_bar + 16 + 128;  // + slack to align the stripe to 128 bytes
  return g;
}

// Sums v[0..15] over the 32 lanes of a warp with sixteen shuffles.  On
// return lanes 2k and 2k + 1 hold the sum of component k (the same bits).
__device__ __forceinline__ float warp_sum16_transposed(const float (&v)[16]) {
  const int lane = threadIdx.x & 31;
  float w8[8], w4[4], w2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float keep = b4 ? v[k + 8] : v[k];
    const float send = b4 ? v[k] : v[k + 8];
    w8[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float keep = b3 ? w8[k + 4] : w8[k];
    const float send = b3 ? w8[k] : w8[k + 4];
    w4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float keep = b2 ? w4[k + 2] : w4[k];
    const float send = b2 ? w4[k] : w4[k + 2];
    w2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  float w = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
  w += __shfl_xor_sync(0xffffffffu, w, 1);
  return w;
}

// Two elements of da0 from the stripe as a float pair: one access at p0
// when PAIRS (C even, so a pair never straddles a piece and sits on a
// 2-element boundary), else one at p0 and one at p1.
template <typename T, bool PAIRS>
__device__ __forceinline__ float2 lds_gather2(const unsigned char* p0, const unsigned char* p1) {
  if (PAIRS) {
    if constexpr (sizeof(T) == 2) return unpack2w<T>(*reinterpret_cast<const uint32_t*>(p0));
    else return *reinterpret_cast<const float2*>(p0);
  }
  return make_float2(to_f(*reinterpret_cast<const T*>(p0)), to_f(*reinterpret_cast<const T*>(p1)));
}

// Shared memory: stripe [T][pitch] | own ds1 rows [8][D] | own x rows [8][D]
// | red [16][32] float | means [16] float | row statistics [2][8] float2
// (rstd, -mean * rstd; by sample parity) | two mbarriers (stripe, own rows).
// Both passes gather da0 from the stripe, so the next sample's copies are
// issued once the second pass is done.
template <typename T, bool PAIRS>
__global__ void __launch_bounds__(kLn0MaxThreads, 3)
    k_ln0_bwd_gather(const __grid_constant__ CUtensorMap stripe_map, const Ln0GatherArgs a) {
  pdl_enter();
  constexpr int E = VecN<T>::value;
  constexpr int es = (int)sizeof(T);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int Tn = a.T, D = a.D, C = a.C;
  const Ln0Geom geo = ln0_geom(Tn, D, es);
  const int j0 = blockIdx.x * kRowsPerCta;
  const int bbeg = blockIdx.y * a.spc;
  const int ns = min(a.B, bbeg + a.spc) - bbeg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int c0 = tid * E;
  const bool active = c0 < D;

  unsigned char* stripe = smem;
  unsigned char* ownd = smem + geo.off_ownd;
  unsigned char* ownx = smem + geo.off_ownx;
  float* red = reinterpret_cast<float*>(smem + geo.off_red);
  float* means = reinterpret_cast<float*>(smem + geo.off_means);
  float2* rowst = reinterpret_cast<float2*>(smem + geo.off_st);
  // Threads 0..7 stage the norm0 statistics of sample index si's rows.
  auto load_stats = [&](int si) {
    if (tid < kRowsPerCta) {
      const size_t row = (size_t)(bbeg + si) * Tn + j0 + tid;
      const float r = a.rs[row];
      rowst[(si & 1) * kRowsPerCta + tid] = make_float2(r, -a.mu[row] * r);
    }
  };
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + geo.off_bar);  // [0] stripe, [1] own rows
  __shared__ int abort_flag;

  const T* ds1 = reinterpret_cast<const T*>(a.ds1);
  const T* xg = reinterpret_cast<const T*>(a.x);
  // Warp 0 issues a sample's copies: lane 0 arms the barrier, the lanes
  // share the copies.
  auto issue_stripe = [&](int b) {
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(&bar[0]), (uint32_t)(Tn * geo.stripe_pitch));
      tma_load_2d(smem_u32(stripe), &stripe_map, smem_u32(&bar[0]), j0 * C, b * Tn);
    }
  };
  auto issue_own = [&](int b) {
    if (lane == 0) mbar_arrive_expect_tx(smem_u32(&bar[1]), (uint32_t)(2 * kRowsPerCta * geo.row_bytes));
    __syncwarp();
    // The eight own rows are consecutive in memory: one copy per tensor.
    if (lane < 2) {
      const T* src = (lane == 0 ? ds1 : xg) + ((size_t)b * Tn + j0) * D;
      bulk_g2s(smem_u32(lane == 0 ? ownd : ownx), src, (uint32_t)(kRowsPerCta * geo.row_bytes), smem_u32(&bar[1]));
    }
  };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    fence_mbar_init();
  }
  if (ns > 0) load_stats(0);
  __syncthreads();
  if (warp == 0 && ns > 0) {
    issue_stripe(bbeg);
    issue_own(bbeg);
  }

  // Stripe byte offsets of the thread's columns (row 0 of the eight).  The
  // element math runs on column pairs with the packed fp32x2 instructions
  // (each rounds as the scalar one).
  constexpr int P = E / 2;
  constexpr int NOFF = PAIRS ? P : E;  // a pair's second element follows its first when C is even
  int soff[NOFF];
  float2 gam[P], pg[P], pb[P];
#pragma unroll
  for (int e = 0; e < NOFF; ++e) {
    const int d = min(c0 + (PAIRS ? 2 * e : e), D - 1);
    const int i = d / C;
    soff[e] = i * geo.stripe_pitch + (d - i * C) * es;
  }
  auto gather = [&](const unsigned char* sp, int k) {
    return PAIRS ? lds_gather2<T, true>(sp + soff[k], nullptr)
                 : lds_gather2<T, false>(sp + soff[2 * k], sp + soff[(2 * k + 1) % NOFF]);
  };
#pragma unroll
  for (int k = 0; k < P; ++k) pg[k] = pb[k] = f2(0.f);
  if (active) ld16p<T>(reinterpret_cast<const T*>(a.gamma) + c0, gam);

  const float invD = 1.0f / (float)D;
  const size_t piece_row = (size_t)C * es;  // stripe bytes between consecutive own rows
  int si = 0;
  bool aborted = false;
  for (; si < ns; ++si) {
    const int b = bbeg + si;
    const uint32_t ph = (uint32_t)(si & 1);
    bool ok = mbar_wait_bounded(smem_u32(&bar[0]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                (volatile int*)&abort_flag);
    ok = ok && mbar_wait_bounded(smem_u32(&bar[1]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                 (volatile int*)&abort_flag);
    // Pass 1: gather da0, g = gamma0 * da0 and the row sums (the column
    // partials wait for pass 2, after the barrier, which gathers da0 again:
    // less work before the barrier every warp waits at).
    float sums[16];
#pragma unroll
    for (int jl = 0; jl < kRowsPerCta; ++jl) {
      const float2 rc = rowst[(si & 1) * kRowsPerCta + jl];
      const float2 r = f2(rc.x), cst = f2(rc.y);
      float2 s0 = f2(0.f), s1 = f2(0.f);
      if (ok && active) {
        float2 xv[P];
        ld16p<T>(reinterpret_cast<const T*>(ownx + (size_t)jl * geo.row_bytes) + c0, xv);
        const unsigned char* sp = stripe + (size_t)jl * piece_row;
#pragma unroll
        for (int k = 0; k < P; ++k) {
          const float2 da = gather(sp, k);
          const float2 xh = fma2(xv[k], r, cst);
          const float2 gg = mul2(gam[k], da);
          s0 = add2(s0, gg);
          s1 = fma2(gg, xh, s1);
        }
      }
      sums[2 * jl] = s0.x + s0.y;
      sums[2 * jl + 1] = s1.x + s1.y;
    }
    {
      const float k = warp_sum16_transposed(sums);
      if ((lane & 1) == 0) red[(lane >> 1) * 32 + warp] = k;
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid < 16) {
      float v = 0.f;
      for (int w = 0; w < nw; ++w) v += red[tid * 32 + w];
      means[tid] = v * invD;
    }
    __syncthreads();
    // Pass 2: with xh = x * r + cst, out = r * (g - mg - xh * mgx)
    //   = r * g + (-r * r * mgx) * x + (-r * mg - r * mgx * cst); dx = out + ds1.
    if (active) {
#pragma unroll
      for (int jl = 0; jl < kRowsPerCta; ++jl) {
        const size_t row = (size_t)b * Tn + j0 + jl;
        const float2 rc = rowst[(si & 1) * kRowsPerCta + jl];
        const float r = rc.x, cst = rc.y;
        const float mg = means[2 * jl], mgx = means[2 * jl + 1];
        const float2 A = f2(-r * r * mgx), Bc = f2(-r * mg - r * mgx * cst), r2 = f2(r), c2 = f2(cst);
        float2 xv[P], dv[P], o[P];
        ld16p<T>(reinterpret_cast<const T*>(ownx + (size_t)jl * geo.row_bytes) + c0, xv);
        ld16p<T>(reinterpret_cast<const T*>(ownd + (size_t)jl * geo.row_bytes) + c0, dv);
        const unsigned char* sp = stripe + (size_t)jl * piece_row;
#pragma unroll
        for (int k = 0; k < P; ++k) {
          const float2 da = gather(sp, k);
          o[k] = add2(fma2(r2, mul2(gam[k], da), fma2(A, xv[k], Bc)), dv[k]);
          pg[k] = fma2(da, fma2(xv[k], r2, c2), pg[k]);
          pb[k] = add2(pb[k], da);
        }
        st16p<T>(reinterpret_cast<T*>(a.dx) + row * D + c0, o);
      }
    }
    // The next sample's statistics go to the other parity slot: its last
    // reader was the previous sample's second pass, before the last barrier.
    if (si + 1 < ns) load_stats(si + 1);
    __syncthreads();
    // Every thread is done with the stripe and the own rows: fetch the next
    // sample's.
    if (warp == 0 && si + 1 < ns) {
      issue_stripe(b + 1);
      issue_own(b + 1);
    }
  }

  if (aborted) {
    // Give this sample's copies (the only ones that can be in flight) a
    // bounded time to land before the CTA's shared memory goes away.
    if (tid == 0) {
      volatile int no_abort = 0;
      const uint32_t ph = (uint32_t)(si & 1);
      mbar_wait_bounded(smem_u32(&bar[0]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS, &no_abort);
      mbar_wait_bounded(smem_u32(&bar[1]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS, &no_abort);
    }
    return;
  }
  if (active) {
    const size_t p = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
#pragma unroll
    for (int k = 0; k < P; k += 2) {
      *reinterpret_cast<float4*>(a.pg + p * D + c0 + 2 * k) = make_float4(pg[k].x, pg[k].y, pg[k + 1].x, pg[k + 1].y);
      *reinterpret_cast<float4*>(a.pb + p * D + c0 + 2 * k) = make_float4(pb[k].x, pb[k].y, pb[k + 1].x, pb[k + 1].y);
    }
  }
}

template <typename T, bool PAIRS>
cudaError_t launch_typed(const Ln0GatherArgs& a, int dtype, cudaStream_t st) {
  constexpr int E = VecN<T>::value;
  constexpr int es = (int)sizeof(T);
  const Ln0Geom g = ln0_geom(a.T, a.D, es);
  // ds1 as [B*T][D]; one box = the stripe of one sample (T rows).
  CUtensorMap map;
  if (!make_tensor_map_2d(&map, a.ds1, dtype, (uint64_t)a.D, (uint64_t)a.B * a.T, (uint64_t)a.D * es,
                          (uint32_t)(g.stripe_pitch / es), (uint32_t)a.T))
    return cudaErrorInvalidValue;
  auto k = k_ln0_bwd_gather<T, PAIRS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem);
  if (e != cudaSuccess) return e;
  const int threads = (a.D / E + 31) / 32 * 32;
  const dim3 grid(a.T / kRowsPerCta, (a.B + a.spc - 1) / a.spc);
  return launch_k(k, grid, dim3(threads), g.smem, st, 1, map, a);
}

}  // namespace

int ln0_bwd_partial_rows(const RowArgs& ra) {
  return ra.B > 0 ? (ra.B + kLn0SamplesPerCta - 1) / kLn0SamplesPerCta * (ra.T / kRowsPerCta) : 0;
}

bool ln0_bwd_gather_supported(const RowArgs& ra) {
  if (ra.Dl != ra.D) return false;  // padded rows: the general form masks the padding
  const int e = ra.dtype == 0 ? 4 : 2, V = 16 / e;
  if (ra.T % kRowsPerCta || ra.D % ra.T || ra.D % V) return false;
  if ((ra.D / V + 31) / 32 * 32 > kLn0MaxThreads) return false;
  if ((long long)2 * kRowsPerCta * ra.D * e >= (1ll << 20)) return false;  // one mbarrier counts the own rows
  const Ln0Geom g = ln0_geom(ra.T, ra.D, e);
  if (g.stripe_pitch / e > 256 || ra.T > 256) return false;  // TMA box limits
  return (long long)g.smem <= (long long)max_dynamic_smem_bytes() - 1024;
}

cudaError_t launch_ln0_bwd_gather(const RowArgs& ra, const void* ds1, const void* x, const float* mu0,
                                  const float* r0, const void* gamma0, void* dx, float* pg0, float* pb0,
                                  cudaStream_t st) {
  if (!ln0_bwd_gather_supported(ra)) return cudaErrorInvalidValue;
  if (ra.B == 0) return cudaSuccess;
  Ln0GatherArgs a;
  a.ds1 = ds1;
  a.x = x;
  a.mu = mu0;
  a.rs = r0;
  a.gamma = gamma0;
  a.dx = dx;
  a.pg = pg0;
  a.pb = pb0;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidValue;
  a.B = ra.B;
  a.T = ra.T;
  a.D = ra.D;
  a.C = ra.D / ra.T;
  a.spc = kLn0SamplesPerCta;
  const bool pairs = a.C % 2 == 0;
  if (ra.dtype == 0) return pairs ? launch_typed<float, true>(a, 0, st) : launch_typed<float, false>(a, 0, st);
  if (ra.dtype == 1) return pairs ? launch_typed<bf16, true>(a, 1, st) : launch_typed<bf16, false>(a, 1, st);
  return pairs ? launch_typed<f16, true>(a, 2, st) : launch_typed<f16, false>(a, 2, st);
}

}  // namespace rmx
