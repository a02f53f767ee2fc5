// Backward of the three outer LayerNorms, one streaming pass per call.
//
// Page "Subgraph-fusion-based Mega-kernel Generation", section "Exact
// computation": LN(z) = (z - mean) / sqrt(mean((z - mean)^2) + eps) * gamma
// + beta over each row of D.  With xh the normalised row, g = gamma * gin and
// the row means mg = mean(g), mgx = mean(g * xh):
//   out = rstd * (g - mg - xh * mgx)     (+ a residual gradient, by mode)
//   dgamma += gin * xh, dbeta += gin     (column partial sums)
// Modes (kernels.h): LNB_BIAS also sums out over the batch per token (the
// bias gradient of the GEMM that feeds norm2); LNB_MIXED_TOO writes out both
// plainly and token-mixed; LNB_RESID adds a residual gradient to out;
// LNB_PLAIN writes out alone.
//
// One CTA owns the rows b0 <= b < b1 of one token t.  Their input rows stream
// into shared memory through an S-stage ring of bulk copies (one thread
// issues them; a byte-counting mbarrier per stage); thread j owns the j-th
// 16-byte vector of columns.  Per row the CTA takes the two row sums with one
// barrier, then each thread writes its columns and keeps the column partial
// sums in registers.  Every wait is bounded.

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "pairs.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {
namespace {

constexpr int kLnMaxStages = 8;
constexpr int kLnSmemTarget = 52 * 1024;  // about four CTAs per SM

// Sums v[0..3] over a warp with six shuffles: on return lane l holds the sum
// of component 2 * bit4(l) + bit3(l); lanes holding the same component hold
// the same bits.
__device__ __forceinline__ float warp_sum4_transposed(float v0, float v1, float v2, float v3) {
  const int lane = threadIdx.x & 31;
  const bool b4 = lane & 16, b3 = lane & 8;
  float k0 = b4 ? v2 : v0;
  float k1 = b4 ? v3 : v1;
  const float s0 = b4 ? v0 : v2;
  const float s1 = b4 ? v1 : v3;
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  float k = b3 ? k1 : k0;
  const float s = b3 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, s, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// Token mix as an addressing rule: column d = i*C + c of row j of a sample
// goes to row i, column j*C + c.  Writes the V values of columns d0 .. d0+V-1
// of row j to their mixed places (pairs when C is even).  Columns d >= Dl
// (the zero padding of a row of pitch D) stay in row j and are written as
// zeros.
template <typename T, int V>
__device__ __forceinline__ void store_mixed_row(T* sample_base, const float* v, int j, int d0, int C, int D,
                                                int Dl) {
  int i = d0 / C, c = d0 - i * C;
  if ((C & 1) == 0) {
#pragma unroll
    for (int e = 0; e < V; e += 2) {
      const bool pad = d0 + e >= Dl;  // Dl = T * C is even: pairs never straddle it
      T* dst = pad ? sample_base + (size_t)j * D + d0 + e : sample_base + (size_t)i * D + j * C + c;
      const float a = pad ? 0.f : v[e], b = pad ? 0.f : v[e + 1];
      if (sizeof(T) == 2) {
        T pr[2] = {from_f<T>(a), from_f<T>(b)};
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(pr);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(a, b);
      }
      c += 2;
      while (c >= C) {
        c -= C;
        ++i;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < V; ++e) {
      if (d0 + e >= Dl) sample_base[(size_t)j * D + d0 + e] = from_f<T>(0.f);
      else sample_base[(size_t)i * D + j * C + c] = from_f<T>(v[e]);
      if (++c == C) {
        c = 0;
        ++i;
      }
    }
  }
}

struct LnBwdArgs {
  const void* gin;     // [N, D] upstream gradient
  const void* s;       // [N, D] LayerNorm input
  const void* resid;   // [N, D] LNB_RESID: gradient added to the output
  const float* mu;     // [N] forward statistics
  const float* rs;
  const void* gamma;   // [D]
  void* out;           // [N, D]
  void* out_mixed;     // [N, D] LNB_MIXED_TOO: token-mixed copy of out
  float* pg;           // [nbblk*T, D] column partials of dgamma
  float* pb;           // [nbblk*T, D] column partials of dbeta
  float* pbias;        // [nbblk, T, D] LNB_BIAS: column partials of sum_b out
  unsigned int* err;
  int B, T, D, C, nb, stages;
  int Dl;              // real columns of a row of pitch D (the rest are zero padding)
};

// Per-row statistics area, rounded up so the ring starts 16-byte aligned.
__host__ __device__ inline size_t stats_bytes(int nb) { return ((size_t)nb * 8 + 15) & ~(size_t)15; }

template <int MODE> struct LnRows {
  // Row tensors staged per row: gin, s, then resid.
  static constexpr int value = MODE == LNB_RESID ? 3 : 2;
};

// Shared memory: stats [nb] float2 | red [2][4][32] float | stages x rows |
// mbarriers.  Two rows are taken per barrier: their four row sums are reduced
// together, which halves the per-row reduction and barrier work.  At most 96
// registers a thread (128 where the token-mixed copy is written too), so
// that four CTAs of 160 threads share an SM.
template <typename T, int MODE>
__global__ void __maxnreg__(MODE == LNB_MIXED_TOO ? 128 : 96) k_ln_bwd_ring(const LnBwdArgs a) {
  pdl_enter();
  constexpr int E = VecN<T>::value;
  constexpr int NR = LnRows<MODE>::value;
  extern __shared__ __align__(16) unsigned char smem[];
  const int D = a.D, S = a.stages;
  const int t = blockIdx.x, bblk = blockIdx.y;
  const int b0 = bblk * a.nb;
  const int nrows = min(a.B, b0 + a.nb) - b0;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31, nw = nthreads >> 5;
  const int c0 = tid * E;
  const bool active = c0 < D;

  float2* st_row = reinterpret_cast<float2*>(smem);                    // (rstd, -mean*rstd) per row
  float* red = reinterpret_cast<float*>(smem + stats_bytes(a.nb));     // [2][4][32]
  unsigned char* ring = reinterpret_cast<unsigned char*>(red + 2 * 4 * 32);
  const size_t tensor_bytes = (size_t)D * sizeof(T);
  const size_t row_bytes = NR * tensor_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)S * row_bytes);
  __shared__ int abort_flag;

  const T* third = reinterpret_cast<const T*>(a.resid);
  auto issue = [&](int i, int s) {  // row i of this CTA into stage s
    const size_t r = (size_t)(b0 + i) * a.T + t;
    const uint32_t bar = smem_u32(&full[s]);
    const uint32_t dst = smem_u32(ring + (size_t)s * row_bytes);
    mbar_arrive_expect_tx(bar, (uint32_t)row_bytes);
    bulk_g2s(dst, reinterpret_cast<const T*>(a.gin) + r * D, (uint32_t)tensor_bytes, bar);
    bulk_g2s(dst + (uint32_t)tensor_bytes, reinterpret_cast<const T*>(a.s) + r * D, (uint32_t)tensor_bytes, bar);
    if (NR == 3) bulk_g2s(dst + 2 * (uint32_t)tensor_bytes, third + r * D, (uint32_t)tensor_bytes, bar);
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < min(S, nrows); ++i) issue(i, i);
  for (int i = tid; i < nrows; i += nthreads) {
    const size_t r = (size_t)(b0 + i) * a.T + t;
    const float rstd = a.rs[r];
    st_row[i] = make_float2(rstd, -a.mu[r] * rstd);
  }
  // The element math runs on column pairs with the packed fp32x2
  // instructions (each rounds as the scalar one).
  constexpr int P = E / 2;
  float2 gam[P];
  if (active) ld16p<T>(reinterpret_cast<const T*>(a.gamma) + c0, gam);
  __syncthreads();

  float2 ag[P], ab[P], ao[P];
#pragma unroll
  for (int k = 0; k < P; ++k) ag[k] = ab[k] = ao[k] = f2(0.f);

  const float invD = 1.0f / (float)a.Dl;
  const bool tail = c0 + E > a.Dl;  // this thread owns padding columns
  const size_t row_step = (size_t)a.T * D;
  T* out_row = reinterpret_cast<T*>(a.out) + ((size_t)b0 * a.T + t) * D;
  int issued = min(S, nrows);
  bool aborted = false;
  int s = 0;
  uint32_t ph = 0;
  for (int i = 0; i < nrows; i += 2, out_row += 2 * row_step) {
    const int nr = min(2, nrows - i);  // rows in this step
    const int s1 = s + 1 == S ? 0 : s + 1;
    const uint32_t ph1 = s + 1 == S ? ph ^ 1u : ph;
    bool ok = mbar_wait_bounded(smem_u32(&full[s]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                (volatile int*)&abort_flag);
    if (nr == 2)
      ok = ok && mbar_wait_bounded(smem_u32(&full[s1]), ph1, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                   (volatile int*)&abort_flag);
    float2 g[2][P], xh[2][P], rv[2][P];
    float2 rs2[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
    float rstd[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float2 sr = st_row[min(i + r, nrows - 1)];
      rstd[r] = sr.x;
      if (ok && active && r < nr) {
        const T* st = reinterpret_cast<const T*>(ring + (size_t)(r == 0 ? s : s1) * row_bytes);
        float2 gv[P], sv[P];
        ld16p<T>(st + c0, gv);
        ld16p<T>(st + D + c0, sv);
        if (MODE == LNB_RESID) ld16p<T>(st + 2 * D + c0, rv[r]);
        const float2 sa = f2(sr.x), sb = f2(sr.y);
#pragma unroll
        for (int k = 0; k < P; ++k) {
          xh[r][k] = fma2(sv[k], sa, sb);
          g[r][k] = mul2(gam[k], gv[k]);
          rs2[2 * r] = add2(rs2[2 * r], g[r][k]);
          rs2[2 * r + 1] = fma2(g[r][k], xh[r][k], rs2[2 * r + 1]);
          ag[k] = fma2(gv[k], xh[r][k], ag[k]);
          ab[k] = add2(ab[k], gv[k]);
        }
      }
    }
    const float rsum[4] = {rs2[0].x + rs2[0].y, rs2[1].x + rs2[1].y, rs2[2].x + rs2[2].y, rs2[3].x + rs2[3].y};
    float* rb = red + ((i >> 1) & 1) * 4 * 32;
    {
      const float k = warp_sum4_transposed(rsum[0], rsum[1], rsum[2], rsum[3]);
      if ((lane & 7) == 0) rb[(lane >> 3) * 32 + warp] = k;
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid == 0) {
      if (issued < nrows) issue(issued++, s);
      if (nr == 2 && issued < nrows) issue(issued++, s1);
    }
    for (int r = 0; r < nr; ++r) {
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    float m[4];
    {
      // Lane l adds warps (l & 7) and (l & 7) + 8 (at most 16 warps) of sum
      // l >> 3; the eight lanes of each sum then combine.
      const int c = lane >> 3, w0 = lane & 7;
      float v = (w0 < nw ? rb[c * 32 + w0] : 0.f) + (w0 + 8 < nw ? rb[c * 32 + w0 + 8] : 0.f);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
#pragma unroll
      for (int k = 0; k < 4; ++k) m[k] = __shfl_sync(0xffffffffu, v, k * 8) * invD;
    }
    if (active) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r < nr) {
          const float2 nmgx = f2(-m[2 * r + 1]), rs = f2(rstd[r]), q0 = f2(-rstd[r] * m[2 * r]);
          float2 o[P];
#pragma unroll
          for (int k = 0; k < P; ++k) o[k] = fma2(rs, fma2(nmgx, xh[r][k], g[r][k]), q0);
          if (tail) {  // padding columns are written as zeros
#pragma unroll
            for (int k = 0; k < P; ++k) {
              if (c0 + 2 * k >= a.Dl) o[k].x = 0.f;
              if (c0 + 2 * k + 1 >= a.Dl) o[k].y = 0.f;
            }
          }
          if (MODE == LNB_BIAS) {
#pragma unroll
            for (int k = 0; k < P; ++k) ao[k] = add2(ao[k], o[k]);
          }
          if (MODE == LNB_MIXED_TOO)
            store_mixed_row<T, E>(reinterpret_cast<T*>(a.out_mixed) + (size_t)(b0 + i + r) * a.T * D,
                                  reinterpret_cast<const float*>(o), t, c0, a.C, D, a.Dl);
          if (MODE == LNB_RESID) {
#pragma unroll
            for (int k = 0; k < P; ++k) o[k] = add2(o[k], rv[r][k]);
          }
          st16p<T>(out_row + r * row_step + c0, o);
        }
      }
    }
  }

  if (aborted) {
    // Wait (bounded) for the newest copy issued into each stage before the
    // CTA's shared memory goes away.
    if (tid == 0) {
      volatile int no_abort = 0;
      for (int i = max(0, issued - S); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % S]), (uint32_t)((i / S) & 1), kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                          &no_abort);
    }
    return;
  }
  if (active) {
    const size_t p = (size_t)bblk * a.T + t;
    auto put = [&](float* dst, const float* v) {
#pragma unroll
      for (int k = 0; k < E; k += 4)
        *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
    };
    put(a.pg + p * D + c0, reinterpret_cast<const float*>(ag));
    put(a.pb + p * D + c0, reinterpret_cast<const float*>(ab));
    if (MODE == LNB_BIAS) put(a.pbias + p * D + c0, reinterpret_cast<const float*>(ao));
  }
}

// Threads, ring stages and shared memory of a ring CTA of nb rows.
template <typename T, int MODE>
size_t ring_shape(int D, int nb, int& threads, int& stages) {
  constexpr int E = VecN<T>::value;
  threads = (D / E + 31) / 32 * 32;
  const size_t fixed = stats_bytes(nb) + 2 * 4 * 32 * 4;
  const size_t row_bytes = (size_t)LnRows<MODE>::value * D * sizeof(T);
  long long room = ((long long)kLnSmemTarget - (long long)fixed) / (long long)(row_bytes + 8);
  if (room < 2) room = 2;
  if (room > kLnMaxStages) room = kLnMaxStages;
  stages = (int)room;
  return fixed + (size_t)stages * (row_bytes + 8);
}

template <typename T, int MODE>
int ring_ctas_per_sm(int D) {
  int threads = 0, stages = 0;
  const size_t smem = ring_shape<T, MODE>(D, kLnBwdMaxRows, threads, stages);
  auto k = k_ln_bwd_ring<T, MODE>;
  int n = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess || n < 1)
    return 1;
  return n;
}

template <typename T, int MODE>
cudaError_t launch_ring(const LnBwdArgs& base, cudaStream_t st) {
  LnBwdArgs a = base;
  int threads = 0;
  const size_t smem = ring_shape<T, MODE>(a.D, a.nb, threads, a.stages);
  if ((long long)smem > (long long)max_dynamic_smem_bytes() - 1024) return cudaErrorInvalidValue;
  auto k = k_ln_bwd_ring<T, MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(k, dim3(a.T, (a.B + a.nb - 1) / a.nb), dim3(threads), smem, st, 1, a);
}

template <typename T>
cudaError_t launch_mode(const LnBwdArgs& a, int mode, cudaStream_t st) {
  if (mode == LNB_BIAS) return launch_ring<T, LNB_BIAS>(a, st);
  if (mode == LNB_MIXED_TOO) return launch_ring<T, LNB_MIXED_TOO>(a, st);
  if (mode == LNB_PLAIN) return launch_ring<T, LNB_PLAIN>(a, st);
  return launch_ring<T, LNB_RESID>(a, st);
}

}  // namespace

int ln_bwd_ctas_per_sm(const RowArgs& ra) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const auto key = std::make_tuple(dev, ra.dtype, ra.D);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const int n = ra.dtype == 0 ? ring_ctas_per_sm<float, LNB_BIAS>(ra.D)
                : ra.dtype == 1 ? ring_ctas_per_sm<bf16, LNB_BIAS>(ra.D)
                                : ring_ctas_per_sm<f16, LNB_BIAS>(ra.D);
  cache[key] = n;
  return n;
}

cudaError_t launch_ln_bwd(const RowArgs& ra, int mode, const void* gin, const void* s, const float* mu,
                          const float* rs, const void* gamma, const void* resid, void* out, void* out_mixed, float* pg, float* pb, float* pbias, cudaStream_t st) {
  const int V = ra.dtype == 0 ? 4 : 8;
  if (ra.D % V || ra.D / V > 512 || ra.nb_ln < 1 || ra.nb_ln > kLnBwdMaxRows || ra.Dl % ra.T || ra.Dl > ra.D)
    return cudaErrorInvalidValue;
  LnBwdArgs a;
  a.gin = gin;
  a.s = s;
  a.resid = resid;
  a.mu = mu;
  a.rs = rs;
  a.gamma = gamma;
  a.out = out;
  a.out_mixed = out_mixed;
  a.pg = pg;
  a.pb = pb;
  a.pbias = pbias;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidValue;
  a.B = ra.B;
  a.T = ra.T;
  a.D = ra.D;
  a.Dl = ra.Dl;
  a.C = ra.Dl / ra.T;
  a.nb = ra.nb_ln;
  a.stages = 0;
  if (ra.dtype == 0) return launch_mode<float>(a, mode, st);
  if (ra.dtype == 1) return launch_mode<bf16>(a, mode, st);
  return launch_mode<f16>(a, mode, st);
}

cudaError_t launch_ln2_bwd(const RowArgs& a, const void* dy, const void* s2, const float* mu2, const float* r2,
                           const void* g2, void* ds2, float* pg2, float* pb2, float* pbo, cudaStream_t st) {
  return launch_ln_bwd(a, LNB_BIAS, dy, s2, mu2, r2, g2, nullptr, ds2, nullptr, pg2, pb2, pbo, st);
}

}  // namespace rmx
