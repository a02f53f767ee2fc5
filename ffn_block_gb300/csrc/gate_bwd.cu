// Backward of hidden = LN_x(U) * silu(LN_gate(G)) in one streaming pass.
//
// Page "Subgraph-fusion-based Mega-kernel Generation", section "Exact
// computation" (the dense_ffn_v2 subgraph); the chain rule written out, with
// Uh, Gh the normalised halves of Z, u = wx*Uh + bx, g = wg*Gh + bg and
// s = sigmoid(g):
//   du = dh * g * s,  dg = dh * u * s * (1 + g * (1 - s)),
//   gU = wx * du,     gG = wg * dg,
//   dU = rU * (gU - mean(gU) - Uh * mean(gU * Uh)), the same for dG,
//   dZ = [dU | dG];   dwx += du*Uh, dbx += du, dwg += dg*Gh, dbg += dg,
//   db1[t] += dZ.
//
// One CTA owns the rows b0 <= b < b1 of one token t and every column: thread
// j holds columns 8j ... 8j + 7 of both halves.  The dh and Z rows stream
// into shared memory through an S-stage ring of bulk copies (one thread
// issues them; a byte-counting mbarrier per stage says when a row has
// landed).  A row at a time (two when the LayerNorm weights live in shared
// memory) the CTA takes its four row sums with one barrier, then every
// thread finishes its own columns from registers, writes dZ and keeps the
// column partial sums in registers.  The element math runs
// on column pairs with the packed fp32x2 instructions (the same roundings as
// scalar fp32, half the instructions).  dh and Z are read from HBM once;
// every wait is bounded.

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {
namespace {

constexpr int kGateMaxStages = 8;

// Sums v[0..NS-1] (NS = 4 or 8) over the 32 lanes of a warp.  The first
// log2(NS) exchanges each halve the values a lane carries (it keeps one half
// and sends the other), the rest are plain butterflies.  On return lane l
// holds the sum of component l / (32 / NS); all lanes holding a component
// hold the same bits.
template <int NS>
__device__ __forceinline__ float warp_sum_transposed(const float (&v)[NS]) {
  static_assert(NS == 4 || NS == 8, "4 or 8 sums");
  const int lane = threadIdx.x & 31;
  float w[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) w[k] = v[k];
  int n = NS;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool hi = lane & off;
      const int h = n / 2;
#pragma unroll
      for (int k = 0; k < NS / 2; ++k)
        if (k < h) w[k] = (hi ? w[k + h] : w[k]) + __shfl_xor_sync(0xffffffffu, hi ? w[k] : w[k + h], off);
      n = h;
    } else {
      w[0] += __shfl_xor_sync(0xffffffffu, w[0], off);
    }
  }
  return w[0];
}

struct GateBwdArgs {
  const void* dh;        // [N, H]
  const void* Z;         // [N, 2H]
  const float* muU;      // [N] statistics of the forward's inner LayerNorms
  const float* rU;
  const float* muG;
  const float* rG;
  const void* wx;        // [H] LN_x weight / bias, LN_gate weight / bias
  const void* bx;
  const void* wg;
  const void* bg;
  void* dZ;              // [N, 2H]
  float* pwx;            // [P, H] column partials, P = nbblk * T
  float* pbx;
  float* pwg;
  float* pbg;
  float* pb1;            // [P, 2H]
  unsigned int* err;
  int B, T, H, nb, stages;
  int Hl;                // real columns of each half of pitch H (the rest are zero padding)
};

// Shared memory: stats [nb] float4 | red [2][16][8] float | weights [4][H]
// float (only when they do not stay in registers) | stages x (dh row | Z
// row) | mbarriers.  Thread `tid` owns the eight columns c0 = 8 * tid ...
// c0 + 7 of both halves (one 16-byte vector of a 16-bit type, two of
// float), as four pairs for the packed fp32x2 arithmetic.
// WREG: the thread's weights stay in registers (one CTA per SM leaves room
// for them when the CTA has at most 320 threads).  Register caps: each of
// the SM's four schedulers holds its warps' registers in its own quarter of
// the register file (16384), so a CTA of 10 warps (3 on some scheduler) may
// use at most 168 per thread, one of up to 16 warps at most 128.
constexpr int kGateE = 8;             // columns per thread and half
constexpr int kGateMaxThreads = 480;  // H up to 3840 (k = 3 at D = 1280)
constexpr int kGateRedWarps = 16;     // reduction buffer rows (at least kGateMaxThreads / 32)

template <typename T, bool WREG, int R>
__global__ void __maxnreg__(WREG ? 168 : 128) k_gate_bwd(const GateBwdArgs a) {
  pdl_enter();
  static_assert(R == 1 || R == 2, "rows per barrier");
  constexpr int NS = 4 * R;        // row sums per barrier
  constexpr int LPS = 32 / NS;     // lanes holding one sum after the warp reduction
  extern __shared__ __align__(16) unsigned char smem[];
  const int H = a.H, S = a.stages;
  const int bblk = blockIdx.x, t = blockIdx.y;
  const int b0 = bblk * a.nb;
  const int nrows = min(a.B, b0 + a.nb) - b0;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31, nw = nthreads >> 5;
  const int c0 = tid * kGateE;
  const bool active = c0 < H;

  float4* st_row = reinterpret_cast<float4*>(smem);                  // (rU, -mU*rU, rG, -mG*rG) per row
  float* red = reinterpret_cast<float*>(smem + (size_t)a.nb * 16);   // [2][16 warps][NS]
  float* wsm = red + 2 * kGateRedWarps * NS;                         // [4][H] (not WREG)
  unsigned char* ring = reinterpret_cast<unsigned char*>(wsm + (WREG ? 0 : 4 * (size_t)H));
  const size_t row_bytes = (size_t)3 * H * sizeof(T);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)S * row_bytes);
  __shared__ int abort_flag;

  const T* dh = reinterpret_cast<const T*>(a.dh);
  const T* Z = reinterpret_cast<const T*>(a.Z);
  auto issue = [&](int i, int s) {  // row i of this CTA into stage s
    const size_t r = (size_t)(b0 + i) * a.T + t;
    const uint32_t bar = smem_u32(&full[s]);
    unsigned char* dst = ring + (size_t)s * row_bytes;
    mbar_arrive_expect_tx(bar, (uint32_t)row_bytes);
    bulk_g2s(smem_u32(dst), dh + r * H, (uint32_t)(H * sizeof(T)), bar);
    bulk_g2s(smem_u32(dst + (size_t)H * sizeof(T)), Z + r * 2 * H, (uint32_t)(2 * H * sizeof(T)), bar);
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < min(S, nrows); ++i) issue(i, i);
  // Per-row statistics and the weights while the first rows are in flight.
  for (int i = tid; i < nrows; i += nthreads) {
    const size_t r = (size_t)(b0 + i) * a.T + t;
    const float sU = a.rU[r], sG = a.rG[r];
    st_row[i] = make_float4(sU, -a.muU[r] * sU, sG, -a.muG[r] * sG);
  }
  const T* wp[4] = {reinterpret_cast<const T*>(a.wx), reinterpret_cast<const T*>(a.bx),
                    reinterpret_cast<const T*>(a.wg), reinterpret_cast<const T*>(a.bg)};
  float2 rw[WREG ? 4 : 1][4];
  if (WREG) {
    if (active) {
#pragma unroll
      for (int k = 0; k < (WREG ? 4 : 1); ++k) ld8<T>(wp[k] + c0, rw[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      for (int c = tid; c < H; c += nthreads) wsm[k * H + c] = to_f(wp[k][c]);
  }
  __syncthreads();

  // Column partial sums of dwx, dbx, dwg, dbg and db1 (U and G halves).
  float2 awx[4], abx[4], awg[4], abg[4], a1u[4], a1g[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) awx[k] = abx[k] = awg[k] = abg[k] = a1u[k] = a1g[k] = f2(0.f);

  const float invH = 1.0f / (float)a.Hl;
  const bool tail = c0 + kGateE > a.Hl;  // this thread owns padding columns (written as zeros)
  T* dZrow = reinterpret_cast<T*>(a.dZ) + ((size_t)b0 * a.T + t) * 2 * H;
  const size_t dZstep = (size_t)a.T * 2 * H;
  int issued = min(S, nrows);
  bool aborted = false;
  int s = 0;          // stage of row i
  uint32_t ph = 0;    // parity of that stage's current phase
  for (int i = 0; i < nrows; i += R, dZrow += R * dZstep) {
    const int nr = min(R, nrows - i);  // rows in this step
    const int s1 = s + 1 == S ? 0 : s + 1;
    const uint32_t ph1 = s + 1 == S ? ph ^ 1u : ph;
    bool ok = mbar_wait_bounded(smem_u32(&full[s]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                (volatile int*)&abort_flag);
    if (nr == 2)
      ok = ok && mbar_wait_bounded(smem_u32(&full[s1]), ph1, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                   (volatile int*)&abort_flag);
    // Pass 1: everything that needs only this element, plus the row sums;
    // gU, Uh, gG, Gh stay in registers for pass 2.
    float2 kgU[R][4], kUh[R][4], kgG[R][4], kGh[R][4];
    float rsum[NS];
    float sUr[R], sGr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4 sr = st_row[min(i + r, nrows - 1)];
      sUr[r] = sr.x;
      sGr[r] = sr.z;
      float2 rs[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
      if (ok && active && r < nr) {
        const T* st = reinterpret_cast<const T*>(ring + (size_t)(r == 0 ? s : s1) * row_bytes);
        float2 dhv[4], zu[4], zg[4], w[4][4];
        ld8<T>(st + c0, dhv);
        ld8<T>(st + H + c0, zu);
        ld8<T>(st + 2 * H + c0, zg);
        if (WREG) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) w[k][q] = rw[WREG ? k : 0][q];
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 lo = *reinterpret_cast<const float4*>(wsm + k * H + c0);
            const float4 hi = *reinterpret_cast<const float4*>(wsm + k * H + c0 + 4);
            w[k][0] = make_float2(lo.x, lo.y);
            w[k][1] = make_float2(lo.z, lo.w);
            w[k][2] = make_float2(hi.x, hi.y);
            w[k][3] = make_float2(hi.z, hi.w);
          }
        }
        const float2 sU = f2(sr.x), cU = f2(sr.y), sG = f2(sr.z), cG = f2(sr.w);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 Uh = fma2(zu[q], sU, cU);
          const float2 Gh = fma2(zg[q], sG, cG);
          const float2 u = fma2(w[0][q], Uh, w[1][q]);
          const float2 g = fma2(w[2][q], Gh, w[3][q]);
          const float2 sg = sigmoid_fast2(g);
          const float2 gs = mul2(g, sg);
          const float2 du = mul2(dhv[q], gs);
          // silu'(g) = s + g s (1 - s) = s + (gs - gs * s)
          const float2 dsilu = add2(sg, fma2(gs, make_float2(-sg.x, -sg.y), gs));
          const float2 dg = mul2(mul2(dhv[q], u), dsilu);
          const float2 gU = mul2(w[0][q], du), gG = mul2(w[2][q], dg);
          rs[0] = add2(rs[0], gU);
          rs[1] = fma2(gU, Uh, rs[1]);
          rs[2] = add2(rs[2], gG);
          rs[3] = fma2(gG, Gh, rs[3]);
          awx[q] = fma2(du, Uh, awx[q]);
          abx[q] = add2(abx[q], du);
          awg[q] = fma2(dg, Gh, awg[q]);
          abg[q] = add2(abg[q], dg);
          kgU[r][q] = gU;
          kUh[r][q] = Uh;
          kgG[r][q] = gG;
          kGh[r][q] = Gh;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) rsum[4 * r + k] = rs[k].x + rs[k].y;
    }
    // Row sums over the CTA: per warp (lane LPS*c holds sum c), then over
    // the warps in a fixed order, the same bits in every thread.  Stored
    // warp-major, so that neither the stores nor the reads below conflict.
    float* rb = red + ((i / R) & 1) * kGateRedWarps * NS;
    {
      const float k = warp_sum_transposed<NS>(rsum);
      if (lane % LPS == 0) rb[warp * NS + lane / LPS] = k;
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
    float m[NS];
    {
      // Lane l adds warps (l % LPS) + LPS*k of sum l / LPS (at most 16 warps),
      // then the LPS lanes of each sum combine.
      const int c = lane / LPS, w0 = lane % LPS;
      float v = 0.f;
#pragma unroll
      for (int w = w0; w < kGateRedWarps; w += LPS)
        if (w < nw) v += rb[w * NS + c];
#pragma unroll
      for (int off = LPS / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
#pragma unroll
      for (int k = 0; k < NS; ++k) m[k] = __shfl_sync(0xffffffffu, v, k * LPS) * invH;
    }
    if (active) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r < nr) {
          const float sU = sUr[r], sG = sGr[r];
          const float2 pU = f2(-m[4 * r + 1]), qU = f2(-sU * m[4 * r]);
          const float2 pG = f2(-m[4 * r + 3]), qG = f2(-sG * m[4 * r + 2]);
          float2 oU[4], oG[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            oU[q] = fma2(f2(sU), fma2(pU, kUh[r][q], kgU[r][q]), qU);
            oG[q] = fma2(f2(sG), fma2(pG, kGh[r][q], kgG[r][q]), qG);
            if (tail) {
              const int c = c0 + 2 * q;
              if (c >= a.Hl) oU[q].x = oG[q].x = 0.f;
              if (c + 1 >= a.Hl) oU[q].y = oG[q].y = 0.f;
            }
            a1u[q] = add2(a1u[q], oU[q]);
            a1g[q] = add2(a1g[q], oG[q]);
          }
          st8<T>(dZrow + r * dZstep + c0, oU);
          st8<T>(dZrow + r * dZstep + H + c0, oG);
        }
      }
    }
  }

  if (aborted) {
    // Wait (bounded) for the copies still in flight before the CTA's shared
    // memory goes away: the newest copy issued into each stage.
    if (tid == 0) {
      volatile int no_abort = 0;
      for (int i = max(0, issued - S); i < issued; ++i) {
        mbar_wait_bounded(smem_u32(&full[i % S]), (uint32_t)((i / S) & 1), kWaitLimitNs, a.err,
                          ERRBIT_WAIT_ROWS, &no_abort);
      }
    }
    return;
  }

  if (active) {
    const size_t p = (size_t)bblk * a.T + t;
    auto put = [&](float* dst, const float2 (&v)[4]) {
      *reinterpret_cast<float4*>(dst) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
    };
    put(a.pwx + p * H + c0, awx);
    put(a.pbx + p * H + c0, abx);
    put(a.pwg + p * H + c0, awg);
    put(a.pbg + p * H + c0, abg);
    put(a.pb1 + p * 2 * H + c0, a1u);
    put(a.pb1 + p * 2 * H + H + c0, a1g);
  }
}

// Rows per barrier: one with the weights in registers (measured 2% faster
// than two at H = 2560), two when they live in shared memory.
template <bool WREG> constexpr int gate_rows() { return WREG ? 1 : 2; }

// Threads, ring stages and shared memory of a CTA of nb rows (0 if even two
// stages do not fit).
template <typename T, bool WREG>
size_t gate_shape(int H, int nb, int& threads, int& stages) {
  threads = (H / kGateE + 31) / 32 * 32;
  const size_t fixed = (size_t)nb * 16 + 2 * kGateRedWarps * 8 * 4 + (WREG ? 0 : (size_t)4 * H * 4);
  const size_t row_bytes = (size_t)3 * H * sizeof(T);
  const int cap = max_dynamic_smem_bytes() - 1024;  // static shared memory and slack
  const long long room = ((long long)cap - (long long)fixed) / (long long)(row_bytes + 8);
  if (room < 2) return 0;
  stages = (int)(room < kGateMaxStages ? room : kGateMaxStages);
  return fixed + (size_t)stages * row_bytes + (size_t)stages * 8;
}

template <typename T, bool WREG>
int gate_ctas_per_sm(int H) {
  int threads = 0, stages = 0;
  const size_t smem = gate_shape<T, WREG>(H, kGateBwdMaxRows, threads, stages);
  if (smem == 0) return 1;
  auto k = k_gate_bwd<T, WREG, gate_rows<WREG>()>;
  int n = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess || n < 1)
    return 1;
  return n;
}

template <typename T, bool WREG>
cudaError_t launch_typed(const GateBwdArgs& base, cudaStream_t st, dim3 grid) {
  GateBwdArgs a = base;
  int threads = 0;
  const size_t smem = gate_shape<T, WREG>(a.H, a.nb, threads, a.stages);
  if (smem == 0) return cudaErrorInvalidValue;
  auto k = k_gate_bwd<T, WREG, gate_rows<WREG>()>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(k, grid, dim3(threads), smem, st, 1, a);
}

}  // namespace

int gate_bwd_ctas_per_sm(const RowArgs& ra) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const auto key = std::make_tuple(dev, ra.dtype, ra.H);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const bool wreg = ra.H / kGateE <= 320;
  int n = 1;
  if (ra.dtype == 0) n = wreg ? gate_ctas_per_sm<float, true>(ra.H) : gate_ctas_per_sm<float, false>(ra.H);
  else if (ra.dtype == 1) n = wreg ? gate_ctas_per_sm<bf16, true>(ra.H) : gate_ctas_per_sm<bf16, false>(ra.H);
  else n = wreg ? gate_ctas_per_sm<f16, true>(ra.H) : gate_ctas_per_sm<f16, false>(ra.H);
  cache[key] = n;
  return n;
}

bool gate_bwd_fused_supported(const RowArgs& a) {
  // Eight columns of each half per thread, at most kGateMaxThreads threads.
  return a.H % kGateE == 0 && (a.H / kGateE + 31) / 32 * 32 <= kGateMaxThreads && a.nb <= kGateBwdMaxRows;
}

cudaError_t launch_gate_bwd(const RowArgs& ra, const void* dh, const void* Z, const float* muU, const float* rU,
                            const float* muG, const float* rG, const void* wx, const void* bx, const void* wg,
                            const void* bg, void* dZ, float* pwx, float* pbx, float* pwg, float* pbg, float* pb1,
                            cudaStream_t st) {
  if (!gate_bwd_fused_supported(ra)) return cudaErrorInvalidValue;
  GateBwdArgs a;
  a.dh = dh;
  a.Z = Z;
  a.muU = muU;
  a.rU = rU;
  a.muG = muG;
  a.rG = rG;
  a.wx = wx;
  a.bx = bx;
  a.wg = wg;
  a.bg = bg;
  a.dZ = dZ;
  a.pwx = pwx;
  a.pbx = pbx;
  a.pwg = pwg;
  a.pbg = pbg;
  a.pb1 = pb1;
  a.err = device_error_word();
  a.B = ra.B;
  a.T = ra.T;
  a.H = ra.H;
  a.Hl = ra.Hl;
  a.nb = ra.nb;
  a.stages = 0;
  if (!a.err) return cudaErrorInvalidValue;
  const dim3 grid(ra.nbblk, ra.T);
  const bool wreg = ra.H / kGateE <= 320;
  if (ra.dtype == 0) return wreg ? launch_typed<float, true>(a, st, grid) : launch_typed<float, false>(a, st, grid);
  if (ra.dtype == 1) return wreg ? launch_typed<bf16, true>(a, st, grid) : launch_typed<bf16, false>(a, st, grid);
  return wreg ? launch_typed<f16, true>(a, st, grid) : launch_typed<f16, false>(a, st, grid);
}

}  // namespace rmx
