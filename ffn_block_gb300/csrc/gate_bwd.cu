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
// landed).  A row at a time the CTA takes its four row sums with one
// barrier, then every thread finishes its own columns and writes dZ.  Each
// thread's LayerNorm weights and its 48 column partial sums live either in
// registers (the register form) or in tensor memory (the TMEM form: TMEM is
// otherwise unused here, and moving those 80 values out of the register
// file lets two 320-thread CTAs share an SM); gate_form() picks the faster
// for a shape.  The element math runs on column pairs with the packed
// fp32x2 instructions (the same roundings as scalar fp32, half the
// instructions).  dh and Z are read from HBM once; every wait is bounded,
// and the TMEM columns are freed on every exit.

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
  int tmem_cols;         // k_gate_bwd_tm: TMEM columns the CTA allocates
};

// Thread `tid` owns the eight columns c0 = 8 * tid ... c0 + 7 of both
// halves (one 16-byte vector of a 16-bit type, two of float), as four pairs
// for the packed fp32x2 arithmetic.
constexpr int kGateE = 8;             // columns per thread and half
constexpr int kGateMaxThreads = 480;  // H up to 3840 (k = 3 at D = 1280)
constexpr int kGateRedWarps = 16;     // reduction buffer rows (at least kGateMaxThreads / 32)

// ---------------------------------------------------------------- register form
// The pass with each thread's weights (WREG) and column partial sums in
// registers: one CTA of up to 320 threads per SM at H = 2560, two at
// H <= 1536.  It wins over the TMEM form below when the TMEM form would not
// hold more CTAs per SM, or when there are few rows per SM (its start-up,
// allocating and filling tensor memory, is then not paid back).  Shared
// memory: stats [nb] float4 | red [2][16][NS] float | weights [4][H] float
// (not WREG) | stages x (dh row | Z row) | mbarriers.  Register caps: each of
// the SM's four schedulers holds its warps' registers in its own quarter of
// the register file (16384), so a CTA of 10 warps (3 on some scheduler) may
// use at most 168 per thread.
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
          }
          if (tail) {  // padding columns are written as zeros
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c = c0 + 2 * q;
              if (c >= a.Hl) oU[q].x = oG[q].x = 0.f;
              if (c + 1 >= a.Hl) oU[q].y = oG[q].y = 0.f;
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
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

// ---------------------------------------------------------------- the pass
// Each thread owns 80 TMEM columns of its own lane (the warps of one lane
// quarter side by side): its weights as fp32 ([wx | wg] then [bx | bg], 16
// columns each) and its 48 partials ([dwx | dbx], [dwg | dbg], [db1 of U |
// of G]), all for its eight column pairs.  Per row it loads the weights, adds
// the row's terms to the partials with 16-column loads and stores, and takes
// one barrier for the row sums.  Measured against the same pass with the
// weights and partials in registers (one CTA per SM): 0.382 against 0.434 ms
// at c3, 0.389 against 0.479 ms at c4.
__device__ __forceinline__ void tm_ld16(uint32_t taddr, float2 (&v)[8]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = make_float2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
}
// 32 consecutive columns in one load: the first 16 into a, the next 16 into b.
__device__ __forceinline__ void tm_ld32(uint32_t taddr, float2 (&a)[8], float2 (&b)[8]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    a[k] = make_float2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
    b[k] = make_float2(__uint_as_float(r[16 + 2 * k]), __uint_as_float(r[16 + 2 * k + 1]));
  }
}
__device__ __forceinline__ void tm_st16(uint32_t taddr, const float2 (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(__float_as_uint(v[0].x)), "r"(__float_as_uint(v[0].y)), "r"(__float_as_uint(v[1].x)),
        "r"(__float_as_uint(v[1].y)), "r"(__float_as_uint(v[2].x)), "r"(__float_as_uint(v[2].y)),
        "r"(__float_as_uint(v[3].x)), "r"(__float_as_uint(v[3].y)), "r"(__float_as_uint(v[4].x)),
        "r"(__float_as_uint(v[4].y)), "r"(__float_as_uint(v[5].x)), "r"(__float_as_uint(v[5].y)),
        "r"(__float_as_uint(v[6].x)), "r"(__float_as_uint(v[6].y)), "r"(__float_as_uint(v[7].x)),
        "r"(__float_as_uint(v[7].y))
      : "memory");
}
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tm_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <typename T>
__global__ void __maxnreg__(96) k_gate_bwd_tm(const GateBwdArgs a) {
  pdl_enter();
  constexpr int NS = 4;         // row sums per barrier
  constexpr int LPS = 32 / NS;  // lanes holding one sum after the warp reduction
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
  unsigned char* ring = reinterpret_cast<unsigned char*>(red + 2 * kGateRedWarps * NS);
  const size_t row_bytes = (size_t)3 * H * sizeof(T);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)S * row_bytes);
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;

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

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }
  tm_fence_before();
  __syncthreads();
  tm_fence_after();
  const uint32_t tbase = tmem_slot;
  // Lane quarter warp % 4 (the lanes a warp may access); the warps of one
  // quarter take 80 columns each: weights at tw, partials at tp.
  const uint32_t tw = tbase + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * 80);
  const uint32_t tp = tw + 32;
  if (tid == 0)
    for (int i = 0; i < min(S, nrows); ++i) issue(i, i);
  for (int i = tid; i < nrows; i += nthreads) {
    const size_t r = (size_t)(b0 + i) * a.T + t;
    const float sU = a.rU[r], sG = a.rG[r];
    st_row[i] = make_float4(sU, -a.muU[r] * sU, sG, -a.muG[r] * sG);
  }
  {
    float2 w[8], z[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = z[k] = f2(0.f);
    if (active) {
      float2 v[4];
      ld8<T>(reinterpret_cast<const T*>(a.wx) + c0, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = v[q];
      ld8<T>(reinterpret_cast<const T*>(a.wg) + c0, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) w[4 + q] = v[q];
    }
    tm_st16(tw, w);  // [wx | wg]
    if (active) {
      float2 v[4];
      ld8<T>(reinterpret_cast<const T*>(a.bx) + c0, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = v[q];
      ld8<T>(reinterpret_cast<const T*>(a.bg) + c0, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) w[4 + q] = v[q];
    }
    tm_st16(tw + 16, w);  // [bx | bg]
    tm_st16(tp, z);
    tm_st16(tp + 16, z);
    tm_st16(tp + 32, z);
    tm_wait_st();
  }
  __syncthreads();

  const float invH = 1.0f / (float)a.Hl;
  const bool tail = c0 + kGateE > a.Hl;  // this thread owns padding columns (written as zeros)
  T* dZrow = reinterpret_cast<T*>(a.dZ) + ((size_t)b0 * a.T + t) * 2 * H;
  const size_t dZstep = (size_t)a.T * 2 * H;
  int issued = min(S, nrows);
  bool aborted = false;
  int s = 0;          // stage of row i
  uint32_t ph = 0;    // parity of that stage's current phase
  for (int i = 0; i < nrows; ++i, dZrow += dZstep) {
    const bool ok = mbar_wait_bounded(smem_u32(&full[s]), ph, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                      (volatile int*)&abort_flag);
    const float4 sr = st_row[i];
    // Pass 1: du, dg and the normalised halves stay in registers for pass 2
    // (zeros for a lane with no columns or a row that never landed, assigned
    // on that path only, so that the common path carries no zeroing).
    float2 kdu[4], kUh[4], kdg[4], kGh[4];
    float2 rs[4];
    float2 wa[8], wb[8];  // [wx | wg], [bx | bg]
    tm_ld32(tw, wa, wb);
    if (!(ok && active)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) kdu[q] = kUh[q] = kdg[q] = kGh[q] = rs[q] = f2(0.f);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) rs[q] = f2(0.f);
      const T* st = reinterpret_cast<const T*>(ring + (size_t)s * row_bytes);
      float2 dhv[4], zu[4], zg[4];
      ld8<T>(st + c0, dhv);
      ld8<T>(st + H + c0, zu);
      ld8<T>(st + 2 * H + c0, zg);
      const float2 sU = f2(sr.x), cU = f2(sr.y), sG = f2(sr.z), cG = f2(sr.w);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 w0 = wa[q], w1 = wb[q], w2 = wa[4 + q], w3 = wb[4 + q];
        const float2 Uh = fma2(zu[q], sU, cU);
        const float2 Gh = fma2(zg[q], sG, cG);
        const float2 u = fma2(w0, Uh, w1);
        const float2 g = fma2(w2, Gh, w3);
        const float2 sg = sigmoid_fast2(g);
        const float2 gs = mul2(g, sg);
        const float2 du = mul2(dhv[q], gs);
        // silu'(g) = s + g s (1 - s) = s + (gs - gs * s)
        const float2 dsilu = add2(sg, fma2(gs, make_float2(-sg.x, -sg.y), gs));
        const float2 dg = mul2(mul2(dhv[q], u), dsilu);
        const float2 gU = mul2(w0, du), gG = mul2(w2, dg);
        rs[0] = add2(rs[0], gU);
        rs[1] = fma2(gU, Uh, rs[1]);
        rs[2] = add2(rs[2], gG);
        rs[3] = fma2(gG, Gh, rs[3]);
        kdu[q] = du;
        kUh[q] = Uh;
        kdg[q] = dg;
        kGh[q] = Gh;
      }
    }
    // Row sums over the CTA: per warp, then over the warps in a fixed order.
    float* rb = red + (i & 1) * kGateRedWarps * NS;
    {
      const float rsum[NS] = {rs[0].x + rs[0].y, rs[1].x + rs[1].y, rs[2].x + rs[2].y, rs[3].x + rs[3].y};
      const float k = warp_sum_transposed<NS>(rsum);
      if (lane % LPS == 0) rb[warp * NS + lane / LPS] = k;
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid == 0 && issued < nrows) issue(issued++, s);
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
    // (After the barrier: the TMEM round trips of the partial updates then
    // overlap the other warps' arrival instead of delaying it.)
    {
      // Column partials of dwx, dbx, then dwg, dbg (inactive lanes add zeros).
      // The previous row's store of the db1 partials has long been issued:
      // waiting for it here rather than at the end of that row costs little.
      tm_wait_st();
      float2 p[8];
      tm_ld16(tp, p);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p[q] = fma2(kdu[q], kUh[q], p[q]);
        p[4 + q] = add2(p[4 + q], kdu[q]);
      }
      tm_st16(tp, p);
      tm_ld16(tp + 16, p);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p[q] = fma2(kdg[q], kGh[q], p[q]);
        p[4 + q] = add2(p[4 + q], kdg[q]);
      }
      tm_st16(tp + 16, p);
    }
    float m[NS];
    {
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
    float2 oU[4], oG[4];
    tm_ld16(tw, wa);
    if (!active) {
#pragma unroll
      for (int q = 0; q < 4; ++q) oU[q] = oG[q] = f2(0.f);
    } else {
      const float sU = sr.x, sG = sr.z;
      const float2 pU = f2(-m[1]), qU = f2(-sU * m[0]);
      const float2 pG = f2(-m[3]), qG = f2(-sG * m[2]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 gU = mul2(wa[q], kdu[q]), gG = mul2(wa[4 + q], kdg[q]);
        oU[q] = fma2(f2(sU), fma2(pU, kUh[q], gU), qU);
        oG[q] = fma2(f2(sG), fma2(pG, kGh[q], gG), qG);
      }
      if (tail) {  // padding columns are written as zeros
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = c0 + 2 * q;
          if (c >= a.Hl) oU[q].x = oG[q].x = 0.f;
          if (c + 1 >= a.Hl) oU[q].y = oG[q].y = 0.f;
        }
      }
      st8<T>(dZrow + c0, oU);
      st8<T>(dZrow + H + c0, oG);
    }
    {
      // db1 partials of the U and G halves.
      float2 p[8];
      tm_ld16(tp + 32, p);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p[q] = add2(p[q], oU[q]);
        p[4 + q] = add2(p[4 + q], oG[q]);
      }
      tm_st16(tp + 32, p);
    }
  }

  if (aborted) {
    tm_wait_st();
    // Wait (bounded) for the copies still in flight before the CTA's shared
    // memory goes away: the newest copy issued into each stage.
    if (tid == 0) {
      volatile int no_abort = 0;
      for (int i = max(0, issued - S); i < issued; ++i) {
        mbar_wait_bounded(smem_u32(&full[i % S]), (uint32_t)((i / S) & 1), kWaitLimitNs, a.err,
                          ERRBIT_WAIT_ROWS, &no_abort);
      }
    }
  } else {
    float2 p0[8], p1[8], p2[8];
    tm_wait_st();
    tm_ld16(tp, p0);
    tm_ld16(tp + 16, p1);
    tm_ld16(tp + 32, p2);
    if (active) {
      const size_t pr = (size_t)bblk * a.T + t;
      auto put = [&](float* dst, const float2* v) {
        *reinterpret_cast<float4*>(dst) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
      };
      put(a.pwx + pr * H + c0, p0);
      put(a.pbx + pr * H + c0, p0 + 4);
      put(a.pwg + pr * H + c0, p1);
      put(a.pbg + pr * H + c0, p1 + 4);
      put(a.pb1 + pr * 2 * H + c0, p2);
      put(a.pb1 + pr * 2 * H + H + c0, p2 + 4);
    }
  }
  // Every thread's tensor-memory accesses are complete: free the columns.
  tm_fence_before();
  __syncthreads();
  if (warp == 0) {
    tm_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(a.tmem_cols) : "memory");
  }
}

// The tensor-memory columns a CTA of `threads` allocates (80 per warp of a
// lane quarter, a power of two of at least 32), and the ring sized for the
// CTAs per SM those columns allow.
int gate_tm_cols(int threads) {
  const int per_quarter = ((threads / 32) + 3) / 4;
  int cols = 32;
  while (cols < 80 * per_quarter) cols *= 2;
  return cols;
}
int sm_smem_bytes() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) return 0;
  return v;
}
template <typename T>
size_t gate_tm_shape(int H, int nb, int& threads, int& stages) {
  threads = (H / kGateE + 31) / 32 * 32;
  const size_t fixed = (size_t)nb * 16 + 2 * kGateRedWarps * 4 * 4;
  const size_t row_bytes = (size_t)3 * H * sizeof(T);
  // As many CTAs per SM as the tensor memory holds (two, or one for rows
  // wider than 2560), each with its reservation and static shared memory.
  const int ctas = 512 / gate_tm_cols(threads);
  const int cap = ctas >= 2 ? sm_smem_bytes() / 2 - 2048 : max_dynamic_smem_bytes() - 1024;
  const long long room = ((long long)cap - (long long)fixed) / (long long)(row_bytes + 8);
  if (room < 2) return 0;
  stages = (int)(room < kGateMaxStages ? room : kGateMaxStages);
  return fixed + (size_t)stages * row_bytes + (size_t)stages * 8;
}
template <typename T>
int gate_tm_ctas_per_sm(int H) {
  int threads = 0, stages = 0;
  const size_t smem = gate_tm_shape<T>(H, kGateBwdMaxRows, threads, stages);
  if (smem == 0) return 1;
  auto k = k_gate_bwd_tm<T>;
  int n = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess || n < 1)
    return 1;
  const int by_tmem = 512 / gate_tm_cols(threads);
  return n < by_tmem ? n : by_tmem;
}
template <typename T>
cudaError_t launch_tm(const GateBwdArgs& base, cudaStream_t st, dim3 grid) {
  GateBwdArgs a = base;
  int threads = 0;
  const size_t smem = gate_tm_shape<T>(a.H, a.nb, threads, a.stages);
  if (smem == 0) return cudaErrorInvalidValue;
  a.tmem_cols = gate_tm_cols(threads);
  auto k = k_gate_bwd_tm<T>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(k, grid, dim3(threads), smem, st, 1, a);
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

// CTAs per SM of each form and the form a shape takes: the TMEM form for
// rows the register form cannot hold (H > 2560), else only where the
// register form holds one CTA per SM and there are at least 96 rows per SM
// (measured at the block's shapes: the register form is faster at B <= 128
// with T = 64, D = 1280, and at H = 1536, where it holds two CTAs per SM).
// The runtime's occupancy query reports one CTA per SM for the TMEM form
// although the SM holds two (the profiler's occupancy limits and its
// achieved warps per SM both show two).  The grid is sized for the two that
// run from 192 rows per SM up, for the query's one below (measured: two
// faster at B = 512 and 1024 with T = 64, one faster at B = 256).
struct GateForm {
  bool tm;
  int ctas;
};
GateForm gate_form(const RowArgs& ra) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, std::pair<int, int>> cache;  // (tm, register) CTAs per SM
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return {true, 1};
  const bool wide = ra.H / kGateE > 320;
  std::pair<int, int> n;
  {
    const auto key = std::make_tuple(dev, ra.dtype, ra.H);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      n = it->second;
    } else {
      n.first = ra.dtype == 0   ? gate_tm_ctas_per_sm<float>(ra.H)
                : ra.dtype == 1 ? gate_tm_ctas_per_sm<bf16>(ra.H)
                                : gate_tm_ctas_per_sm<f16>(ra.H);
      n.second = wide ? 0
                 : ra.dtype == 0 ? gate_ctas_per_sm<float, true>(ra.H)
                 : ra.dtype == 1 ? gate_ctas_per_sm<bf16, true>(ra.H)
                                 : gate_ctas_per_sm<f16, true>(ra.H);
      cache[key] = n;
    }
  }
  if (wide) return {true, n.first};
  const long long rows_per_sm = (long long)ra.B * ra.T / (sm_count() > 0 ? sm_count() : 1);
  if (n.second < 2 && rows_per_sm >= 96) {
    const int resident = 512 / gate_tm_cols((ra.H / kGateE + 31) / 32 * 32);
    return {true, rows_per_sm >= 192 && resident > n.first ? resident : n.first};
  }
  return {false, n.second};
}

}  // namespace

int gate_bwd_ctas_per_sm(const RowArgs& ra) { return gate_form(ra).ctas; }

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
  a.tmem_cols = 0;
  if (!a.err) return cudaErrorInvalidValue;
  const dim3 grid(ra.nbblk, ra.T);
  if (gate_form(ra).tm) {
    if (ra.dtype == 0) return launch_tm<float>(a, st, grid);
    if (ra.dtype == 1) return launch_tm<bf16>(a, st, grid);
    return launch_tm<f16>(a, st, grid);
  }
  if (ra.dtype == 0) return launch_typed<float, true>(a, st, grid);
  if (ra.dtype == 1) return launch_typed<bf16, true>(a, st, grid);
  return launch_typed<f16, true>(a, st, grid);
}

}  // namespace rmx
