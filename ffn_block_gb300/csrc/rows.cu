// Row passes of the RankMixer block: the three outer LayerNorms (with the
// token mix folded into how two of them read or write their rows), the
// LN-gated SiLU of the FFN, their backwards, and the deterministic column
// reductions of the parameter gradients.
//
// Operation: page "Subgraph-fusion-based Mega-kernel Generation", section
// "Exact computation".  LN(z) = (z - mean) / sqrt(mean((z - mean)^2) + eps)
// * gamma + beta over the last axis; token mixing = reshape [B,T,T,D/T] and
// swap the two T axes, i.e. m[b,i,j*C+c] = a[b,j,i*C+c] with C = D/T.
//
// All statistics and arithmetic are float32; tensors are read and written in
// the storage type T with 16-byte vector accesses where rows allow it.
// Every reduction runs in a fixed order (no float atomics), so results are
// bitwise repeatable.

#include "common.cuh"
#include "pairs.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {

namespace {

#define RMX_DISPATCH_T(dtype, ...)                 \
  do {                                             \
    if ((dtype) == 0) {                            \
      typedef float T;                             \
      __VA_ARGS__;                                 \
    } else if ((dtype) == 1) {                     \
      typedef bf16 T;                              \
      __VA_ARGS__;                                 \
    } else {                                       \
      typedef f16 T;                               \
      __VA_ARGS__;                                 \
    }                                              \
  } while (0)

inline int elem_bytes(int dtype) { return dtype == 0 ? 4 : 2; }
inline int vec_elems(int dtype) { return 16 / elem_bytes(dtype); }


// -------------------------------------------------------------------------
// Token mix as an addressing rule.  Mixing moves column d = i*C + c of row j
// to row i, column j*C + c (within one sample); it is its own inverse.  The
// forward writes norm0's output rows already mixed, and the backward of norm1
// writes its gradient rows both as they are and mixed, so every LayerNorm
// pass reads and writes whole rows.
// -------------------------------------------------------------------------
// Columns d >= Dl (the zero padding of a row of pitch D) stay in row j and
// are written as zeros.
template <typename T, int V>
__device__ __forceinline__ void store_mixed(T* sample_base, const float* v, int j, int d0, int C, int D, int Dl) {
  int i = d0 / C, c = d0 - i * C;
  if ((C & 1) == 0) {
    // d0 even and C even: elements (e, e+1) always share a chunk (and Dl,
    // a multiple of C, is even).
#pragma unroll
    for (int e = 0; e < V; e += 2) {
      const bool pad = d0 + e >= Dl;
      T pr[2] = {from_f<T>(pad ? 0.f : v[e]), from_f<T>(pad ? 0.f : v[e + 1])};
      T* dst = pad ? sample_base + (size_t)j * D + d0 + e : sample_base + (size_t)i * D + j * C + c;
      if (sizeof(T) == 2) *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(pr);
      else *reinterpret_cast<float2*>(dst) = make_float2(pad ? 0.f : v[e], pad ? 0.f : v[e + 1]);
      c += 2;
      while (c >= C) { c -= C; ++i; }
    }
  } else {
#pragma unroll
    for (int e = 0; e < V; ++e) {
      if (d0 + e >= Dl) sample_base[(size_t)j * D + d0 + e] = from_f<T>(0.f);
      else sample_base[(size_t)i * D + j * C + c] = from_f<T>(v[e]);
      if (++c == C) { c = 0; ++i; }
    }
  }
}

// =========================================================================
// LayerNorm forward, one warp per row, the row held in registers as 16-byte
// vectors (lane owns vectors lane + 32 q, MAXV >= ceil(D / V / 32)):
//   LNF_PLAIN      y = LN(s)                       (norm2)
//   LNF_MIXED_OUT  y = LN(s), written token-mixed  (norm0: a0 -> mix)
//   LNF_SUM_IN     y = LN(s + s_add)               (norm1: mix + x)
// Saves the row mean and 1/sqrt(var + eps).  Rows of pitch D hold Dl real
// columns followed by zeros; the statistics cover the real columns.  The
// grid is persistent (the warps stride over the rows); each CTA first stages
// gamma and beta in shared memory as fp32, a float4 {g, g', b, b'} per column
// pair laid out [pair k of the vector][vector].  The arithmetic runs on
// column pairs with the packed fp32x2 instructions.
// =========================================================================
template <typename T, int MODE, int MAXV>
__global__ void __launch_bounds__(256) k_ln_fwd(const T* __restrict__ s, const T* __restrict__ s_add,
                                                const T* __restrict__ g, const T* __restrict__ be,
                                                T* __restrict__ y, float* __restrict__ mu, float* __restrict__ rs,
                                                T* __restrict__ s_out, int N, int Tn, int D, int C, float eps,
                                                int Dl) {
  pdl_enter();
  constexpr int V = VecN<T>::value;
  constexpr int P = V / 2;
  extern __shared__ float4 gsm[];  // [P][nv]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const int nv = D / V;
  for (int idx = threadIdx.x; idx < P * nv; idx += blockDim.x) {
    const int k = idx / nv, vi = idx - k * nv, c = vi * V + 2 * k;
    gsm[k * nv + vi] = make_float4(to_f(g[c]), to_f(g[c + 1]), to_f(be[c]), to_f(be[c + 1]));
  }
  __syncthreads();
  const bool padded = Dl != D;
  const float invD = 1.0f / (float)Dl;
  // The row stays in registers: packed as loaded when it is one tensor, as
  // fp32 pairs when it is the sum of two.
  constexpr bool SUM = MODE == LNF_SUM_IN;
  for (int row = blockIdx.x * wpb + warp; row < N; row += gridDim.x * wpb) {
    const T* srow = s + (size_t)row * D;
    uint4 raw[SUM ? 1 : MAXV];
    float2 vf[SUM ? MAXV : 1][P];
    auto get = [&](int q, float2* v) {
      if (SUM) {
#pragma unroll
        for (int k = 0; k < P; ++k) v[k] = vf[q][k];
      } else {
        ld16p<T>(&raw[q], v);
      }
    };
    float2 sum2 = f2(0.f);
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int vi = lane + 32 * q;
      if (vi < nv) {
        if (SUM) {
          float2 a[P];
          ld16p<T>(srow + vi * V, vf[q]);
          ld16p<T>(s_add + (size_t)row * D + vi * V, a);
#pragma unroll
          for (int k = 0; k < P; ++k) {
            vf[q][k] = add2(vf[q][k], a[k]);
            if constexpr (sizeof(T) == 2) vf[q][k] = unpack2w<T>(pack2w<T>(vf[q][k]));  // the stored s1
          }
        } else {
          raw[q] = *reinterpret_cast<const uint4*>(srow + vi * V);
        }
        float2 v[P];
        get(q, v);
#pragma unroll
        for (int k = 0; k < P; ++k) sum2 = add2(sum2, v[k]);
      }
    }
    const float mean = warp_sum(sum2.x + sum2.y) * invD;
    const float2 nm = f2(-mean);
    float2 q2 = f2(0.f);
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int vi = lane + 32 * q;
      if (vi < nv) {
        float2 v[P];
        get(q, v);
#pragma unroll
        for (int k = 0; k < P; ++k) {
          float2 c = add2(v[k], nm);
          if (padded) {
            if (vi * V + 2 * k >= Dl) c.x = 0.f;
            if (vi * V + 2 * k + 1 >= Dl) c.y = 0.f;
          }
          q2 = fma2(c, c, q2);
        }
      }
    }
    const float rstd = 1.0f / sqrtf(warp_sum(q2.x + q2.y) * invD + eps);
    const float2 r2 = f2(rstd);
    const int b = row / Tn, j = row - b * Tn;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int vi = lane + 32 * q;
      if (vi < nv) {
        float2 v[P], o[P];
        get(q, v);
#pragma unroll
        for (int k = 0; k < P; ++k) {
          const float4 w = gsm[k * nv + vi];
          o[k] = fma2(mul2(add2(v[k], nm), r2), make_float2(w.x, w.y), make_float2(w.z, w.w));
        }
        if (MODE == LNF_MIXED_OUT)
          store_mixed<T, V>(y + (size_t)b * Tn * D, reinterpret_cast<const float*>(o), j, vi * V, C, D, Dl);
        else st16p<T>(y + (size_t)row * D + vi * V, o);
        if (SUM) st16p<T>(s_out + (size_t)row * D + vi * V, v);
      }
    }
    if (lane == 0) {
      mu[row] = mean;
      rs[row] = rstd;
    }
  }
}

// =========================================================================
// Z statistics for the FFMA path: one warp per (row, 256-column tile) of
// Z = [U | G]; {mean, M2} of the tile's U columns and of its G columns, from
// the stored values (the tensor-core GEMM writes the same numbers from its
// epilogue).
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(256) k_zstats(const T* __restrict__ Z, float* __restrict__ zstats, int N, int H,
                                                int tiles) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (item >= (long long)N * tiles) return;
  const int r = (int)(item / tiles), j = (int)(item - (long long)r * tiles);
  const T* zr = Z + (size_t)r * 2 * H;
  float s[2] = {0.f, 0.f}, n[2] = {0.f, 0.f};
  float v[kZStatsTile / 32];
#pragma unroll
  for (int q = 0; q < kZStatsTile / 32; ++q) {
    const int col = j * kZStatsTile + lane + 32 * q;
    v[q] = col < 2 * H ? to_f(zr[col]) : 0.f;
    if (col < 2 * H) {
      const int h = col < H ? 0 : 1;
      s[h] += v[q];
      n[h] += 1.f;
    }
  }
  float mean[2], m2[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float tot = warp_sum(s[h]), cnt = warp_sum(n[h]);
    mean[h] = cnt > 0.f ? tot / cnt : 0.f;
  }
#pragma unroll
  for (int q = 0; q < kZStatsTile / 32; ++q) {
    const int col = j * kZStatsTile + lane + 32 * q;
    if (col < 2 * H) {
      const int h = col < H ? 0 : 1;
      m2[h] += (v[q] - mean[h]) * (v[q] - mean[h]);
    }
  }
  m2[0] = warp_sum(m2[0]);
  m2[1] = warp_sum(m2[1]);
  if (lane == 0)
    *reinterpret_cast<float4*>(zstats + ((size_t)r * tiles + j) * 4) = make_float4(mean[0], m2[0], mean[1], m2[1]);
}

// =========================================================================
// F3: hidden = LN_x(U) * silu(LN_gate(G)), Z = [U | G], one warp per row.
// The warp first merges the row's group statistics (lane l takes groups l,
// l+32, ... in order with Chan, Golub and LeVeque's pairwise update, then
// the lanes merge pairwise in a fixed order, so every lane holds the same
// bits), writes mean and 1/sqrt(var + eps) of U and G for the backward, and
// then streams the row: lane l owns the 16-byte vectors l, l+32, ... of both
// halves.  Each lane's next kGateFwdDepth vectors are in flight through
// cp.async into a per-warp shared-memory buffer (the first before the
// statistics merge), which keeps several row loads per warp outstanding
// without the registers a deeper unroll would take.
// =========================================================================
// Row r's statistics of U and G from its group statistics (every lane of
// the warp ends with the same bits); lane 0 writes them for the backward.
// Z rows of pitch 2H whose halves hold Hl real columns and H - Hl zeros: the
// merged statistics then cover H values per half, and are converted to the
// Hl real ones (same sum; the zeros add nothing to the sum of squares).
__device__ __forceinline__ void gate_row_stats(const float* __restrict__ zstats, long long r, int H, int Hl,
                                               float eps, float* __restrict__ muU, float* __restrict__ rU,
                                               float* __restrict__ muG, float* __restrict__ rG, float& sU,
                                               float& cU, float& sG, float& cG) {
  const int lane = threadIdx.x & 31;
  const int tiles = zstats_tiles(H);
  Moments u = {0.f, 0.f, 0.f}, g = {0.f, 0.f, 0.f};
  for (int j = lane; j < tiles; j += 32) {
    const float4 t = *reinterpret_cast<const float4*>(zstats + ((size_t)r * tiles + j) * 4);
    const int lo = j * kZStatsTile, hi = min(2 * H, lo + kZStatsTile);
    const float nu = (float)max(0, min(H, hi) - lo);
    const float ng = (float)max(0, hi - max(H, lo));
    if (nu > 0.f) u = merge_moments(u, Moments{nu, t.x, t.y});
    if (ng > 0.f) g = merge_moments(g, Moments{ng, t.z, t.w});
  }
  u = warp_merge_moments(u);
  g = warp_merge_moments(g);
  if (Hl != H) {
    auto real_only = [&](Moments& m) {
      const float mean = m.mean * ((float)H / (float)Hl);
      m.m2 = fmaxf(m.m2 + (float)H * m.mean * m.mean - (float)Hl * mean * mean, 0.f);
      m.mean = mean;
    };
    real_only(u);
    real_only(g);
  }
  sU = 1.0f / sqrtf(u.m2 / (float)Hl + eps);
  sG = 1.0f / sqrtf(g.m2 / (float)Hl + eps);
  if (lane == 0) {
    muU[r] = u.mean;
    rU[r] = sU;
    muG[r] = g.mean;
    rG[r] = sG;
  }
  cU = -u.mean * sU;
  cG = -g.mean * sG;
}

// cp.async (16 bytes, bypassing L1) into shared memory and its group waits.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kGateFwdDepth = 3;  // iterations of each lane's Z vectors in flight

template <typename T>
__global__ void __launch_bounds__(256, 5) k_gate_fwd(const T* __restrict__ Z, const float* __restrict__ zstats,
                                                  float* __restrict__ muU, float* __restrict__ rU,
                                                  float* __restrict__ muG, float* __restrict__ rG,
                                                  const T* __restrict__ wx, const T* __restrict__ bx,
                                                  const T* __restrict__ wg, const T* __restrict__ bg,
                                                  T* __restrict__ hidden, int N, int H, float eps, int Hl) {
  pdl_enter();
  constexpr int V = VecN<T>::value;
  // Per warp: kGateFwdDepth slots x (U, G) x 32 lanes x 16 bytes.
  __shared__ __align__(16) unsigned char zbuf[8][kGateFwdDepth][2][32 * 16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * (blockDim.x >> 5) + warp;
  if (r >= N) return;
  const T* zr = Z + (size_t)r * 2 * H;
  const int nv = H / V;
  const int iters = nv > lane ? (nv - lane + 31) / 32 : 0;
  // Each lane copies, and later reads, only its own 16-byte slots.
  auto fetch = [&](int it) {
    if (it < iters) {
      const int h0 = (lane + 32 * it) * V;
      const int sl = it % kGateFwdDepth;
      cp_async16(smem_u32(&zbuf[warp][sl][0][lane * 16]), zr + h0);
      cp_async16(smem_u32(&zbuf[warp][sl][1][lane * 16]), zr + H + h0);
    }
    cp_async_commit();  // an empty group keeps the counting uniform
  };
#pragma unroll
  for (int it = 0; it < kGateFwdDepth; ++it) fetch(it);
  float sU, cU, sG, cG;
  gate_row_stats(zstats, r, H, Hl, eps, muU, rU, muG, rG, sU, cU, sG, cG);
  T* hr = hidden + (size_t)r * H;
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    cp_async_wait<kGateFwdDepth - 1>();  // this iteration's group has landed
    const int h0 = (lane + 32 * it) * V;
    const int sl = it % kGateFwdDepth;
    float zu[V], zg[V], fwx[V], fbx[V], fwg[V], fbg[V], o[V];
    load_vec(reinterpret_cast<const T*>(&zbuf[warp][sl][0][lane * 16]), zu);
    load_vec(reinterpret_cast<const T*>(&zbuf[warp][sl][1][lane * 16]), zg);
    load_vec(wx + h0, fwx);
    load_vec(bx + h0, fbx);
    load_vec(wg + h0, fwg);
    load_vec(bg + h0, fbg);
#pragma unroll
    for (int e = 0; e < V; ++e) {
      const float uu = fmaf(fmaf(zu[e], sU, cU), fwx[e], fbx[e]);
      const float gg = fmaf(fmaf(zg[e], sG, cG), fwg[e], fbg[e]);
      o[e] = uu * (gg * sigmoid_fast(gg));
    }
    // Refill the slot just read: its values are consumed above, so this
    // lane's shared-memory reads of it are complete.
    fetch(it + kGateFwdDepth);
    store_vec(hr + h0, o);
  }
  cp_async_wait<0>();
}

// =========================================================================
// F3 with the statistics taken in-pass (16-bit rows of at most
// kGateRowVecs 16-byte vectors per half and lane, H <= 2560): one warp per
// row holds the row's U and G halves in registers as loaded (packed), takes
// the statistics of each half in one pass over the registers (sums and sums
// of squares shifted by the half's first element; padded rows: the mean, then
// the centred sum of squares over the Hl real columns), writes them and
// hidden = LN_x(U) * silu(LN_gate(G)).  The GEMM that produces Z then needs
// no statistics epilogue.  Every lane's loads are issued before the first
// use, so a warp has its whole row (10 KB at H = 2560) in flight.  The grid
// is persistent (two CTAs per SM, the warps striding over the rows); each
// CTA first stages the four LayerNorm weight vectors in shared memory as
// fp32, a float4 {w, w', b, b'} per column pair laid out [LN][pair k of the
// vector][vector], so that the lanes of a warp read consecutive 16 bytes.
// =========================================================================
constexpr int kGateRowVecs = 10;

template <typename T>
__global__ void __launch_bounds__(256, 2) k_gate_fwd_rows(const T* __restrict__ Z, float* __restrict__ muU,
                                                          float* __restrict__ rU, float* __restrict__ muG,
                                                          float* __restrict__ rG, const T* __restrict__ wx,
                                                          const T* __restrict__ bx, const T* __restrict__ wg,
                                                          const T* __restrict__ bg, T* __restrict__ hidden, int N,
                                                          int H, float eps, int Hl) {
  pdl_enter();
  constexpr int V = 8;  // 16-bit: eight columns per 16-byte vector
  extern __shared__ float4 wsm[];  // [2][4][nv]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nv = H / V;
  for (int idx = threadIdx.x; idx < 4 * nv; idx += blockDim.x) {
    const int k = idx / nv, vi = idx - k * nv, c = vi * V + 2 * k;
    wsm[k * nv + vi] = make_float4(to_f(wx[c]), to_f(wx[c + 1]), to_f(bx[c]), to_f(bx[c + 1]));
    wsm[(4 + k) * nv + vi] = make_float4(to_f(wg[c]), to_f(wg[c + 1]), to_f(bg[c]), to_f(bg[c + 1]));
  }
  __syncthreads();
  const bool padded = Hl != H;
  for (int r = blockIdx.x * (blockDim.x >> 5) + warp; r < N; r += gridDim.x * (blockDim.x >> 5)) {
  const T* zr = Z + (size_t)r * 2 * H;
  uint4 u[kGateRowVecs], g[kGateRowVecs];
#pragma unroll
  for (int q = 0; q < kGateRowVecs; ++q) {
    const int vi = lane + 32 * q;
    if (vi < nv) {
      u[q] = __ldcs(reinterpret_cast<const uint4*>(zr + vi * V));
      g[q] = __ldcs(reinterpret_cast<const uint4*>(zr + H + vi * V));
    }
  }
  auto pairs = [](const uint4& w, float2 (&p)[4]) { ld8<T>(reinterpret_cast<const T*>(&w), p); };
  const float inv = 1.0f / (float)Hl;
  float mU, mG, sU, sG;
  if (!padded) {
    // One pass over the registers: sums and sums of squares of each half
    // shifted by its first element (lane 0's, a value of the row's scale,
    // so that the difference of the two moments loses little).
    float2 a0[4], b0[4];
    pairs(u[0], a0);
    pairs(g[0], b0);
    const float2 nkU = f2(-__shfl_sync(0xffffffffu, a0[0].x, 0));
    const float2 nkG = f2(-__shfl_sync(0xffffffffu, b0[0].x, 0));
    float2 su = f2(0.f), sg = f2(0.f), qu = f2(0.f), qg = f2(0.f);
#pragma unroll
    for (int q = 0; q < kGateRowVecs; ++q) {
      if (lane + 32 * q < nv) {
        float2 a[4], b[4];
        pairs(u[q], a);
        pairs(g[q], b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 du = add2(a[k], nkU), dg = add2(b[k], nkG);
          su = add2(su, du);
          qu = fma2(du, du, qu);
          sg = add2(sg, dg);
          qg = fma2(dg, dg, qg);
        }
      }
    }
    const float dmU = warp_sum(su.x + su.y) * inv, dmG = warp_sum(sg.x + sg.y) * inv;
    const float vU = fmaxf(warp_sum(qu.x + qu.y) * inv - dmU * dmU, 0.f);
    const float vG = fmaxf(warp_sum(qg.x + qg.y) * inv - dmG * dmG, 0.f);
    mU = dmU - nkU.x;
    mG = dmG - nkG.x;
    sU = 1.0f / sqrtf(vU + eps);
    sG = 1.0f / sqrtf(vG + eps);
  } else {
    // Padded rows: the mean, then the centred sum of squares over the real
    // columns (the padding columns hold zeros).
    float2 su = f2(0.f), sg = f2(0.f);
#pragma unroll
    for (int q = 0; q < kGateRowVecs; ++q) {
      if (lane + 32 * q < nv) {
        float2 a[4], b[4];
        pairs(u[q], a);
        pairs(g[q], b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          su = add2(su, a[k]);
          sg = add2(sg, b[k]);
        }
      }
    }
    mU = warp_sum(su.x + su.y) * inv;
    mG = warp_sum(sg.x + sg.y) * inv;
    float2 qu = f2(0.f), qg = f2(0.f);
    const float2 nmU = f2(-mU), nmG = f2(-mG);
#pragma unroll
    for (int q = 0; q < kGateRowVecs; ++q) {
      const int vi = lane + 32 * q;
      if (vi < nv) {
        float2 a[4], b[4];
        pairs(u[q], a);
        pairs(g[q], b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float2 du = add2(a[k], nmU), dg = add2(b[k], nmG);
          const int c = vi * V + 2 * k;
          if (c >= Hl) du.x = dg.x = 0.f;
          if (c + 1 >= Hl) du.y = dg.y = 0.f;
          qu = fma2(du, du, qu);
          qg = fma2(dg, dg, qg);
        }
      }
    }
    sU = 1.0f / sqrtf(warp_sum(qu.x + qu.y) * inv + eps);
    sG = 1.0f / sqrtf(warp_sum(qg.x + qg.y) * inv + eps);
  }
  if (lane == 0) {
    muU[r] = mU;
    rU[r] = sU;
    muG[r] = mG;
    rG[r] = sG;
  }
  const float2 sU2 = f2(sU), cU2 = f2(-mU * sU), sG2 = f2(sG), cG2 = f2(-mG * sG);
  T* hr = hidden + (size_t)r * H;
#pragma unroll
  for (int q = 0; q < kGateRowVecs; ++q) {
    const int vi = lane + 32 * q;
    if (vi < nv) {
      const int h0 = vi * V;
      float2 a[4], b[4], o[4];
      pairs(u[q], a);
      pairs(g[q], b);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 wu = wsm[k * nv + vi], wgt = wsm[(4 + k) * nv + vi];
        const float2 uu = fma2(fma2(a[k], sU2, cU2), make_float2(wu.x, wu.y), make_float2(wu.z, wu.w));
        const float2 gg = fma2(fma2(b[k], sG2, cG2), make_float2(wgt.x, wgt.y), make_float2(wgt.z, wgt.w));
        o[k] = mul2(uu, mul2(gg, sigmoid_fast2(gg)));
      }
      st8<T>(hr + h0, o);
    }
  }
  }
}

// =========================================================================
// R: column sums of partials, several jobs per launch, fixed summation order.
//
// Cluster form (every J a multiple of 4): one launch of clusters of
// kColsumCluster CTAs of 256 threads, each cluster within one job.  A job of
// more than kColsumWideRows partial rows takes one cluster per 128 columns (a
// float4 per lane): CTA r sums rows [r*cr, r*cr + cr), cr = ceil(P / 8),
// warp w rows w, w+8, ... of them with four loads in flight, the eight warps
// combined in order; the CTAs' sums go to CTA 0 of the cluster through
// distributed shared memory, which adds them in rank order and writes the
// result.  A job of few rows (per-token bias gradients summed over a few
// sample blocks) is summed wide: each warp takes 128 columns of all rows.
// One-pass form (some J not a multiple of 4): block (32, 16), x the column,
// y a stripe of rows p = y, y+16, ..., stripes combined in order.
// =========================================================================
constexpr int kColsumCluster = 8;
constexpr int kColsumCols = 128;  // columns per cluster or per warp (32 lanes x float4)
constexpr int kColsumWideRows = 32;

struct ColsumArgs {
  ColsumJob job[kMaxColsumJobs];
  int ncg[kMaxColsumJobs];           // column groups of kColsumCols
  int wide[kMaxColsumJobs];          // 1: summed wide
  int block_start[kMaxColsumJobs + 1];
  int njobs;
};

__device__ __forceinline__ int colsum_job_of(const ColsumArgs& a) {
  int jb = 0;
  while (jb + 1 < a.njobs && (int)blockIdx.x >= a.block_start[jb + 1]) ++jb;
  return jb;
}

template <typename T>
__device__ __forceinline__ void store4(void* out, int j, float4 v) {
  T* o = reinterpret_cast<T*>(out) + j;
  o[0] = from_f<T>(v.x);
  o[1] = from_f<T>(v.y);
  o[2] = from_f<T>(v.z);
  o[3] = from_f<T>(v.w);
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ __forceinline__ void cs_cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cs_cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cs_cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cs_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Stores v at the shared address `addr` (this CTA's view) of CTA `rank` of the cluster.
__device__ __forceinline__ void cs_st_cluster_f4(uint32_t addr, uint32_t rank, float4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// Sum of rows p, p + 8, ... below p1 of the four columns at col (J floats
// per row), four loads in flight.
__device__ __forceinline__ float4 colsum_rows(const float* col, size_t J, int p, int p1) {
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (; p + 24 < p1; p += 32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = add4(acc[k], *reinterpret_cast<const float4*>(col + (size_t)(p + 8 * k) * J));
  }
#pragma unroll
  for (int k = 0; k < 3; ++k)
    if (p + 8 * k < p1) acc[k] = add4(acc[k], *reinterpret_cast<const float4*>(col + (size_t)(p + 8 * k) * J));
  return add4(add4(acc[0], acc[1]), add4(acc[2], acc[3]));
}

template <typename T>
__global__ void __launch_bounds__(256) k_colsums_cluster(const ColsumArgs a) {
  pdl_enter();
  __shared__ float4 part[8][32];
  __shared__ float4 chunk[kColsumCluster][32];
  const int jb = colsum_job_of(a);
  const ColsumJob& job = a.job[jb];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int local = (int)blockIdx.x - a.block_start[jb];
  const size_t J = (size_t)job.J;
  if (a.wide[jb]) {  // the whole cluster: no exchange
    const int j = (local * 8 + warp) * kColsumCols + lane * 4;
    if (j >= job.J) return;
    const float* col = job.part + j;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    int p = 0;
    for (; p + 3 < job.P; p += 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = add4(acc[k], *reinterpret_cast<const float4*>(col + (size_t)(p + k) * J));
    }
    for (; p < job.P; ++p) acc[0] = add4(acc[0], *reinterpret_cast<const float4*>(col + (size_t)p * J));
    store4<T>(job.out, j, add4(add4(acc[0], acc[1]), add4(acc[2], acc[3])));
    return;
  }
  // CTA 0's shared memory is written only once every CTA of the cluster is
  // known to be running: arrive now, wait before the first remote store.
  cs_cluster_arrive_relaxed();
  const uint32_t r = cs_cluster_rank();
  const int cg = local / kColsumCluster;
  const int j = cg * kColsumCols + lane * 4;
  const int cr = (job.P + kColsumCluster - 1) / kColsumCluster;
  const int p0 = (int)r * cr, p1 = min(job.P, p0 + cr);
  part[warp][lane] = j < job.J ? colsum_rows(job.part + j, J, p0 + warp, p1) : make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  cs_cluster_wait_acquire();
  if (warp == 0) {
    float4 tot = part[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) tot = add4(tot, part[w][lane]);
    cs_st_cluster_f4(smem_u32(&chunk[r][lane]), 0u, tot);
  }
  cs_cluster_arrive_release();
  cs_cluster_wait_acquire();
  if (r == 0 && warp == 0 && j < job.J) {
    float4 tot = chunk[0][lane];
#pragma unroll
    for (int k = 1; k < kColsumCluster; ++k) tot = add4(tot, chunk[k][lane]);
    store4<T>(job.out, j, tot);
  }
}

template <typename T>
__global__ void __launch_bounds__(512) k_colsums_onepass(const ColsumArgs a) {
  pdl_enter();
  __shared__ float part[16][33];
  const int jb = colsum_job_of(a);
  const ColsumJob& job = a.job[jb];
  const int j = (blockIdx.x - a.block_start[jb]) * 32 + threadIdx.x;
  float s = 0.f;
  if (j < job.J) {
    for (int p = threadIdx.y; p < job.P; p += 16) s += job.part[(size_t)p * job.J + j];
  }
  part[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && j < job.J) {
    float tot = 0.f;
#pragma unroll
    for (int y = 0; y < 16; ++y) tot += part[y][threadIdx.x];
    reinterpret_cast<T*>(job.out)[j] = from_f<T>(tot);
  }
}

}  // namespace

int max_dynamic_smem_bytes() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return v;
}

cudaError_t launch_ln_fwd(const RowArgs& a, int mode, const void* s, const void* s_add, const void* g,
                          const void* be, void* y, float* mu, float* rs, void* s_out, cudaStream_t st) {
  const int N = a.B * a.T;
  if (N == 0) return cudaSuccess;
  const int nv = a.D / vec_elems(a.dtype);
  const int q = (nv + 31) / 32;
  const size_t smem = (size_t)a.D / 2 * sizeof(float4);  // a float4 per column pair
  // Persistent grid: as many 8-row CTAs as fit at once (registers bound it
  // near four per SM; the staged parameters take at most 40 KB).
  const int fit = 4 * sm_count();
  const int grid = (N + 7) / 8 < fit ? (N + 7) / 8 : fit;
  const int C = a.Dl / a.T;
  cudaError_t err = cudaSuccess;
#define RMX_LNF(M, MAXV)                                                                                    \
  RMX_DISPATCH_T(a.dtype, {                                                                                 \
    err = launch_k(k_ln_fwd<T, M, MAXV>, dim3(grid), dim3(256), smem, st, 1, (const T*)s, (const T*)s_add,  \
                   (const T*)g, (const T*)be, (T*)y, mu, rs, (T*)s_out, N, a.T, a.D, C, 1e-3f, a.Dl);       \
  })
#define RMX_LNF_Q(M)                          \
  if (q <= 1) RMX_LNF(M, 1);                  \
  else if (q <= 2) RMX_LNF(M, 2);             \
  else if (q <= 4) RMX_LNF(M, 4);             \
  else if (q <= 6) RMX_LNF(M, 6);             \
  else if (q <= 10) RMX_LNF(M, 10);           \
  else return cudaErrorInvalidValue;
  if (mode == LNF_PLAIN) { RMX_LNF_Q(LNF_PLAIN) }
  else if (mode == LNF_MIXED_OUT) { RMX_LNF_Q(LNF_MIXED_OUT) }
  else { RMX_LNF_Q(LNF_SUM_IN) }
#undef RMX_LNF_Q
#undef RMX_LNF
  return err;
}

cudaError_t launch_zstats(const RowArgs& a, const void* Z, float* zstats, cudaStream_t st) {
  const int N = a.B * a.T;
  const int tiles = zstats_tiles(a.H);
  const long long items = (long long)N * tiles;
  const int grid = (int)((items + 7) / 8);
  cudaError_t err = cudaSuccess;
  RMX_DISPATCH_T(a.dtype, {
    err = launch_k(k_zstats<T>, dim3(grid), dim3(256), 0, st, 1, (const T*)Z, zstats, N, a.H, tiles);
  });
  return err;
}

bool gate_fwd_rows_supported(const RowArgs& a) {
  return a.dtype != 0 && a.H % 8 == 0 && a.H / 8 <= 32 * kGateRowVecs;
}

cudaError_t launch_gate_fwd_rows(const RowArgs& a, const void* Z, float* muU, float* rU, float* muG, float* rG,
                                 const void* wx, const void* bx, const void* wg, const void* bg, void* hidden,
                                 cudaStream_t st) {
  if (!gate_fwd_rows_supported(a)) return cudaErrorInvalidValue;
  const int N = a.B * a.T;
  if (N == 0) return cudaSuccess;
  const size_t smem = (size_t)a.H * 4 * sizeof(float);  // 8 * (H / 8) float4
  const int ctas = (N + 7) / 8 < 2 * sm_count() ? (N + 7) / 8 : 2 * sm_count();
  if (a.dtype == 1)
    return launch_k(k_gate_fwd_rows<bf16>, dim3(ctas), dim3(256), smem, st, 1, (const bf16*)Z, muU, rU, muG, rG,
                    (const bf16*)wx, (const bf16*)bx, (const bf16*)wg, (const bf16*)bg, (bf16*)hidden, N, a.H,
                    1e-5f, a.Hl);
  return launch_k(k_gate_fwd_rows<f16>, dim3(ctas), dim3(256), smem, st, 1, (const f16*)Z, muU, rU, muG, rG,
                  (const f16*)wx, (const f16*)bx, (const f16*)wg, (const f16*)bg, (f16*)hidden, N, a.H, 1e-5f,
                  a.Hl);
}

cudaError_t launch_gate_fwd(const RowArgs& a, const void* Z, const float* zstats, float* muU, float* rU,
                            float* muG, float* rG, const void* wx, const void* bx, const void* wg, const void* bg,
                            void* hidden, cudaStream_t st) {
  const int N = a.B * a.T;
  cudaError_t err = cudaSuccess;
  RMX_DISPATCH_T(a.dtype, {
    err = launch_k(k_gate_fwd<T>, dim3((N + 7) / 8), dim3(256), 0, st, 1, (const T*)Z, zstats, muU, rU, muG, rG,
                   (const T*)wx, (const T*)bx, (const T*)wg, (const T*)bg, (T*)hidden, N, a.H, 1e-5f, a.Hl);
  });
  return err;
}

namespace {
// Fills the launch arguments; returns false for the one-pass form.
bool colsum_plan(const ColsumJob* jobs, int njobs, ColsumArgs& a) {
  a.njobs = njobs;
  bool cluster = true;
  for (int i = 0; i < njobs; ++i) cluster = cluster && jobs[i].J % 4 == 0 && jobs[i].P > 0;
  int blocks = 0;
  for (int i = 0; i < njobs; ++i) {
    a.job[i] = jobs[i];
    a.ncg[i] = (jobs[i].J + kColsumCols - 1) / kColsumCols;
    a.wide[i] = cluster && jobs[i].P <= kColsumWideRows ? 1 : 0;
    a.block_start[i] = blocks;
    if (!cluster) {
      blocks += (jobs[i].J + 31) / 32;
    } else if (a.wide[i]) {
      const int nb = (a.ncg[i] + 7) / 8;  // eight warps of 128 columns per CTA
      blocks += (nb + kColsumCluster - 1) / kColsumCluster * kColsumCluster;
    } else {
      blocks += a.ncg[i] * kColsumCluster;
    }
  }
  a.block_start[njobs] = blocks;
  return cluster;
}
}  // namespace

cudaError_t launch_colsums(const ColsumJob* jobs, int njobs, int dtype, cudaStream_t st) {
  if (njobs <= 0 || njobs > kMaxColsumJobs) return cudaErrorInvalidValue;
  ColsumArgs a;
  const bool cluster = colsum_plan(jobs, njobs, a);
  const int blocks = a.block_start[njobs];
  if (blocks == 0) return cudaSuccess;
  cudaError_t err = cudaSuccess;
  if (!cluster) {
    RMX_DISPATCH_T(dtype, { err = launch_k(k_colsums_onepass<T>, dim3(blocks), dim3(32, 16), 0, st, 1, a); });
    return err;
  }
  RMX_DISPATCH_T(dtype, {
    err = launch_k(k_colsums_cluster<T>, dim3(blocks), dim3(256), 0, st, kColsumCluster, a);
  });
  return err;
}

}  // namespace rmx
