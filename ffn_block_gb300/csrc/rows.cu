// Row passes of the RankMixer block: the three outer LayerNorms with the
// token mix and residuals, the LN-gated SiLU of the FFN, their backwards, and
// the deterministic column reductions of the parameter gradients.
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
#include "kernels.h"

namespace rmx {

namespace {

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

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
inline int round32(int v) { return (v + 31) / 32 * 32; }


// =========================================================================
// F1: norm0 -> token mix -> + x -> norm1, one CTA per sample b.
// x[b] ([T,D], storage type) is staged in shared memory; warp w handles rows
// w, w + nwarps, ...; each lane keeps its columns k = lane + 32 q in
// registers (MAXQ >= ceil(D/32)).
// =========================================================================
template <typename T, int MAXQ>
__global__ void __launch_bounds__(256) k_ln0_mix_ln1_fwd(
    const T* __restrict__ x, const T* __restrict__ g0, const T* __restrict__ be0,
    const T* __restrict__ g1, const T* __restrict__ be1, T* __restrict__ out1,
    float* __restrict__ mu0, float* __restrict__ r0, float* __restrict__ mu1,
    float* __restrict__ r1, int Tn, int D, int C, float eps) {
  extern __shared__ __align__(16) unsigned char sm[];
  T* xs = reinterpret_cast<T*>(sm);
  float* smu = reinterpret_cast<float*>(sm + align16((size_t)Tn * D * sizeof(T)));
  float* srs = smu + Tn;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const size_t base = (size_t)b * Tn * D;

  const int n16 = (int)((size_t)Tn * D * sizeof(T) / 16);
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  for (int i = threadIdx.x; i < n16; i += blockDim.x) reinterpret_cast<uint4*>(xs)[i] = src[i];
  __syncthreads();

  const float invD = 1.0f / (float)D;
  // norm0 statistics of every row j of x[b].
  for (int j = warp; j < Tn; j += nw) {
    float v[MAXQ];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < MAXQ; ++q) {
      const int k = lane + 32 * q;
      v[q] = (k < D) ? to_f(xs[j * D + k]) : 0.f;
      s += v[q];
    }
    const float mean = warp_sum(s) * invD;
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < MAXQ; ++q) {
      const int k = lane + 32 * q;
      const float c = v[q] - mean;
      ss += (k < D) ? c * c : 0.f;
    }
    const float rstd = 1.0f / sqrtf(warp_sum(ss) * invD + eps);
    if (lane == 0) {
      smu[j] = mean;
      srs[j] = rstd;
      mu0[(size_t)b * Tn + j] = mean;
      r0[(size_t)b * Tn + j] = rstd;
    }
  }
  __syncthreads();

  // Row i of s1 = token_mix(norm0(x))[i] + x[i]; element k = j*C + c comes
  // from row j, column d = i*C + c of norm0(x).
  for (int i = warp; i < Tn; i += nw) {
    float v[MAXQ];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < MAXQ; ++q) {
      const int k = lane + 32 * q;
      float val = 0.f;
      if (k < D) {
        const int j = k / C, c = k - j * C, d = i * C + c;
        const float a0 = (to_f(xs[j * D + d]) - smu[j]) * srs[j] * to_f(g0[d]) + to_f(be0[d]);
        val = a0 + to_f(xs[i * D + k]);
      }
      v[q] = val;
      s += val;
    }
    const float mean = warp_sum(s) * invD;
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < MAXQ; ++q) {
      const int k = lane + 32 * q;
      const float c = v[q] - mean;
      ss += (k < D) ? c * c : 0.f;
    }
    const float rstd = 1.0f / sqrtf(warp_sum(ss) * invD + eps);
    T* orow = out1 + base + (size_t)i * D;
#pragma unroll
    for (int q = 0; q < MAXQ; ++q) {
      const int k = lane + 32 * q;
      if (k < D) orow[k] = from_f<T>((v[q] - mean) * rstd * to_f(g1[k]) + to_f(be1[k]));
    }
    if (lane == 0) {
      mu1[(size_t)b * Tn + i] = mean;
      r1[(size_t)b * Tn + i] = rstd;
    }
  }
}

// =========================================================================
// F5: y = LN(s) for every row (norm2).  One warp per row, 16-byte vectors;
// lane owns vectors lane + 32 q (MAXV >= ceil(D / V / 32)).
// =========================================================================
template <typename T, int MAXV>
__global__ void __launch_bounds__(256) k_ln_rows_fwd(const T* __restrict__ s, const T* __restrict__ g,
                                                     const T* __restrict__ be, T* __restrict__ y,
                                                     float* __restrict__ mu, float* __restrict__ rs,
                                                     int N, int D, float eps) {
  constexpr int V = VecN<T>::value;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= N) return;
  const int nv = D / V;
  const T* srow = s + (size_t)row * D;
  float v[MAXV][V];
  float sum = 0.f;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int vi = lane + 32 * q;
    if (vi < nv) {
      load_vec(srow + vi * V, v[q]);
#pragma unroll
      for (int e = 0; e < V; ++e) sum += v[q][e];
    }
  }
  const float invD = 1.0f / (float)D;
  const float mean = warp_sum(sum) * invD;
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int vi = lane + 32 * q;
    if (vi < nv) {
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float c = v[q][e] - mean;
        ss += c * c;
      }
    }
  }
  const float rstd = 1.0f / sqrtf(warp_sum(ss) * invD + eps);
  T* yrow = y + (size_t)row * D;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int vi = lane + 32 * q;
    if (vi < nv) {
      float gg[V], bb[V], o[V];
      load_vec(g + vi * V, gg);
      load_vec(be + vi * V, bb);
#pragma unroll
      for (int e = 0; e < V; ++e) o[e] = (v[q][e] - mean) * rstd * gg[e] + bb[e];
      store_vec(yrow + vi * V, o);
    }
  }
  if (lane == 0) {
    mu[row] = mean;
    rs[row] = rstd;
  }
}

// -------------------------------------------------------------------------
// Row streaming for the per-token passes.  Each CTA walks a list of rows; its
// first thread keeps S rows in flight with cp.async.bulk copies into a ring
// of shared-memory stages (one mbarrier per stage, completion counted in
// bytes).  A stage is refilled right after the block-wide reduction of the
// row that used it, when every thread has finished reading it.  Waits are
// bounded; a wait that gives up sets the device error word and the block
// leaves the loop together after its next barrier.
// -------------------------------------------------------------------------
constexpr int kRingStages = 4;
constexpr uint64_t kRowWaitLimitNs = 2000ull * 1000ull * 1000ull;

struct RowRing {
  uint32_t base;        // shared address of stage 0
  uint32_t stage_bytes; // bytes per stage (multiple of 128)
  uint32_t bars;        // shared address of the S mbarriers
  __device__ uint32_t stage(int i) const { return base + (uint32_t)(i % kRingStages) * stage_bytes; }
  __device__ uint32_t bar(int i) const { return bars + 8u * (uint32_t)(i % kRingStages); }
};

__device__ __forceinline__ RowRing ring_setup(unsigned char* sm, uint32_t stage_bytes, volatile int* abort_flag) {
  RowRing r;
  r.base = smem_u32(sm);
  r.stage_bytes = stage_bytes;
  r.bars = r.base + kRingStages * stage_bytes;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingStages; ++i) mbar_init(r.bars + 8u * i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  return r;
}

// Thread 0: after an abort, wait (bounded) for the copies still in flight so
// the CTA does not exit while they write its shared memory.
__device__ __forceinline__ void ring_drain(const RowRing& r, int consumed, int issued, unsigned int* err) {
  if (threadIdx.x != 0) return;
  volatile int no_abort = 0;
  for (int j = consumed; j < issued; ++j)
    mbar_wait_bounded(r.bar(j), (uint32_t)(j / kRingStages) & 1u, 50ull * 1000ull * 1000ull, err,
                      ERRBIT_WAIT_DRAIN, &no_abort);
}

__host__ __device__ inline uint32_t ring_stage_bytes(size_t row_bytes) { return (uint32_t)((row_bytes + 127) / 128 * 128); }
inline size_t ring_smem_bytes(size_t row_bytes) { return (size_t)kRingStages * ring_stage_bytes(row_bytes) + 64; }

// =========================================================================
// Z statistics for the FFMA path: one warp per (row, 256-column tile) of
// Z = [U | G]; {mean, M2} of the tile's U columns and of its G columns, from
// the stored values (the tensor-core GEMM writes the same numbers from its
// epilogue).
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(256) k_zstats(const T* __restrict__ Z, float* __restrict__ zstats, int N, int H,
                                                int tiles) {
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
// F3: hidden = LN_x(U) * silu(LN_gate(G)), Z = [U | G] per row.  A CTA takes
// `rpc` rows: first one thread per row merges the row's tile statistics
// (Chan, Golub and LeVeque's pairwise update, tiles in order) into mean and
// 1/sqrt(var + eps) of U and G; then thread v handles columns v*V .. v*V+V-1
// of both halves of every row, so the pass is one read of Z and one write of
// hidden with no per-row barrier.
// =========================================================================
constexpr int kGateRows = 16;

template <typename T>
__global__ void __launch_bounds__(512) k_gate_fwd(const T* __restrict__ Z, const float* __restrict__ zstats,
                                                  const T* __restrict__ wx, const T* __restrict__ bx,
                                                  const T* __restrict__ wg, const T* __restrict__ bg,
                                                  T* __restrict__ hidden, float* __restrict__ muU,
                                                  float* __restrict__ rU, float* __restrict__ muG,
                                                  float* __restrict__ rG, int N, int H, float eps) {
  constexpr int V = VecN<T>::value;
  __shared__ float st[kGateRows][4];
  const int r0 = blockIdx.x * kGateRows;
  const int nrows = min(kGateRows, N - r0);
  const int tiles = zstats_tiles(H);
  if ((int)threadIdx.x < nrows) {
    const int r = r0 + threadIdx.x;
    Moments u = {0.f, 0.f, 0.f}, g = {0.f, 0.f, 0.f};
    for (int j = 0; j < tiles; ++j) {
      const float4 t = *reinterpret_cast<const float4*>(zstats + ((size_t)r * tiles + j) * 4);
      const int lo = j * kZStatsTile, hi = min(2 * H, lo + kZStatsTile);
      const float nu = (float)max(0, min(H, hi) - lo);
      const float ng = (float)max(0, hi - max(H, lo));
      if (nu > 0.f) u = merge_moments(u, Moments{nu, t.x, t.y});
      if (ng > 0.f) g = merge_moments(g, Moments{ng, t.z, t.w});
    }
    const float rsu = 1.0f / sqrtf(u.m2 / (float)H + eps);
    const float rsg = 1.0f / sqrtf(g.m2 / (float)H + eps);
    st[threadIdx.x][0] = u.mean;
    st[threadIdx.x][1] = rsu;
    st[threadIdx.x][2] = g.mean;
    st[threadIdx.x][3] = rsg;
    muU[r] = u.mean;
    rU[r] = rsu;
    muG[r] = g.mean;
    rG[r] = rsg;
  }
  __syncthreads();
  const int nv = H / V;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const int h0 = v * V;
    float fwx[V], fbx[V], fwg[V], fbg[V];
    load_vec(wx + h0, fwx);
    load_vec(bx + h0, fbx);
    load_vec(wg + h0, fwg);
    load_vec(bg + h0, fbg);
#pragma unroll 4
    for (int i = 0; i < nrows; ++i) {
      const T* zr = Z + (size_t)(r0 + i) * 2 * H;
      float u[V], g[V], o[V];
      load_vec(zr + h0, u);
      load_vec(zr + H + h0, g);
      const float mU = st[i][0], sU = st[i][1], mG = st[i][2], sG = st[i][3];
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float uu = (u[e] - mU) * sU * fwx[e] + fbx[e];
        const float gg = (g[e] - mG) * sG * fwg[e] + fbg[e];
        o[e] = uu * (gg / (1.0f + expf(-gg)));
      }
      store_vec(hidden + (size_t)(r0 + i) * H + h0, o);
    }
  }
}

// =========================================================================
// G1: backward of norm2.  CTA (bblk, t) handles rows (b, t) for b in its
// block; thread v owns columns d = v*V ...  With g = gamma2 * dy and
// xh = (s2 - mean) * rstd:
//   ds2 = rstd * (g - mean(g) - xh * mean(g * xh)),
//   dgamma2 += dy * xh, dbeta2 += dy, dbout[t] += ds2 (per-CTA partials).
// Rows stream through the shared-memory ring (dy row, then s2 row).
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(512) k_ln2_bwd(const T* __restrict__ dy, const T* __restrict__ s2,
                                                 const float* __restrict__ mu2, const float* __restrict__ r2,
                                                 const T* __restrict__ g2, T* __restrict__ ds2,
                                                 float* __restrict__ pg2, float* __restrict__ pb2,
                                                 float* __restrict__ pbo, int B, int Tn, int D, int nb,
                                                 unsigned int* err) {
  constexpr int V = VecN<T>::value;
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ float red[2 * 32 * 2];
  __shared__ int abort_flag;
  const size_t half = (size_t)D * sizeof(T);
  const RowRing ring = ring_setup(sm, ring_stage_bytes(2 * half), &abort_flag);
  int slot = 0;
  const int bblk = blockIdx.x, t = blockIdx.y;
  const int v = threadIdx.x;
  const bool act = v * V < D;
  const int d0 = v * V;
  float gam[V], ag[V], ab[V], ao[V];
#pragma unroll
  for (int e = 0; e < V; ++e) ag[e] = ab[e] = ao[e] = 0.f;
  if (act) load_vec(g2 + d0, gam);
  const float invD = 1.0f / (float)D;
  const int b0 = bblk * nb;
  const int nrows = max(0, min(B, b0 + nb) - b0);
  auto issue = [&](int i) {
    const size_t r = (size_t)(b0 + i) * Tn + t;
    mbar_arrive_expect_tx(ring.bar(i), (uint32_t)(2 * half));
    bulk_g2s(ring.stage(i), dy + r * D, (uint32_t)half, ring.bar(i));
    bulk_g2s(ring.stage(i) + (uint32_t)half, s2 + r * D, (uint32_t)half, ring.bar(i));
  };
  int issued = 0;
  if (v == 0)
    for (; issued < min(kRingStages, nrows); ++issued) issue(issued);
  int i = 0;
  for (; i < nrows; ++i) {
    mbar_wait_bounded(ring.bar(i), (uint32_t)(i / kRingStages) & 1u, kRowWaitLimitNs, err, ERRBIT_WAIT_PRODUCER,
                      &abort_flag);
    const T* st = reinterpret_cast<const T*>(sm + (size_t)(i % kRingStages) * ring.stage_bytes);
    const size_t r = (size_t)(b0 + i) * Tn + t;
    const float mean = mu2[r], rstd = r2[r];
    float dyv[V], xh[V], g[V];
    float sums[2] = {0.f, 0.f};
    if (act) {
      float sv[V];
      load_vec(st + d0, dyv);
      load_vec(st + D + d0, sv);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        xh[e] = (sv[e] - mean) * rstd;
        g[e] = gam[e] * dyv[e];
        sums[0] += g[e];
        sums[1] += g[e] * xh[e];
      }
    }
    block_sum<2>(sums, red, slot);
    if (abort_flag) break;
    if (v == 0 && issued < nrows) {
      fence_proxy_async_smem();
      issue(issued++);
    }
    const float mg = sums[0] * invD, mgx = sums[1] * invD;
    if (act) {
      float o[V];
#pragma unroll
      for (int e = 0; e < V; ++e) {
        o[e] = rstd * (g[e] - mg - xh[e] * mgx);
        ag[e] += dyv[e] * xh[e];
        ab[e] += dyv[e];
        ao[e] += o[e];
      }
      store_vec(ds2 + r * D + d0, o);
    }
  }
  if (abort_flag) ring_drain(ring, i, issued, err);
  if (act) {
    const size_t p = (size_t)bblk * Tn + t;
#pragma unroll
    for (int e = 0; e < V; ++e) {
      pg2[p * D + d0 + e] = ag[e];
      pb2[p * D + d0 + e] = ab[e];
      pbo[p * D + d0 + e] = ao[e];
    }
  }
}

// =========================================================================
// G4: backward of hidden = LN_x(U) * silu(LN_gate(G)).  With Uh, Gh the
// normalised halves, u = wx*Uh + bx, g = wg*Gh + bg, s = sigmoid(g):
//   du = dh * g * s,  dg = dh * u * s * (1 + g * (1 - s)),
//   gU = wx * du,     gG = wg * dg,
//   dU = rU * (gU - mean(gU) - Uh * mean(gU * Uh)), same for dG,
//   dZ = [dU | dG];   dwx += du*Uh, dbx += du, dwg += dg*Gh, dbg += dg,
//   db1[t] += dZ.
// Two streaming passes: (1) one warp per row takes the four row sums
// (sum gU, sum gU*Uh, sum gG, sum gG*Gh); (2) CTA (bblk, t), thread v owns
// columns v*V ... of both halves for every row of its block, writes dZ and
// keeps the column partial sums in registers.  No per-row barrier.
// =========================================================================
template <int E>
__device__ __forceinline__ void gate_bwd_elem(const float* dhv, const float* zu, const float* zg, float mU, float sU,
                                              float mG, float sG, const float* fwx, const float* fbx,
                                              const float* fwg, const float* fbg, float* Uh, float* Gh, float* du,
                                              float* dg) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    Uh[e] = (zu[e] - mU) * sU;
    Gh[e] = (zg[e] - mG) * sG;
    const float u = fwx[e] * Uh[e] + fbx[e];
    const float g = fwg[e] * Gh[e] + fbg[e];
    const float sg = 1.0f / (1.0f + expf(-g));
    du[e] = dhv[e] * (g * sg);
    dg[e] = dhv[e] * u * (sg * (1.0f + g * (1.0f - sg)));
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_gate_bwd_rowsums(
    const T* __restrict__ dh, const T* __restrict__ Z, const float* __restrict__ muU, const float* __restrict__ rU,
    const float* __restrict__ muG, const float* __restrict__ rG, const T* __restrict__ wx,
    const T* __restrict__ bx, const T* __restrict__ wg, const T* __restrict__ bg, float* __restrict__ rowsum, int N,
    int H) {
  constexpr int V = VecN<T>::value;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= N) return;
  const float mU = muU[r], sU = rU[r], mG = muG[r], sG = rG[r];
  const T* dhr = dh + (size_t)r * H;
  const T* zr = Z + (size_t)r * 2 * H;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const int nv = H / V;
#pragma unroll 2
  for (int v = lane; v < nv; v += 32) {
    const int h0 = v * V;
    float dhv[V], zu[V], zg[V], fwx[V], fbx[V], fwg[V], fbg[V];
    load_vec(dhr + h0, dhv);
    load_vec(zr + h0, zu);
    load_vec(zr + H + h0, zg);
    load_vec(wx + h0, fwx);
    load_vec(bx + h0, fbx);
    load_vec(wg + h0, fwg);
    load_vec(bg + h0, fbg);
    float Uh[V], Gh[V], du[V], dg[V];
    gate_bwd_elem<V>(dhv, zu, zg, mU, sU, mG, sG, fwx, fbx, fwg, fbg, Uh, Gh, du, dg);
#pragma unroll
    for (int e = 0; e < V; ++e) {
      const float gU = fwx[e] * du[e], gG = fwg[e] * dg[e];
      a0 += gU;
      a1 += gU * Uh[e];
      a2 += gG;
      a3 += gG * Gh[e];
    }
  }
  a0 = warp_sum(a0);
  a1 = warp_sum(a1);
  a2 = warp_sum(a2);
  a3 = warp_sum(a3);
  if (lane == 0) *reinterpret_cast<float4*>(rowsum + (size_t)r * 4) = make_float4(a0, a1, a2, a3);
}

// Thread owns E = 4 columns of each half (8-byte accesses for 16-bit types)
// so the six column partial sums fit in registers at good occupancy;
// blockIdx.z picks which part of the H columns the CTA covers.
template <typename T>
__global__ void __launch_bounds__(512) k_gate_bwd_apply(
    const T* __restrict__ dh, const T* __restrict__ Z, const float* __restrict__ muU, const float* __restrict__ rU,
    const float* __restrict__ muG, const float* __restrict__ rG, const float* __restrict__ rowsum,
    const T* __restrict__ wx, const T* __restrict__ bx, const T* __restrict__ wg, const T* __restrict__ bg,
    T* __restrict__ dZ, float* __restrict__ pwx, float* __restrict__ pbx, float* __restrict__ pwg,
    float* __restrict__ pbg, float* __restrict__ pb1, int B, int Tn, int H, int nb) {
  constexpr int E = 4;
  const int bblk = blockIdx.x, t = blockIdx.y;
  const int h0 = (blockIdx.z * blockDim.x + threadIdx.x) * E;
  if (h0 >= H) return;
  const float invH = 1.0f / (float)H;
  float fwx[E], fbx[E], fwg[E], fbg[E];
  load_n<T, E>(wx + h0, fwx);
  load_n<T, E>(bx + h0, fbx);
  load_n<T, E>(wg + h0, fwg);
  load_n<T, E>(bg + h0, fbg);
  float awx[E], abx[E], awg[E], abg[E], a1u[E], a1g[E];
#pragma unroll
  for (int e = 0; e < E; ++e) awx[e] = abx[e] = awg[e] = abg[e] = a1u[e] = a1g[e] = 0.f;
  const int b_end = min(B, (bblk + 1) * nb);
#pragma unroll 2
  for (int b = bblk * nb; b < b_end; ++b) {
    const size_t r = (size_t)b * Tn + t;
    float dhv[E], zu[E], zg[E];
    load_n<T, E>(dh + r * H + h0, dhv);
    load_n<T, E>(Z + r * 2 * H + h0, zu);
    load_n<T, E>(Z + r * 2 * H + H + h0, zg);
    const float4 rs = *reinterpret_cast<const float4*>(rowsum + r * 4);
    const float sU = rU[r], sG = rG[r];
    float Uh[E], Gh[E], du[E], dg[E], oU[E], oG[E];
    gate_bwd_elem<E>(dhv, zu, zg, muU[r], sU, muG[r], sG, fwx, fbx, fwg, fbg, Uh, Gh, du, dg);
    const float m0 = rs.x * invH, m1 = rs.y * invH, m2 = rs.z * invH, m3 = rs.w * invH;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      oU[e] = sU * (fwx[e] * du[e] - m0 - Uh[e] * m1);
      oG[e] = sG * (fwg[e] * dg[e] - m2 - Gh[e] * m3);
      awx[e] += du[e] * Uh[e];
      abx[e] += du[e];
      awg[e] += dg[e] * Gh[e];
      abg[e] += dg[e];
      a1u[e] += oU[e];
      a1g[e] += oG[e];
    }
    store_n<T, E>(dZ + r * 2 * H + h0, oU);
    store_n<T, E>(dZ + r * 2 * H + H + h0, oG);
  }
  const size_t p = (size_t)bblk * Tn + t;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    pwx[p * H + h0 + e] = awx[e];
    pbx[p * H + h0 + e] = abx[e];
    pwg[p * H + h0 + e] = awg[e];
    pbg[p * H + h0 + e] = abg[e];
    pb1[p * 2 * H + h0 + e] = a1u[e];
    pb1[p * 2 * H + H + h0 + e] = a1g[e];
  }
}

// =========================================================================
// G7: backward of norm1, the token mix and norm0 for one sample b per CTA.
// x[b] is staged in shared memory; s1 = token_mix(norm0(x)) + x is
// recomputed from it and the saved statistics.  Thread v owns columns
// k = v*V ... of every row.  Row sums are deferred: a first sweep writes one
// partial per (row, warp), a second sweep finishes the rows, so each phase
// needs one barrier instead of one per row.
//   phase A: ds1 = LN1-backward(dout1)                  -> scratch (fp32)
//   phase B: da0 = token_mix(ds1) (the mix is its own inverse),
//            dx = ds1 + LN0-backward(da0)
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(512) k_ln1_mix_ln0_bwd(
    const T* __restrict__ x, const T* __restrict__ dout1, const float* __restrict__ mu0,
    const float* __restrict__ r0, const float* __restrict__ mu1, const float* __restrict__ r1,
    const T* __restrict__ g0, const T* __restrict__ be0, const T* __restrict__ g1, float* ds1,
    T* __restrict__ dx, float* __restrict__ pg0, float* __restrict__ pb0, float* __restrict__ pg1,
    float* __restrict__ pbe1, int Tn, int D, int C) {
  constexpr int V = VecN<T>::value;
  extern __shared__ __align__(16) unsigned char sm[];
  T* xs = reinterpret_cast<T*>(sm);
  float* s_mu0 = reinterpret_cast<float*>(sm + align16((size_t)Tn * D * sizeof(T)));
  float* s_r0 = s_mu0 + Tn;
  float* s_mu1 = s_r0 + Tn;
  float* s_r1 = s_mu1 + Tn;
  float* red = s_r1 + Tn;  // [Tn][nw][2]
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = blockDim.x >> 5;
  const size_t base = (size_t)b * Tn * D;

  const int n16 = (int)((size_t)Tn * D * sizeof(T) / 16);
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  for (int i = tid; i < n16; i += blockDim.x) reinterpret_cast<uint4*>(xs)[i] = src[i];
  for (int i = tid; i < Tn; i += blockDim.x) {
    s_mu0[i] = mu0[(size_t)b * Tn + i];
    s_r0[i] = r0[(size_t)b * Tn + i];
    s_mu1[i] = mu1[(size_t)b * Tn + i];
    s_r1[i] = r1[(size_t)b * Tn + i];
  }
  __syncthreads();

  const bool act = tid * V < D;
  const int k0 = tid * V;
  const float invD = 1.0f / (float)D;
  float gam0[V], gam1[V];
  if (act) {
    load_vec(g0 + k0, gam0);
    load_vec(g1 + k0, gam1);
  }

  // xh1 of row i for this thread's columns (recomputed from x).
  auto xhat1 = [&](int i, float* xh) {
#pragma unroll
    for (int e = 0; e < V; ++e) {
      const int k = k0 + e;
      const int j = k / C, c = k - j * C, d = i * C + c;
      const float a0 = (to_f(xs[j * D + d]) - s_mu0[j]) * s_r0[j] * to_f(g0[d]) + to_f(be0[d]);
      const float s1 = a0 + to_f(xs[i * D + k]);
      xh[e] = (s1 - s_mu1[i]) * s_r1[i];
    }
  };
  // da0 of row j = token_mix(ds1)[j]: element k' = i*C + c is ds1[i, j*C + c].
  auto gather_da0 = [&](int j, float* da) {
#pragma unroll
    for (int e = 0; e < V; ++e) {
      const int kp = k0 + e;
      const int i = kp / C, c = kp - i * C;
      da[e] = ds1[base + (size_t)i * D + j * C + c];
    }
  };

  // ---- phase A, sweep 1: row partial sums of g = gamma1*dout1 and g*xh1.
  for (int i = 0; i < Tn; ++i) {
    float ps = 0.f, psx = 0.f;
    if (act) {
      float xh[V], d1[V];
      xhat1(i, xh);
      load_vec(dout1 + base + (size_t)i * D + k0, d1);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float g = gam1[e] * d1[e];
        ps += g;
        psx += g * xh[e];
      }
    }
    ps = warp_sum(ps);
    psx = warp_sum(psx);
    if (lane == 0) {
      red[(i * nw + warp) * 2 + 0] = ps;
      red[(i * nw + warp) * 2 + 1] = psx;
    }
  }
  __syncthreads();
  // ---- phase A, sweep 2: ds1 rows and the norm1 parameter partials.
  {
    float ag[V], ab[V];
#pragma unroll
    for (int e = 0; e < V; ++e) ag[e] = ab[e] = 0.f;
    for (int i = 0; i < Tn; ++i) {
      float t0 = 0.f, t1 = 0.f;
      for (int w = 0; w < nw; ++w) {
        t0 += red[(i * nw + w) * 2 + 0];
        t1 += red[(i * nw + w) * 2 + 1];
      }
      if (act) {
        const float mg = t0 * invD, mgx = t1 * invD, rs = s_r1[i];
        float xh[V], d1[V];
        xhat1(i, xh);
        load_vec(dout1 + base + (size_t)i * D + k0, d1);
        float* drow = ds1 + base + (size_t)i * D + k0;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float g = gam1[e] * d1[e];
          drow[e] = rs * (g - mg - xh[e] * mgx);
          ag[e] += d1[e] * xh[e];
          ab[e] += d1[e];
        }
      }
    }
    if (act) {
#pragma unroll
      for (int e = 0; e < V; ++e) {
        pg1[(size_t)b * D + k0 + e] = ag[e];
        pbe1[(size_t)b * D + k0 + e] = ab[e];
      }
    }
  }
  __syncthreads();  // ds1 of this sample is complete and visible to the block

  // ---- phase B, sweep 1: row partial sums for norm0's backward.
  for (int j = 0; j < Tn; ++j) {
    float ps = 0.f, psx = 0.f;
    if (act) {
      float da[V];
      gather_da0(j, da);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float xh0 = (to_f(xs[j * D + k0 + e]) - s_mu0[j]) * s_r0[j];
        const float g = gam0[e] * da[e];
        ps += g;
        psx += g * xh0;
      }
    }
    ps = warp_sum(ps);
    psx = warp_sum(psx);
    if (lane == 0) {
      red[(j * nw + warp) * 2 + 0] = ps;
      red[(j * nw + warp) * 2 + 1] = psx;
    }
  }
  __syncthreads();
  // ---- phase B, sweep 2: dx rows and the norm0 parameter partials.
  {
    float ag[V], ab[V];
#pragma unroll
    for (int e = 0; e < V; ++e) ag[e] = ab[e] = 0.f;
    for (int j = 0; j < Tn; ++j) {
      float t0 = 0.f, t1 = 0.f;
      for (int w = 0; w < nw; ++w) {
        t0 += red[(j * nw + w) * 2 + 0];
        t1 += red[(j * nw + w) * 2 + 1];
      }
      if (act) {
        const float mg = t0 * invD, mgx = t1 * invD, rs = s_r0[j];
        float da[V], o[V];
        gather_da0(j, da);
        const float* drow = ds1 + base + (size_t)j * D + k0;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float xh0 = (to_f(xs[j * D + k0 + e]) - s_mu0[j]) * s_r0[j];
          const float g = gam0[e] * da[e];
          o[e] = drow[e] + rs * (g - mg - xh0 * mgx);
          ag[e] += da[e] * xh0;
          ab[e] += da[e];
        }
        store_vec(dx + base + (size_t)j * D + k0, o);
      }
    }
    if (act) {
#pragma unroll
      for (int e = 0; e < V; ++e) {
        pg0[(size_t)b * D + k0 + e] = ag[e];
        pb0[(size_t)b * D + k0 + e] = ab[e];
      }
    }
  }
}

// =========================================================================
// R: column sums of partials, several jobs in one launch.  Block (32, 16):
// x picks the column, y a stripe of partial rows p = y, y+16, ...; stripes
// are combined in a fixed order.
// =========================================================================
struct ColsumArgs {
  ColsumJob job[kMaxColsumJobs];
  int block_start[kMaxColsumJobs + 1];
  int njobs;
};

template <typename T>
__global__ void __launch_bounds__(512) k_colsums(const ColsumArgs a) {
  __shared__ float part[16][33];
  int jb = 0;
  while (jb + 1 < a.njobs && (int)blockIdx.x >= a.block_start[jb + 1]) ++jb;
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

// ---------------------------------------------------------------- launch helpers
template <typename Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

int max_dynamic_smem_bytes() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return v;
}

size_t per_sample_smem_bytes(const RowArgs& a) {
  const size_t xs = align16((size_t)a.T * a.D * elem_bytes(a.dtype));
  const int nthreads = round32(a.D / vec_elems(a.dtype));
  const size_t g7 = xs + (size_t)4 * a.T * 4 + (size_t)a.T * (nthreads / 32) * 2 * 4;
  const size_t f1 = xs + (size_t)2 * a.T * 4;
  return g7 > f1 ? g7 : f1;
}

cudaError_t launch_ln0_mix_ln1_fwd(const RowArgs& a, const void* x, const void* g0, const void* be0,
                                   const void* g1, const void* be1, void* out1, float* mu0, float* r0,
                                   float* mu1, float* r1, cudaStream_t st) {
  const size_t smem = align16((size_t)a.T * a.D * elem_bytes(a.dtype)) + (size_t)2 * a.T * 4;
  const int q = (a.D + 31) / 32;
  const int C = a.D / a.T;
  const float eps = 1e-3f;
  cudaError_t err = cudaSuccess;
#define RMX_F1(MAXQ)                                                                              \
  RMX_DISPATCH_T(a.dtype, {                                                                       \
    auto k = k_ln0_mix_ln1_fwd<T, MAXQ>;                                                          \
    err = set_smem(k, smem);                                                                      \
    if (err == cudaSuccess)                                                                       \
      k<<<a.B, 256, smem, st>>>((const T*)x, (const T*)g0, (const T*)be0, (const T*)g1,           \
                                (const T*)be1, (T*)out1, mu0, r0, mu1, r1, a.T, a.D, C, eps);      \
  })
  if (q <= 2) RMX_F1(2);
  else if (q <= 4) RMX_F1(4);
  else if (q <= 8) RMX_F1(8);
  else if (q <= 16) RMX_F1(16);
  else if (q <= 24) RMX_F1(24);
  else if (q <= 40) RMX_F1(40);
  else return cudaErrorInvalidValue;
#undef RMX_F1
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_ln_rows_fwd(const RowArgs& a, const void* s, const void* g, const void* be, void* y,
                               float* mu, float* rs, cudaStream_t st) {
  const int N = a.B * a.T;
  const int nv = a.D / vec_elems(a.dtype);
  const int q = (nv + 31) / 32;
  const int grid = (N + 7) / 8;
#define RMX_F5(MAXV)                                                                               \
  RMX_DISPATCH_T(a.dtype, {                                                                        \
    k_ln_rows_fwd<T, MAXV><<<grid, 256, 0, st>>>((const T*)s, (const T*)g, (const T*)be, (T*)y, mu, \
                                                 rs, N, a.D, 1e-3f);                               \
  })
  if (q <= 1) RMX_F5(1);
  else if (q <= 2) RMX_F5(2);
  else if (q <= 4) RMX_F5(4);
  else if (q <= 6) RMX_F5(6);
  else if (q <= 10) RMX_F5(10);
  else return cudaErrorInvalidValue;
#undef RMX_F5
  return cudaGetLastError();
}

cudaError_t launch_zstats(const RowArgs& a, const void* Z, float* zstats, cudaStream_t st) {
  const int N = a.B * a.T;
  const int tiles = zstats_tiles(a.H);
  const long long items = (long long)N * tiles;
  const int grid = (int)((items + 7) / 8);
  RMX_DISPATCH_T(a.dtype, { k_zstats<T><<<grid, 256, 0, st>>>((const T*)Z, zstats, N, a.H, tiles); });
  return cudaGetLastError();
}

cudaError_t launch_gate_fwd(const RowArgs& a, const void* Z, const float* zstats, const void* wx,
                            const void* bx, const void* wg, const void* bg, void* hidden, float* muU,
                            float* rU, float* muG, float* rG, cudaStream_t st) {
  const int N = a.B * a.T;
  int threads = round32(a.H / vec_elems(a.dtype));
  if (threads > kRowThreadsMax) threads = kRowThreadsMax;
  const int grid = (N + kGateRows - 1) / kGateRows;
  RMX_DISPATCH_T(a.dtype, {
    k_gate_fwd<T><<<grid, threads, 0, st>>>((const T*)Z, zstats, (const T*)wx, (const T*)bx, (const T*)wg,
                                            (const T*)bg, (T*)hidden, muU, rU, muG, rG, N, a.H, 1e-5f);
  });
  return cudaGetLastError();
}

cudaError_t launch_ln2_bwd(const RowArgs& a, const void* dy, const void* s2, const float* mu2,
                           const float* r2, const void* g2, void* ds2, float* pg2, float* pb2,
                           float* pbo, cudaStream_t st) {
  const int threads = round32(a.D / vec_elems(a.dtype));
  if (threads > kRowThreadsMax) return cudaErrorInvalidValue;
  dim3 grid(a.nbblk, a.T);
  const size_t smem = ring_smem_bytes((size_t)2 * a.D * elem_bytes(a.dtype));
  cudaError_t err = cudaSuccess;
  RMX_DISPATCH_T(a.dtype, {
    auto k = k_ln2_bwd<T>;
    err = set_smem(k, smem);
    if (err == cudaSuccess)
      k<<<grid, threads, smem, st>>>((const T*)dy, (const T*)s2, mu2, r2, (const T*)g2, (T*)ds2, pg2, pb2, pbo,
                                     a.B, a.T, a.D, a.nb, device_error_word());
  });
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_gate_bwd(const RowArgs& a, const void* dh, const void* Z, const float* muU,
                            const float* rU, const float* muG, const float* rG, const void* wx,
                            const void* bx, const void* wg, const void* bg, void* dZ, float* pwx,
                            float* pbx, float* pwg, float* pbg, float* pb1, float* rowsum, cudaStream_t st) {
  const int threads = round32(a.H / vec_elems(a.dtype));
  if (threads > kRowThreadsMax) return cudaErrorInvalidValue;
  const int N = a.B * a.T;
  RMX_DISPATCH_T(a.dtype, {
    k_gate_bwd_rowsums<T><<<(N + 7) / 8, 256, 0, st>>>((const T*)dh, (const T*)Z, muU, rU, muG, rG, (const T*)wx,
                                                       (const T*)bx, (const T*)wg, (const T*)bg, rowsum, N, a.H);
  });
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // Apply pass: 4 columns per thread, at most 256 threads per CTA.
  const int quads = a.H / 4;
  const int athreads = quads < 256 ? round32(quads) : 256;
  dim3 grid(a.nbblk, a.T, (quads + athreads - 1) / athreads);
  RMX_DISPATCH_T(a.dtype, {
    k_gate_bwd_apply<T><<<grid, athreads, 0, st>>>((const T*)dh, (const T*)Z, muU, rU, muG, rG, rowsum,
                                                   (const T*)wx, (const T*)bx, (const T*)wg, (const T*)bg, (T*)dZ,
                                                   pwx, pbx, pwg, pbg, pb1, a.B, a.T, a.H, a.nb);
  });
  return cudaGetLastError();
}

cudaError_t launch_ln1_mix_ln0_bwd(const RowArgs& a, const void* x, const void* dout1,
                                   const float* mu0, const float* r0, const float* mu1,
                                   const float* r1, const void* g0, const void* be0, const void* g1,
                                   float* ds1, void* dx, float* pg0, float* pb0, float* pg1,
                                   float* pbe1, cudaStream_t st) {
  const int threads = round32(a.D / vec_elems(a.dtype));
  if (threads > kRowThreadsMax) return cudaErrorInvalidValue;
  const size_t smem = align16((size_t)a.T * a.D * elem_bytes(a.dtype)) + (size_t)4 * a.T * 4 +
                      (size_t)a.T * (threads / 32) * 2 * 4;
  const int C = a.D / a.T;
  cudaError_t err = cudaSuccess;
  RMX_DISPATCH_T(a.dtype, {
    auto k = k_ln1_mix_ln0_bwd<T>;
    err = set_smem(k, smem);
    if (err == cudaSuccess)
      k<<<a.B, threads, smem, st>>>((const T*)x, (const T*)dout1, mu0, r0, mu1, r1, (const T*)g0,
                                    (const T*)be0, (const T*)g1, ds1, (T*)dx, pg0, pb0, pg1, pbe1,
                                    a.T, a.D, C);
  });
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_colsums(const ColsumJob* jobs, int njobs, int dtype, cudaStream_t st) {
  if (njobs <= 0 || njobs > kMaxColsumJobs) return cudaErrorInvalidValue;
  ColsumArgs a;
  a.njobs = njobs;
  int blocks = 0;
  for (int i = 0; i < njobs; ++i) {
    a.job[i] = jobs[i];
    a.block_start[i] = blocks;
    blocks += (jobs[i].J + 31) / 32;
  }
  a.block_start[njobs] = blocks;
  if (blocks == 0) return cudaSuccess;
  RMX_DISPATCH_T(dtype, { k_colsums<T><<<blocks, dim3(32, 16), 0, st>>>(a); });
  return cudaGetLastError();
}

}  // namespace rmx
