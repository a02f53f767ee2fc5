// Per-sample passes of the RankMixer block that contain the token mix:
//   forward:  out1 = norm1(token_mixer(norm0(x)) + x)
//   backward: ds1 = norm1-backward(dout1); da0 = token_mixer(ds1);
//             dx = ds1 + norm0-backward(da0)
// (page "Subgraph-fusion-based Mega-kernel Generation", section "Exact
// computation": token mixing reshapes [B,T,D] to [B,T,T,D/T] and swaps the
// two T axes, i.e. m[b,i,j*C+c] = a[b,j,i*C+c] with C = D/T; the swap is its
// own inverse, so the backward applies the same permutation).
//
// One sample is spread over a thread-block cluster of CL <= 8 CTAs; CTA k
// owns rows [k*R, min(T,(k+1)*R)), R = ceil(T/CL).  The permutation moves
// C-element chunks between rows, i.e. between CTAs: each CTA writes the
// chunks of its own rows straight into the shared memory of the CTA that owns
// the destination row (distributed shared memory), then the cluster
// synchronises and every CTA finishes its own rows locally.  Thread v owns
// the 16-byte column vector v of every row; row sums are taken with one
// deferred barrier per sweep (each warp leaves one partial per row).  All
// arithmetic is fp32, reductions run in a fixed order.

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace rmx {
namespace {

constexpr int kMaxCluster = 8;
constexpr int kMaxRows = 8;       // rows per CTA held in registers (T <= 64)
constexpr int kMixThreads = 320;  // one thread per 4 columns (D <= 1280)
constexpr int kMaxMixPartialRows = kMixPartialRowsMax;

__host__ __device__ inline size_t a16(size_t v) { return (v + 15) & ~size_t(15); }

struct MixGeom {
  int T, D, C, CL, R;
};

inline MixGeom mix_geom(int T, int D) {
  MixGeom g;
  g.T = T;
  g.D = D;
  g.C = D / T;
  g.CL = T < kMaxCluster ? T : kMaxCluster;
  g.R = (T + g.CL - 1) / g.CL;
  return g;
}

// Per-thread geometry: thread tid owns columns k0 .. k0+E-1 of every row.
// For column d = i*C + c (chunk i, offset c) the token mix sends row j's
// element to row i, column j*C + c; the CTA owning row i is i / R and it is
// that CTA's local row i % R.  All of this depends on the column only, so it
// is computed once per thread.
constexpr int E = 4;

struct ColMap {
  int chunk[E];    // i = d / C  (also: source row of mixed column d)
  int off[E];      // c = d % C
  int rank[E];     // owner CTA of row i
  int dst[E];      // (i % R) * D + c: destination offset before adding j*C
};

__device__ __forceinline__ ColMap col_map(int k0, int C, int D, int R) {
  ColMap m;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = k0 + e;
    const int i = d / C, c = d - i * C;
    m.chunk[e] = i;
    m.off[e] = c;
    m.rank[e] = i / R;
    m.dst[e] = (i - m.rank[e] * R) * D + c;
  }
  return m;
}

// Writes this thread's E values of source row j into the receive buffers of
// the rows they belong to after the mix.  Element pairs that share a chunk go
// as one store (C even).
template <typename Elt>
__device__ __forceinline__ void push_row(cg::cluster_group& cluster, Elt* recv, const ColMap& m, const float* vals,
                                         int j, int C, bool pairs) {
  if (pairs) {
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      Elt* dst = cluster.map_shared_rank(recv, m.rank[e]) + m.dst[e] + j * C;
      if (sizeof(Elt) == 4) {
        *reinterpret_cast<float2*>(dst) = make_float2(vals[e], vals[e + 1]);
      } else {
        Elt pr[2] = {from_f<Elt>(vals[e]), from_f<Elt>(vals[e + 1])};
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(pr);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) *(cluster.map_shared_rank(recv, m.rank[e]) + m.dst[e] + j * C) = from_f<Elt>(vals[e]);
  }
}

// Sum of one value per (row, warp) written by the warps' lane 0.
__device__ __forceinline__ float row_total(const float* red, int row, int nw) {
  float s = 0.f;
  for (int w = 0; w < nw; ++w) s += red[row * nw + w];
  return s;
}

// =========================================================================
// Forward: norm0 -> token mix -> + x -> norm1.  One cluster per sample.
// Shared memory: amix [R][D] fp32 (received chunks of norm0(x)), gamma0 and
// beta0 as fp32, row-sum scratch [R][nw].
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(kMixThreads) k_mix_fwd(const T* __restrict__ x, const T* __restrict__ g0,
                                                         const T* __restrict__ be0, const T* __restrict__ g1,
                                                         const T* __restrict__ be1, T* __restrict__ out1,
                                                         float* __restrict__ mu0, float* __restrict__ r0,
                                                         float* __restrict__ mu1, float* __restrict__ r1, int Tn,
                                                         int D, int C, int R, float eps) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char sm[];
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / CL;
  const int row0 = rank * R;
  const int nr = max(0, min(Tn, row0 + R) - row0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  float* amix = reinterpret_cast<float*>(sm);  // [R][D]
  float* red = amix + (size_t)R * D;           // [R][nw]
  const size_t base = (size_t)b * Tn * D;
  const bool act = tid * E < D;
  const int k0 = tid * E;
  const float invD = 1.0f / (float)D;
  const bool pairs = (C & 1) == 0;
  const ColMap cm = col_map(act ? k0 : 0, C, D, R);

  float xv[kMaxRows][E];
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il)
    if (il < nr && act) load_n<T, E>(x + base + (size_t)(row0 + il) * D + k0, xv[il]);
  cluster.sync();  // every CTA of the cluster runs before any remote store

  // norm0 statistics of the own rows: mean, then centred sum of squares.
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) {
    if (il >= nr) break;
    float s = 0.f;
    if (act)
#pragma unroll
      for (int e = 0; e < E; ++e) s += xv[il][e];
    s = warp_sum(s);
    if (lane == 0) red[il * nw + warp] = s;
  }
  __syncthreads();
  float mean0[kMaxRows];
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) mean0[il] = il < nr ? row_total(red, il, nw) * invD : 0.f;
  __syncthreads();
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) {
    if (il >= nr) break;
    float s = 0.f;
    if (act)
#pragma unroll
      for (int e = 0; e < E; ++e) s += (xv[il][e] - mean0[il]) * (xv[il][e] - mean0[il]);
    s = warp_sum(s);
    if (lane == 0) red[il * nw + warp] = s;
  }
  __syncthreads();
  float gg[E], bb[E];
  if (act) {
    load_n<T, E>(g0 + k0, gg);
    load_n<T, E>(be0 + k0, bb);
  }
  // norm0(x) of the own rows, sent to the CTAs that own the mixed rows.
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) {
    if (il >= nr) break;
    const float rstd = 1.0f / sqrtf(row_total(red, il, nw) * invD + eps);
    if (tid == 0) {
      mu0[(size_t)b * Tn + row0 + il] = mean0[il];
      r0[(size_t)b * Tn + row0 + il] = rstd;
    }
    if (act) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = (xv[il][e] - mean0[il]) * rstd * gg[e] + bb[e];
      push_row<float>(cluster, amix, cm, a, row0 + il, C, pairs);
    }
  }
  cluster.sync();  // every chunk of the mixed rows has arrived

  // s1 = token_mix(norm0(x)) + x for the own rows, then norm1.
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) {
    if (il >= nr) break;
    float s = 0.f;
    if (act) {
      const float4 am = *reinterpret_cast<const float4*>(amix + (size_t)il * D + k0);
      xv[il][0] += am.x;
      xv[il][1] += am.y;
      xv[il][2] += am.z;
      xv[il][3] += am.w;
#pragma unroll
      for (int e = 0; e < E; ++e) s += xv[il][e];
    }
    s = warp_sum(s);
    if (lane == 0) red[il * nw + warp] = s;
  }
  __syncthreads();
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) mean0[il] = il < nr ? row_total(red, il, nw) * invD : 0.f;
  __syncthreads();
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) {
    if (il >= nr) break;
    float s = 0.f;
    if (act)
#pragma unroll
      for (int e = 0; e < E; ++e) s += (xv[il][e] - mean0[il]) * (xv[il][e] - mean0[il]);
    s = warp_sum(s);
    if (lane == 0) red[il * nw + warp] = s;
  }
  __syncthreads();
  if (act) {
    load_n<T, E>(g1 + k0, gg);
    load_n<T, E>(be1 + k0, bb);
  }
#pragma unroll
  for (int il = 0; il < kMaxRows; ++il) {
    if (il >= nr) break;
    const float rstd = 1.0f / sqrtf(row_total(red, il, nw) * invD + eps);
    const size_t row = (size_t)b * Tn + row0 + il;
    if (tid == 0) {
      mu1[row] = mean0[il];
      r1[row] = rstd;
    }
    if (act) {
      float o[E];
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = (xv[il][e] - mean0[il]) * rstd * gg[e] + bb[e];
      store_n<T, E>(out1 + row * D + k0, o);
    }
  }
}

// =========================================================================
// Backward: norm1 backward, the token mix, norm0 backward and the residual.
// Persistent: cluster q handles samples q, q + nclusters, ...; each CTA keeps
// its partial sums of dgamma0, dbeta0, dgamma1, dbeta1 in registers and
// writes one partial row at the end.
// Shared memory: xs [R][D] own rows of x, xmix [R][D] received chunks of x,
// da0 [R][D] fp32 received chunks of ds1, gamma0 / beta0 (fp32), statistics
// of the sample, row-sum scratch [2][R][nw].
// =========================================================================
template <typename T>
__global__ void __launch_bounds__(kMixThreads) k_mix_bwd(
    const T* __restrict__ x, const T* __restrict__ dout1, const float* __restrict__ mu0,
    const float* __restrict__ r0, const float* __restrict__ mu1, const float* __restrict__ r1,
    const T* __restrict__ g0, const T* __restrict__ be0, const T* __restrict__ g1, T* __restrict__ dx,
    float* __restrict__ pg0, float* __restrict__ pb0, float* __restrict__ pg1, float* __restrict__ pbe1, int B,
    int Tn, int D, int C, int R, int nclusters) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char sm[];
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int q = blockIdx.x / CL;
  const int row0 = rank * R;
  const int nr = max(0, min(Tn, row0 + R) - row0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  T* xs = reinterpret_cast<T*>(sm);
  T* xmix = reinterpret_cast<T*>(sm + a16((size_t)R * D * sizeof(T)));
  float* da0 = reinterpret_cast<float*>(sm + 2 * a16((size_t)R * D * sizeof(T)));
  float* sg0 = da0 + (size_t)R * D;  // gamma0 [D]
  float* sb0 = sg0 + D;              // beta0 [D]
  float* s_mu0 = sb0 + D;            // [Tn]
  float* s_r0 = s_mu0 + Tn;          // [Tn]
  float* red = s_r0 + Tn;            // [2][R][nw]
  const bool act = tid * E < D;
  const int k0 = tid * E;
  const float invD = 1.0f / (float)D;
  const bool pairs = (C & 1) == 0;
  const ColMap cm = col_map(act ? k0 : 0, C, D, R);

  for (int i = tid; i < D; i += blockDim.x) {
    sg0[i] = to_f(g0[i]);
    sb0[i] = to_f(be0[i]);
  }
  float gam0[E], gam1[E], ag0[E], ab0[E], ag1[E], ab1[E];
#pragma unroll
  for (int e = 0; e < E; ++e) ag0[e] = ab0[e] = ag1[e] = ab1[e] = 0.f;
  if (act) {
    load_n<T, E>(g0 + k0, gam0);
    load_n<T, E>(g1 + k0, gam1);
  }
  cluster.sync();  // every CTA of the cluster runs before any remote store; sg0/sb0 ready

  for (int b = q; b < B; b += nclusters) {
    const size_t base = (size_t)b * Tn * D;
    for (int p = tid; p < Tn; p += blockDim.x) {
      s_mu0[p] = mu0[(size_t)b * Tn + p];
      s_r0[p] = r0[(size_t)b * Tn + p];
    }
    // ---- own rows of x (kept for norm0's backward) sent to the mixed rows;
    // dout1 of the own rows.
    float d1[kMaxRows][E];
#pragma unroll
    for (int il = 0; il < kMaxRows; ++il) {
      if (il >= nr) continue;
      if (act) {
        float xv[E];
        load_n<T, E>(x + base + (size_t)(row0 + il) * D + k0, xv);
        store_n<T, E>(xs + (size_t)il * D + k0, xv);
        push_row<T>(cluster, xmix, cm, xv, row0 + il, C, pairs);
        load_n<T, E>(dout1 + base + (size_t)(row0 + il) * D + k0, d1[il]);
      }
    }
    cluster.sync();  // (1) xmix complete; s_mu0 / s_r0 visible

    // xh1 of own mixed row i for this thread's columns: element k = j*C + c
    // is norm0(x)[j, i*C + c] + x[i, k].
    auto xhat1 = [&](int il, float m1, float s1r, float* xh) {
      const int i = row0 + il;
      float xm[E], xo[E];
      load_n<T, E>(xmix + (size_t)il * D + k0, xm);
      load_n<T, E>(xs + (size_t)il * D + k0, xo);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int j = cm.chunk[e], d = i * C + cm.off[e];
        const float a0 = (xm[e] - s_mu0[j]) * s_r0[j] * sg0[d] + sb0[d];
        xh[e] = (a0 + xo[e] - m1) * s1r;
      }
    };

    // ---- norm1 backward, sweep 1: row sums of g = gamma1*dout1 and g*xh1.
#pragma unroll
    for (int il = 0; il < kMaxRows; ++il) {
      if (il >= nr) continue;
      const size_t row = (size_t)b * Tn + row0 + il;
      float s0 = 0.f, s1 = 0.f;
      if (act) {
        float xh[E];
        xhat1(il, mu1[row], r1[row], xh);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float g = gam1[e] * d1[il][e];
          s0 += g;
          s1 += g * xh[e];
        }
      }
      s0 = warp_sum(s0);
      s1 = warp_sum(s1);
      if (lane == 0) {
        red[(0 * R + il) * nw + warp] = s0;
        red[(1 * R + il) * nw + warp] = s1;
      }
    }
    __syncthreads();
    // ---- sweep 2: ds1 (kept in registers for the residual), partials, and
    // the chunks of ds1 sent to the rows of da0 = token_mix(ds1).
#pragma unroll
    for (int il = 0; il < kMaxRows; ++il) {
      if (il >= nr) continue;
      const size_t row = (size_t)b * Tn + row0 + il;
      const float mg = row_total(red, 0 * R + il, nw) * invD;
      const float mgx = row_total(red, 1 * R + il, nw) * invD;
      const float s1r = r1[row];
      if (act) {
        float xh[E];
        xhat1(il, mu1[row], s1r, xh);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float dv = d1[il][e];
          const float g = gam1[e] * dv;
          ag1[e] += dv * xh[e];
          ab1[e] += dv;
          d1[il][e] = s1r * (g - mg - xh[e] * mgx);  // now ds1
        }
        push_row<float>(cluster, da0, cm, d1[il], row0 + il, C, pairs);
      }
    }
    cluster.sync();  // (2) da0 complete; every CTA is done reading xmix

    // ---- norm0 backward, sweep 1: row sums of g0 = gamma0*da0 and g0*xh0.
#pragma unroll
    for (int jl = 0; jl < kMaxRows; ++jl) {
      if (jl >= nr) continue;
      const int j = row0 + jl;
      float s0 = 0.f, s1 = 0.f;
      if (act) {
        float xo[E];
        load_n<T, E>(xs + (size_t)jl * D + k0, xo);
        const float4 dr = *reinterpret_cast<const float4*>(da0 + (size_t)jl * D + k0);
        const float dv[E] = {dr.x, dr.y, dr.z, dr.w};
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float g = gam0[e] * dv[e];
          s0 += g;
          s1 += g * (xo[e] - s_mu0[j]) * s_r0[j];
        }
      }
      s0 = warp_sum(s0);
      s1 = warp_sum(s1);
      if (lane == 0) {
        red[(0 * R + jl) * nw + warp] = s0;
        red[(1 * R + jl) * nw + warp] = s1;
      }
    }
    __syncthreads();
    // ---- sweep 2: dx = ds1 + norm0-backward(da0), partials.
#pragma unroll
    for (int jl = 0; jl < kMaxRows; ++jl) {
      if (jl >= nr) continue;
      const int j = row0 + jl;
      const float mg = row_total(red, 0 * R + jl, nw) * invD;
      const float mgx = row_total(red, 1 * R + jl, nw) * invD;
      if (act) {
        float xo[E], o[E];
        load_n<T, E>(xs + (size_t)jl * D + k0, xo);
        const float4 dr = *reinterpret_cast<const float4*>(da0 + (size_t)jl * D + k0);
        const float dv[E] = {dr.x, dr.y, dr.z, dr.w};
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh0 = (xo[e] - s_mu0[j]) * s_r0[j];
          const float g = gam0[e] * dv[e];
          o[e] = d1[jl][e] + s_r0[j] * (g - mg - xh0 * mgx);
          ag0[e] += dv[e] * xh0;
          ab0[e] += dv[e];
        }
        store_n<T, E>(dx + base + (size_t)j * D + k0, o);
      }
    }
    __syncthreads();  // xs, red and the statistics are reused by the next sample
  }
  if (act) {
    const size_t p = (size_t)blockIdx.x * D + k0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      pg0[p + e] = ag0[e];
      pb0[p + e] = ab0[e];
      pg1[p + e] = ag1[e];
      pbe1[p + e] = ab1[e];
    }
  }
}

template <typename Kern, typename... Args>
cudaError_t launch_cluster(Kern k, int grid, int threads, size_t smem, int cl, cudaStream_t st, Args... args) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

inline int mix_threads(int D, int /*dtype*/) { return (D / E + 31) / 32 * 32; }

size_t mix_fwd_smem(const MixGeom& g, int /*dtype*/, int threads) {
  return (size_t)g.R * g.D * 4 + (size_t)g.R * (threads / 32) * 4;
}

size_t mix_bwd_smem(const MixGeom& g, int dtype, int threads) {
  const int e = dtype == 0 ? 4 : 2;
  return 2 * a16((size_t)g.R * g.D * e) + (size_t)g.R * g.D * 4 + (size_t)2 * g.D * 4 + (size_t)2 * g.T * 4 +
         (size_t)2 * g.R * (threads / 32) * 4;
}

}  // namespace

bool mix_supported(const RowArgs& a) {
  const MixGeom g = mix_geom(a.T, a.D);
  const int threads = mix_threads(a.D, a.dtype);
  if (g.R > kMaxRows || threads > kMixThreads || a.D % E) return false;
  const size_t lim = (size_t)max_dynamic_smem_bytes();
  return mix_fwd_smem(g, a.dtype, threads) <= lim && mix_bwd_smem(g, a.dtype, threads) <= lim;
}

int mix_bwd_partial_rows(const RowArgs& a) {
  const MixGeom g = mix_geom(a.T, a.D);
  const int threads = mix_threads(a.D, a.dtype);
  int per_sm = 1;
  const size_t smem = mix_bwd_smem(g, a.dtype, threads);
  const int lim = max_dynamic_smem_bytes();
  if (lim > 0) per_sm = (int)((size_t)(lim + 1024) / (smem + 1024));
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
  int nclusters = sm_count() * per_sm / g.CL;
  if (nclusters > kMaxMixPartialRows / g.CL) nclusters = kMaxMixPartialRows / g.CL;
  if (nclusters > a.B) nclusters = a.B;
  if (nclusters < 1) nclusters = 1;
  return nclusters * g.CL;
}

cudaError_t launch_mix_fwd(const RowArgs& a, const void* x, const void* g0, const void* be0, const void* g1,
                           const void* be1, void* out1, float* mu0, float* r0, float* mu1, float* r1,
                           cudaStream_t st) {
  const MixGeom g = mix_geom(a.T, a.D);
  const int threads = mix_threads(a.D, a.dtype);
  const size_t smem = mix_fwd_smem(g, a.dtype, threads);
  const int grid = a.B * g.CL;
  cudaError_t err = cudaSuccess;
  if (a.dtype == 0)
    err = launch_cluster(k_mix_fwd<float>, grid, threads, smem, g.CL, st, (const float*)x, (const float*)g0,
                         (const float*)be0, (const float*)g1, (const float*)be1, (float*)out1, mu0, r0, mu1, r1,
                         a.T, a.D, g.C, g.R, 1e-3f);
  else if (a.dtype == 1)
    err = launch_cluster(k_mix_fwd<bf16>, grid, threads, smem, g.CL, st, (const bf16*)x, (const bf16*)g0,
                         (const bf16*)be0, (const bf16*)g1, (const bf16*)be1, (bf16*)out1, mu0, r0, mu1, r1, a.T,
                         a.D, g.C, g.R, 1e-3f);
  else
    err = launch_cluster(k_mix_fwd<f16>, grid, threads, smem, g.CL, st, (const f16*)x, (const f16*)g0,
                         (const f16*)be0, (const f16*)g1, (const f16*)be1, (f16*)out1, mu0, r0, mu1, r1, a.T, a.D,
                         g.C, g.R, 1e-3f);
  return err;
}

cudaError_t launch_mix_bwd(const RowArgs& a, const void* x, const void* dout1, const float* mu0, const float* r0,
                           const float* mu1, const float* r1, const void* g0, const void* be0, const void* g1,
                           void* dx, float* pg0, float* pb0, float* pg1, float* pbe1, cudaStream_t st) {
  const MixGeom g = mix_geom(a.T, a.D);
  const int threads = mix_threads(a.D, a.dtype);
  const size_t smem = mix_bwd_smem(g, a.dtype, threads);
  const int ctas = mix_bwd_partial_rows(a);
  const int nclusters = ctas / g.CL;
  cudaError_t err = cudaSuccess;
  if (a.dtype == 0)
    err = launch_cluster(k_mix_bwd<float>, ctas, threads, smem, g.CL, st, (const float*)x, (const float*)dout1, mu0,
                         r0, mu1, r1, (const float*)g0, (const float*)be0, (const float*)g1, (float*)dx, pg0, pb0,
                         pg1, pbe1, a.B, a.T, a.D, g.C, g.R, nclusters);
  else if (a.dtype == 1)
    err = launch_cluster(k_mix_bwd<bf16>, ctas, threads, smem, g.CL, st, (const bf16*)x, (const bf16*)dout1, mu0,
                         r0, mu1, r1, (const bf16*)g0, (const bf16*)be0, (const bf16*)g1, (bf16*)dx, pg0, pb0, pg1,
                         pbe1, a.B, a.T, a.D, g.C, g.R, nclusters);
  else
    err = launch_cluster(k_mix_bwd<f16>, ctas, threads, smem, g.CL, st, (const f16*)x, (const f16*)dout1, mu0, r0,
                         mu1, r1, (const f16*)g0, (const f16*)be0, (const f16*)g1, (f16*)dx, pg0, pb0, pg1, pbe1,
                         a.B, a.T, a.D, g.C, g.R, nclusters);
  return err;
}

}  // namespace rmx
