// norm0 -> token mix -> + x -> norm1 for one whole sample per CTA.
//
// Page "Subgraph-fusion-based Mega-kernel Generation", section "Exact
// computation": out1 = norm1(token_mixer(norm0(x)) + x), with LN(z) = (z -
// mean) / sqrt(mean((z - mean)^2) + eps) * gamma + beta over each row and
// token mixing = reshape [T, T, C] (C = D/T) and swap the two T axes, i.e.
// row i of the mixed sample holds, at column j*C + c, column i*C + c of row j.
//
// The sample's T rows of x are bulk-copied into shared memory once (rows
// padded by 16 bytes so that the gather below spreads over the banks).  Then
// (1) one warp per row takes norm0's statistics from shared memory (two
// passes, exact); (2) one warp per output row i builds
//   s1[i, j*C + c] = norm0(x)[j, i*C + c] + x[i, j*C + c]
// by gathering from shared memory, rounds it to the storage type (the
// backward reads the stored s1, so norm1 is taken of exactly those values),
// takes norm1's statistics of the row held in registers and writes s1 and
// out1.  x is read from HBM once; nothing token-mixed is written.

#include "common.cuh"
#include "kernels.h"

namespace rmx {
namespace {

struct Ln01Args {
  const void* x;       // [B, T, D]
  const void* gamma0;  // [D]
  const void* beta0;
  const void* gamma1;
  const void* beta1;
  void* s1;            // [B, T, D] norm1's input, rounded to the storage type
  void* out1;          // [B, T, D]
  float* mu0;          // [B*T] row statistics
  float* r0;
  float* mu1;
  float* r1;
  unsigned int* err;
  int B, T, D, C;
  float eps;
};

// Shared memory: st0 [T] float2 (mean, rstd of norm0) | g0, b0 [D] float
// (norm0's gamma and beta) | x rows [T][D + pad] | mbarrier.
template <typename T, int MAXV>
__global__ void __launch_bounds__(512, 1) k_ln01_fwd(const Ln01Args a) {
  constexpr int V = VecN<T>::value;
  extern __shared__ __align__(16) unsigned char smem[];
  const int Tn = a.T, D = a.D, C = a.C;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const size_t row_bytes = (size_t)D * sizeof(T);
  const size_t pitch = row_bytes + 16;  // bytes between staged rows
  float2* st0 = reinterpret_cast<float2*>(smem);
  float* g0 = reinterpret_cast<float*>(smem + (((size_t)Tn * 8 + 15) & ~(size_t)15));
  float* b0 = g0 + D;
  unsigned char* xs = reinterpret_cast<unsigned char*>(b0 + D);
  uint64_t* bar = reinterpret_cast<uint64_t*>(xs + (size_t)Tn * pitch);
  __shared__ int abort_flag;

  const T* xb = reinterpret_cast<const T*>(a.x) + (size_t)b * Tn * D;
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(smem_u32(bar), (uint32_t)((size_t)Tn * row_bytes));
    for (int j = 0; j < Tn; ++j)
      bulk_g2s(smem_u32(xs + (size_t)j * pitch), xb + (size_t)j * D, (uint32_t)row_bytes, smem_u32(bar));
  }
  for (int d = tid; d < D; d += blockDim.x) {
    g0[d] = to_f(reinterpret_cast<const T*>(a.gamma0)[d]);
    b0[d] = to_f(reinterpret_cast<const T*>(a.beta0)[d]);
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(smem_u32(bar), 0, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS,
                                    (volatile int*)&abort_flag);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) {
      // Give the copies in flight a bounded time to land before the CTA's
      // shared memory goes away.
      volatile int no_abort = 0;
      mbar_wait_bounded(smem_u32(bar), 0, kWaitLimitNs, a.err, ERRBIT_WAIT_ROWS, &no_abort);
    }
    return;
  }

  const float invD = 1.0f / (float)D;
  const int nv = D / V;
  // (1) norm0 statistics, one warp per row.
  for (int j = warp; j < Tn; j += nw) {
    const T* row = reinterpret_cast<const T*>(xs + (size_t)j * pitch);
    float sum = 0.f;
    for (int vi = lane; vi < nv; vi += 32) {
      float v[V];
      load_vec(row + vi * V, v);
#pragma unroll
      for (int e = 0; e < V; ++e) sum += v[e];
    }
    const float mean = warp_sum(sum) * invD;
    float ss = 0.f;
    for (int vi = lane; vi < nv; vi += 32) {
      float v[V];
      load_vec(row + vi * V, v);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float c = v[e] - mean;
        ss = fmaf(c, c, ss);
      }
    }
    const float rstd = 1.0f / sqrtf(warp_sum(ss) * invD + a.eps);
    if (lane == 0) {
      st0[j] = make_float2(mean, rstd);
      const size_t r = (size_t)b * Tn + j;
      a.mu0[r] = mean;
      a.r0[r] = rstd;
    }
  }
  __syncthreads();

  // (2) one warp per output row i.
  const T* gm1 = reinterpret_cast<const T*>(a.gamma1);
  const T* bt1 = reinterpret_cast<const T*>(a.beta1);
  for (int i = warp; i < Tn; i += nw) {
    const T* own = reinterpret_cast<const T*>(xs + (size_t)i * pitch);
    float sv[MAXV][V];
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int vi = lane + 32 * q;
      if (vi < nv) {
        const int d0 = vi * V;
        float xi[V];
        load_vec(own + d0, xi);
        int j = d0 / C, c = d0 - j * C;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          // norm0(x)[j, i*C + c]: column i*C + c of staged row j.
          const int col = i * C + c;
          const float xj = to_f(reinterpret_cast<const T*>(xs + (size_t)j * pitch)[col]);
          const float2 s0 = st0[j];
          const float a0 = fmaf((xj - s0.x) * s0.y, g0[col], b0[col]);
          const float s = to_f(from_f<T>(a0 + xi[e]));
          sv[q][e] = s;
          sum += s;
          if (++c == C) {
            c = 0;
            ++j;
          }
        }
      }
    }
    const float mean = warp_sum(sum) * invD;
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      if (lane + 32 * q < nv) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float c = sv[q][e] - mean;
          ss = fmaf(c, c, ss);
        }
      }
    }
    const float rstd = 1.0f / sqrtf(warp_sum(ss) * invD + a.eps);
    const size_t r = (size_t)b * Tn + i;
    if (lane == 0) {
      a.mu1[r] = mean;
      a.r1[r] = rstd;
    }
    T* s1row = reinterpret_cast<T*>(a.s1) + r * D;
    T* orow = reinterpret_cast<T*>(a.out1) + r * D;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int vi = lane + 32 * q;
      if (vi < nv) {
        const int d0 = vi * V;
        float gg[V], bb[V], o[V];
        load_vec(gm1 + d0, gg);
        load_vec(bt1 + d0, bb);
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] = fmaf((sv[q][e] - mean) * rstd, gg[e], bb[e]);
        store_vec(s1row + d0, sv[q]);
        store_vec(orow + d0, o);
      }
    }
  }
}

size_t ln01_smem_bytes(int Tn, int D, int esize) {
  return (((size_t)Tn * 8 + 15) & ~(size_t)15) + (size_t)2 * D * 4 + (size_t)Tn * ((size_t)D * esize + 16) + 16;
}

template <typename T, int MAXV>
cudaError_t launch_typed(const Ln01Args& a, cudaStream_t st) {
  const size_t smem = ln01_smem_bytes(a.T, a.D, (int)sizeof(T));
  auto k = k_ln01_fwd<T, MAXV>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int warps = a.T < 16 ? a.T : 16;
  k<<<a.B, 32 * warps, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_v(const Ln01Args& a, int q, cudaStream_t st) {
  if (q <= 1) return launch_typed<T, 1>(a, st);
  if (q <= 2) return launch_typed<T, 2>(a, st);
  if (q <= 4) return launch_typed<T, 4>(a, st);
  if (q <= 6) return launch_typed<T, 6>(a, st);
  return launch_typed<T, 10>(a, st);
}

}  // namespace

bool ln01_fwd_supported(const RowArgs& ra) {
  const int e = ra.dtype == 0 ? 4 : 2, V = 16 / e;
  if (ra.D % V || ra.D % ra.T) return false;
  if ((ra.D / V + 31) / 32 > 10) return false;
  if ((long long)ra.T * ra.D * e >= (1ll << 20)) return false;  // one mbarrier counts the sample's bytes
  return (long long)ln01_smem_bytes(ra.T, ra.D, e) <= (long long)max_dynamic_smem_bytes() - 1024;
}

cudaError_t launch_ln01_fwd(const RowArgs& ra, const void* x, const void* gamma0, const void* beta0,
                            const void* gamma1, const void* beta1, void* s1, void* out1, float* mu0, float* r0,
                            float* mu1, float* r1, cudaStream_t st) {
  if (!ln01_fwd_supported(ra)) return cudaErrorInvalidValue;
  Ln01Args a;
  a.x = x;
  a.gamma0 = gamma0;
  a.beta0 = beta0;
  a.gamma1 = gamma1;
  a.beta1 = beta1;
  a.s1 = s1;
  a.out1 = out1;
  a.mu0 = mu0;
  a.r0 = r0;
  a.mu1 = mu1;
  a.r1 = r1;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidValue;
  a.B = ra.B;
  a.T = ra.T;
  a.D = ra.D;
  a.C = ra.D / ra.T;
  a.eps = 1e-3f;
  const int V = ra.dtype == 0 ? 4 : 8;
  const int q = (ra.D / V + 31) / 32;
  if (ra.dtype == 0) return launch_v<float>(a, q, st);
  if (ra.dtype == 1) return launch_v<bf16>(a, q, st);
  return launch_v<f16>(a, q, st);
}

}  // namespace rmx
