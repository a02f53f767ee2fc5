// Grouped GEMM on the CUDA cores (plain fp32 FMA).
//
// Used for the strict float32 contract (no TF32: the per-token contractions
// of the RankMixer block are computed in IEEE fp32) and for 16-bit shapes
// whose row strides do not meet the tensor-map alignment.  Same layouts and
// epilogues as the tensor-core engine (kernels.h); operands are read through
// generic strides, so NN, NT and TN share one kernel.  The k loop runs in a
// fixed order, so results are bitwise repeatable.

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

struct SimtParams {
  int M, N, K, G;
  const void* A;
  long long a_ms, a_ks, a_gs;
  const void* Bm;
  long long b_ks, b_ns, b_gs;
  void* out;
  long long out_rs, out_gs;
  const void* bias;
  long long bias_gs;
  const void* resid;
  long long res_rs, res_gs;
};

template <typename T, int EPI>
__global__ void __launch_bounds__(256) k_gemm_simt(const SimtParams p) {
  pdl_enter();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int g = blockIdx.z, m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const T* A = reinterpret_cast<const T*>(p.A) + (size_t)g * p.a_gs;
  const T* Bm = reinterpret_cast<const T*>(p.Bm) + (size_t)g * p.b_gs;
  const bool a_k_contig = p.a_ks == 1;
  const bool b_n_contig = p.b_ns == 1;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < p.K; k0 += TK) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = tid + 256 * r;
      int mm, kk;
      if (a_k_contig) { kk = idx % TK; mm = idx / TK; } else { mm = idx % TM; kk = idx / TM; }
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < p.M && k < p.K) ? to_f(A[(size_t)m * p.a_ms + (size_t)k * p.a_ks]) : 0.f;
      int nn, kb;
      if (b_n_contig) { nn = idx % TN; kb = idx / TN; } else { kb = idx % TK; nn = idx / TK; }
      const int n = n0 + nn, kq = k0 + kb;
      Bs[kb][nn] = (n < p.N && kq < p.K) ? to_f(Bm[(size_t)kq * p.b_ks + (size_t)n * p.b_ns]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  T* out = reinterpret_cast<T*>(p.out) + (size_t)g * p.out_gs;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      float v = acc[i][j];
      if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID)
        v += to_f(reinterpret_cast<const T*>(p.bias)[(size_t)g * p.bias_gs + n]);
      if (EPI == EPI_RESID || EPI == EPI_BIAS_RESID)
        v += to_f(reinterpret_cast<const T*>(p.resid)[(size_t)g * p.res_gs + (size_t)m * p.res_rs + n]);
      out[(size_t)m * p.out_rs + n] = from_f<T>(v);
    }
  }
}

template <typename T>
cudaError_t dispatch_simt(const SimtParams& p, int epi, cudaStream_t st) {
  dim3 grid((p.N + TN - 1) / TN, (p.M + TM - 1) / TM, p.G);
  switch (epi) {
    case EPI_STORE: return launch_k(k_gemm_simt<T, EPI_STORE>, grid, dim3(256), 0, st, 1, p);
    case EPI_BIAS:
    case EPI_BIAS_ZSTATS:  // statistics are taken by launch_zstats on this path
      return launch_k(k_gemm_simt<T, EPI_BIAS>, grid, dim3(256), 0, st, 1, p);
    case EPI_BIAS_RESID: return launch_k(k_gemm_simt<T, EPI_BIAS_RESID>, grid, dim3(256), 0, st, 1, p);
    case EPI_RESID: return launch_k(k_gemm_simt<T, EPI_RESID>, grid, dim3(256), 0, st, 1, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t gemm_simt_launch(const GemmDesc& d, cudaStream_t st) {
  if (d.M <= 0 || d.N <= 0 || d.K <= 0 || d.G <= 0) return cudaErrorInvalidValue;
  if (d.G > 65535 || (d.M + TM - 1) / TM > 65535) return cudaErrorInvalidValue;
  const long long M = d.M, N = d.N, K = d.K, G = d.G;
  SimtParams p;
  p.M = d.M;
  p.N = d.N;
  p.K = d.K;
  p.G = d.G;
  p.A = d.A;
  p.Bm = d.Bm;
  p.out = d.C;
  p.bias = d.bias;
  p.resid = d.resid;
  p.bias_gs = N;
  switch (d.kind) {
    case GEMM_FWD:  // A [M,G,K], Bm [G,K,N]
      p.a_ms = G * K; p.a_ks = 1; p.a_gs = K;
      p.b_ks = N; p.b_ns = 1; p.b_gs = K * N;
      p.out_rs = G * N; p.out_gs = N;
      break;
    case GEMM_DGRAD:  // A [M,G,K], Bm [G,N,K]
      p.a_ms = G * K; p.a_ks = 1; p.a_gs = K;
      p.b_ks = 1; p.b_ns = K; p.b_gs = N * K;
      p.out_rs = G * N; p.out_gs = N;
      break;
    case GEMM_WGRAD:  // A [K,G,M], Bm [K,G,N], C [G,M,N]
      p.a_ms = 1; p.a_ks = G * M; p.a_gs = M;
      p.b_ks = G * N; p.b_ns = 1; p.b_gs = N;
      p.out_rs = N; p.out_gs = M * N;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  p.res_rs = p.out_rs;
  p.res_gs = p.out_gs;
  if (d.dtype == 0) return dispatch_simt<float>(p, d.epi, st);
  if (d.dtype == 1) return dispatch_simt<bf16>(p, d.epi, st);
  return dispatch_simt<f16>(p, d.epi, st);
}

}  // namespace rmx
