// Zero-padded staging copies for blocks whose D or H is not a multiple of 8.
//
// The kernels address rows in whole 16-byte vectors and the tensor-core GEMM
// needs 16-byte row strides, so such a block runs on copies whose rows are
// padded with zeros to a multiple of 8 elements: x, dy and the parameters are
// gathered into padded buffers before the passes, y, dx and the gradients are
// gathered back afterwards.  The zeros are exact no-ops for the contractions
// (zero rows and columns of the weights), and the LayerNorm passes take their
// means over the real columns only.  One thread per destination element, so
// every padded place is written (with 0) and nothing needs clearing first.

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {
namespace {

template <typename E>
__global__ void __launch_bounds__(256) k_pad_copy(const E* __restrict__ src, E* __restrict__ dst, PadMap m,
                                                  int pack) {
  pdl_enter();
  const int hs = m.cols / m.halves, hsp = m.cols_p / m.halves;
  const int dcols = pack ? m.cols_p : m.cols, drows = pack ? m.rows_p : m.rows;
  const size_t total = (size_t)m.outer * drows * dcols;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % dcols);
    const size_t rr = idx / dcols;
    const int r = (int)(rr % drows);
    const size_t o = rr / drows;
    if (pack) {
      // padded (o, r, c) <- logical (o, r, h * hs + cc) with c = h * hsp + cc
      const int h = c / hsp, cc = c - h * hsp;
      const bool real = r < m.rows && cc < hs;
      dst[idx] = real ? src[(o * m.rows + r) * (size_t)m.cols + (size_t)h * hs + cc] : E(0);
    } else {
      // logical (o, r, c) <- padded (o, r, h * hsp + cc) with c = h * hs + cc
      const int h = c / hs, cc = c - h * hs;
      dst[idx] = src[(o * m.rows_p + r) * (size_t)m.cols_p + (size_t)h * hsp + cc];
    }
  }
}

// dst[g][c][r] = src[g * gs + r * rs + c] for r < R, 0 for R <= r < Rp: one
// 32 x 32 tile per CTA through shared memory, reads along c and writes
// along r coalesced.
__global__ void __launch_bounds__(256) k_transpose_f32(const float* __restrict__ src, float* __restrict__ dst,
                                                       int R, int Cc, long long gs, long long rs, int Rp) {
  pdl_enter();
  __shared__ float tile[32][33];
  const int g = blockIdx.z, c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const float* s = src + (size_t)g * gs;
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int r = r0 + ty + k, c = c0 + tx;
    tile[ty + k][tx] = (r < R && c < Cc) ? s[(size_t)r * rs + c] : 0.f;
  }
  __syncthreads();
  float* d = dst + (size_t)g * Cc * Rp;
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int c = c0 + ty + k, r = r0 + tx;
    if (c < Cc && r < Rp) d[(size_t)c * Rp + r] = tile[tx][ty + k];
  }
}

}  // namespace

cudaError_t launch_transpose_f32(const float* src, float* dst, int G, int R, int Cc, long long gs, long long rs,
                                 int Rp, cudaStream_t st) {
  if (G < 0 || R < 0 || Cc < 0 || Rp < R) return cudaErrorInvalidValue;
  if (G == 0 || Cc == 0 || Rp == 0) return cudaSuccess;
  const dim3 grid((Cc + 31) / 32, (Rp + 31) / 32, G);
  return launch_k(k_transpose_f32, grid, dim3(256), 0, st, 1, src, dst, R, Cc, gs, rs, Rp);
}

cudaError_t launch_pad_copy(const void* src, void* dst, int dtype, const PadMap& m, bool pack, cudaStream_t st) {
  if (m.outer < 0 || m.rows < 0 || m.rows > m.rows_p || m.cols > m.cols_p || m.halves < 1 ||
      m.cols % m.halves || m.cols_p % m.halves)
    return cudaErrorInvalidValue;
  const size_t total = (size_t)m.outer * (pack ? (size_t)m.rows_p * m.cols_p : (size_t)m.rows * m.cols);
  if (total == 0) return cudaSuccess;
  const size_t want = (total + 255) / 256;
  const int grid = (int)(want < (size_t)sm_count() * 16 ? want : (size_t)sm_count() * 16);
  if (dtype == 0)
    return launch_k(k_pad_copy<uint32_t>, dim3(grid), dim3(256), 0, st, 1, static_cast<const uint32_t*>(src),
                    static_cast<uint32_t*>(dst), m, pack ? 1 : 0);
  return launch_k(k_pad_copy<uint16_t>, dim3(grid), dim3(256), 0, st, 1, static_cast<const uint16_t*>(src),
                  static_cast<uint16_t*>(dst), m, pack ? 1 : 0);
}

}  // namespace rmx
