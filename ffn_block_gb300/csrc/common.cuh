// Shared device helpers for the RankMixer kernels: storage types, 16-byte
// vector access, warp/block reductions, the device error word and bounded
// waits.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace rmx {

typedef __nv_bfloat16 bf16;
typedef __half f16;

// Device error word: bit flags set by kernels, read and cleared by rmx_check.
enum : unsigned int {
  ERRBIT_WAIT_PRODUCER = 1u << 0,
  ERRBIT_WAIT_MMA = 1u << 1,
  ERRBIT_WAIT_EPILOGUE = 1u << 2,
  ERRBIT_WAIT_DRAIN = 1u << 3,
  ERRBIT_WAIT_TEST = 1u << 4,
  ERRBIT_WAIT_ROWS = 1u << 5,
};

unsigned int* device_error_word();  // host: device address of the error word

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(f16 v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ f16 from_f<f16>(float v) { return __float2half_rn(v); }

// Elements of T in one 16-byte vector.
template <typename T> struct VecN { static constexpr int value = 16 / (int)sizeof(T); };

// Load / store one 16-byte vector of T as floats.  p must be 16-byte aligned.
template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float* v) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
  for (int i = 0; i < VecN<T>::value; ++i) v[i] = to_f(e[i]);
}

template <typename T>
__device__ __forceinline__ void store_vec(T* p, const float* v) {
  uint4 raw;
  T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
  for (int i = 0; i < VecN<T>::value; ++i) e[i] = from_f<T>(v[i]);
  *reinterpret_cast<uint4*>(p) = raw;
}

// Load / store N consecutive elements (N * sizeof(T) = 8 or 16 bytes, aligned).
template <typename T, int N>
__device__ __forceinline__ void load_n(const T* p, float* v) {
  static_assert(N * sizeof(T) == 8 || N * sizeof(T) == 16, "8- or 16-byte access");
  if (N * sizeof(T) == 16) {
    uint4 raw = *reinterpret_cast<const uint4*>(p);
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = to_f(e[i]);
  } else {
    uint2 raw = *reinterpret_cast<const uint2*>(p);
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = to_f(e[i]);
  }
}
template <typename T, int N>
__device__ __forceinline__ void store_n(T* p, const float* v) {
  static_assert(N * sizeof(T) == 8 || N * sizeof(T) == 16, "8- or 16-byte access");
  if (N * sizeof(T) == 16) {
    uint4 raw;
    T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = from_f<T>(v[i]);
    *reinterpret_cast<uint4*>(p) = raw;
  } else {
    uint2 raw;
    T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = from_f<T>(v[i]);
    *reinterpret_cast<uint2*>(p) = raw;
  }
}

// ---------------------------------------------------------------- packed pairs
// Eight consecutive elements of T as four float2 pairs (element 2k in .x,
// 2k+1 in .y), for the packed fp32x2 arithmetic of sm_100+ (__ffma2_rn,
// __fadd2_rn, __fmul2_rn: each component rounds exactly as the scalar
// operation does, so a pair costs one instruction and changes no result).
// 16-bit types: one 16-byte access; float: two.  p must be 16-byte aligned.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  // bf16 is the top half of an fp32: shifting into place is exact.
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <typename T> __device__ __forceinline__ void ld8(const T* p, float2 (&v)[4]);
template <> __device__ __forceinline__ void ld8<bf16>(const bf16* p, float2 (&v)[4]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16x2_to_f2(r.x);
  v[1] = bf16x2_to_f2(r.y);
  v[2] = bf16x2_to_f2(r.z);
  v[3] = bf16x2_to_f2(r.w);
}
template <> __device__ __forceinline__ void ld8<f16>(const f16* p, float2 (&v)[4]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&r);
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = __half22float2(h[k]);
}
template <> __device__ __forceinline__ void ld8<float>(const float* p, float2 (&v)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = make_float2(a.x, a.y);
  v[1] = make_float2(a.z, a.w);
  v[2] = make_float2(b.x, b.y);
  v[3] = make_float2(b.z, b.w);
}
template <typename T> __device__ __forceinline__ void st8(T* p, const float2 (&v)[4]);
template <> __device__ __forceinline__ void st8<bf16>(bf16* p, const float2 (&v)[4]) {
  uint4 r;
  uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[k].x, v[k].y);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = r;
}
template <> __device__ __forceinline__ void st8<f16>(f16* p, const float2 (&v)[4]) {
  uint4 r;
  uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 h = __floats2half2_rn(v[k].x, v[k].y);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = r;
}
template <> __device__ __forceinline__ void st8<float>(float* p, const float2 (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
}
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// Logistic function 1 / (1 + e^-g), with e^-g = 2^(-g * log2(e)) (change of
// base) on the hardware's base-2 exponential and its reciprocal, both the
// flush-to-zero approximations of the PTX ISA (ex2.approx.ftz,
// rcp.approx.ftz): a few ulp of error, far inside the block's tolerances.
// The limits come out exactly: e^-g flushes to 0 for large g (result 1) and
// overflows to +inf for very negative g (result 0).
__device__ __forceinline__ float sigmoid_fast(float g) {
  constexpr float kLog2e = 1.4426950408889634f;
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -kLog2e));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}

// The same function on a pair (identical results, component by component).
__device__ __forceinline__ float2 sigmoid_fast2(float2 g) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float2 a = mul2(g, f2(-kLog2e));
  float2 e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(a.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(a.y));
  const float2 d = add2(f2(1.0f), e);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(d.y));
  return r;
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums NV floats over the whole block.  `red` is shared scratch of at least
// 2 * 32 * NV floats; `slot` alternates between calls so that one
// __syncthreads per call suffices.  Every thread gets the same result, summed
// in a fixed order (deterministic).
template <int NV>
__device__ __forceinline__ void block_sum(float* v, float* red, int& slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = warp_sum(v[i]);
  float* r = red + slot * 32 * NV;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) r[warp * NV + i] = v[i];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += r[w * NV + i];
    v[i] = s;
  }
  slot ^= 1;
}

// ---------------------------------------------------------------- timing / waits
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase of `bar` with the given parity has completed, for at
// most `limit_ns` nanoseconds.  On expiry sets `errbit` in the device error
// word and `*abort` (shared), and returns false.  Returns false at once if
// `*abort` is already set.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  unsigned int* err, unsigned int errbit,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (((++n) & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(err, errbit);
        *abort = 1;
        return false;
      }
    }
  }
}

// Default limit for the GEMM pipeline waits: far longer than any tile takes,
// short enough that a broken pipeline returns instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;  // 2 s

}  // namespace rmx

namespace rmx {

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Bulk copy global -> shared (no tensor map): both addresses 16-byte aligned,
// size a multiple of 16; completion is counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// One box of a rank-2 tensor map into shared memory (128-byte aligned),
// completion counted on `bar` in bytes (the whole box, zero-filled parts
// included).  c0 is the inner coordinate in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Chan / Golub / LeVeque merge of (count, mean, M2) partial statistics.
struct Moments {
  float n, mean, m2;
};
__device__ __forceinline__ Moments merge_moments(const Moments& a, const Moments& b) {
  const float n = a.n + b.n;
  if (n == 0.f) return a;
  const float d = b.mean - a.mean;
  const float wb = b.n / n;
  Moments r;
  r.n = n;
  r.mean = a.mean + d * wb;
  r.m2 = a.m2 + b.m2 + d * d * a.n * wb;
  return r;
}
__device__ __forceinline__ Moments warp_merge_moments(Moments m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Moments other;
    other.n = __shfl_xor_sync(0xffffffffu, m.n, o);
    other.mean = __shfl_xor_sync(0xffffffffu, m.mean, o);
    other.m2 = __shfl_xor_sync(0xffffffffu, m.m2, o);
    // Merge in a fixed order (lower lane first) so every lane gets the same bits.
    m = ((threadIdx.x & o) == 0) ? merge_moments(m, other) : merge_moments(other, m);
  }
  return m;
}

}  // namespace rmx
