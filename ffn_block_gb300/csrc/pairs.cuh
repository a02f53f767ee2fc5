// Float-pair access to 16-byte vectors of the storage types, for the packed
// fp32x2 arithmetic of the row kernels (common.cuh holds the arithmetic).
#pragma once

#include "common.cuh"

namespace rmx {

// Two 16-bit elements in one 32-bit word <-> a float pair (lower element in
// .x); packing rounds to nearest even.
template <typename T> __device__ __forceinline__ float2 unpack2w(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2w<bf16>(uint32_t w) { return bf16x2_to_f2(w); }
template <> __device__ __forceinline__ float2 unpack2w<f16>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <typename T> __device__ __forceinline__ uint32_t pack2w(float2 v);
template <> __device__ __forceinline__ uint32_t pack2w<bf16>(float2 v) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2w<f16>(float2 v) {
  const __half2 h = __floats2half2_rn(v.x, v.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// One 16-byte vector of T (16-byte aligned) as 8 / sizeof(T) float pairs.
template <typename T> __device__ __forceinline__ void ld16p(const void* p, float2* v) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 4) {
    v[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
    v[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
  } else {
    v[0] = unpack2w<T>(r.x);
    v[1] = unpack2w<T>(r.y);
    v[2] = unpack2w<T>(r.z);
    v[3] = unpack2w<T>(r.w);
  }
}
template <typename T> __device__ __forceinline__ void st16p(void* p, const float2* v) {
  uint4 r;
  if constexpr (sizeof(T) == 4) {
    r = make_uint4(__float_as_uint(v[0].x), __float_as_uint(v[0].y), __float_as_uint(v[1].x),
                   __float_as_uint(v[1].y));
  } else {
    r = make_uint4(pack2w<T>(v[0]), pack2w<T>(v[1]), pack2w<T>(v[2]), pack2w<T>(v[3]));
  }
  *reinterpret_cast<uint4*>(p) = r;
}
}  // namespace rmx
