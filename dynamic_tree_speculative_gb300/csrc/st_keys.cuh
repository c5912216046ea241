// Order keys of logits and (key, id) composites, shared by the support
// selection kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "st_common.cuh"

namespace st {

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int VEC = 8;
  static constexpr int KEY_BITS = 16;
  static constexpr int ES = 2;
};
template <>
struct Elem<float> {
  static constexpr int VEC = 4;
  static constexpr int KEY_BITS = 32;
  static constexpr int ES = 4;
};

// Order key of element j of a 16-byte vector; flags NaN / +inf.
template <typename T>
__device__ __forceinline__ uint32_t elem_key(const uint4& v, int j, bool& nonfinite);

template <>
__device__ __forceinline__ uint32_t elem_key<__nv_bfloat16>(const uint4& v, int j, bool& nonfinite) {
  const uint32_t w = (j < 2) ? v.x : (j < 4) ? v.y : (j < 6) ? v.z : v.w;
  const uint32_t bits = (w >> (16 * (j & 1))) & 0xffffu;
  if ((bits & 0x7fffu) >= 0x7f80u && bits != 0xff80u) nonfinite = true;  // NaN or +inf
  return bf16_key(bits);
}

template <>
__device__ __forceinline__ uint32_t elem_key<float>(const uint4& v, int j, bool& nonfinite) {
  const uint32_t bits = (j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w;
  if ((bits & 0x7fffffffu) >= 0x7f800000u && bits != 0xff800000u) nonfinite = true;
  return f32_key(bits);
}

template <typename T>
__device__ __forceinline__ uint32_t scalar_key(const uint8_t* row, int v, bool& nonfinite) {
  uint4 x = make_uint4(0, 0, 0, 0);
  if (sizeof(T) == 2) x.x = reinterpret_cast<const uint16_t*>(row)[v];
  else x.x = reinterpret_cast<const uint32_t*>(row)[v];
  return elem_key<T>(x, 0, nonfinite);
}

template <typename T>
__device__ __forceinline__ float key_value(uint32_t key);
template <>
__device__ __forceinline__ float key_value<__nv_bfloat16>(uint32_t key) { return bf16_key_value(key); }
template <>
__device__ __forceinline__ float key_value<float>(uint32_t key) { return __uint_as_float(f32_from_key(key)); }

__device__ __forceinline__ uint64_t make_comp(uint32_t key, uint32_t id) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~id);
}

}  // namespace st
