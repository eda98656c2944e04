// Score element types of the selector: FP32, bfloat16 given as raw 16-bit
// patterns, and FP8 E4M3 given as raw bytes, each widened exactly to FP32.
// Shared by the selector kernels and the optional row sort.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tk {

// A single score, cached in L2 only (one 32-byte sector, no L1 line fill),
// with the given L2 eviction policy.
__device__ __forceinline__ float ld_keep(const float* p, uint64_t policy) {
  float v;
  asm volatile("ld.global.cg.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(policy));
  return v;
}

// Score element types: FP32, bfloat16 given as raw 16-bit patterns, or FP8
// E4M3 given as raw bytes.  Both narrow formats widen exactly to binary32, so
// every comparison, key and threshold below works on the widened FP32 value.
// kPer16: elements per 16 bytes (one vector load of the ring).
template <class E>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kSize = 4, kPer16 = 4;
  // low bits that are zero in the FP32 bits of every value (none)
  static constexpr int kKeyQuantum = 0;
  __device__ static __forceinline__ float load(const float* p) { return *p; }
  __device__ static __forceinline__ float load_keep(const float* p, uint64_t pol) {
    return ld_keep(p, pol);
  }
  // group k of the elements of one 16-byte unit: four widened values
  __device__ static __forceinline__ float4 group(const uint4& u, int) {
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                       __uint_as_float(u.w));
  }
};
template <>
struct Elem<uint16_t> {
  static constexpr int kSize = 2, kPer16 = 8;
  // a widened bfloat16 has 16 zero low bits: distinct values' order keys
  // lie at least 2^16 apart (on each side of zero)
  static constexpr int kKeyQuantum = 16;
  __device__ static __forceinline__ float widen(uint32_t b) { return __uint_as_float(b << 16); }
  __device__ static __forceinline__ float load(const uint16_t* p) { return widen(*p); }
  __device__ static __forceinline__ float load_keep(const uint16_t* p, uint64_t pol) {
    uint16_t v;
    asm volatile("ld.global.cg.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
    return widen(v);
  }
  __device__ static __forceinline__ float4 group(const uint4& u, int k) {
    const uint32_t a = k ? u.z : u.x, b = k ? u.w : u.y;
    return make_float4(widen(a & 0xFFFFu), widen(a >> 16), widen(b & 0xFFFFu), widen(b >> 16));
  }
};

// FP8 E4M3 in the OCP 8-bit floating-point format (the variant without
// infinities): sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent
// field 0 encodes m * 2^-9, the others (1 + m/8) * 2^(e-7); S.1111.111 is NaN
// (not a supported score; it widens to 480 here).  Every value is a binary32
// value, so the widening below is exact.
template <>
struct Elem<uint8_t> {
  static constexpr int kSize = 1, kPer16 = 16;
  // a widened E4M3 value has at most 3 significant bits: 20 zero low bits
  static constexpr int kKeyQuantum = 20;
  __device__ static __forceinline__ float widen(uint32_t b) {
    const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
    const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
    return __uint_as_float(__float_as_uint(mag) | ((b & 0x80u) << 24));
  }
  __device__ static __forceinline__ float load(const uint8_t* p) { return widen(*p); }
  __device__ static __forceinline__ float load_keep(const uint8_t* p, uint64_t pol) {
    uint16_t v;
    asm volatile("ld.global.cg.L2::cache_hint.u8 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
    return widen(v & 0xFFu);
  }
  __device__ static __forceinline__ float4 group(const uint4& u, int k) {
    const uint32_t w = k == 0 ? u.x : k == 1 ? u.y : k == 2 ? u.z : u.w;
    return make_float4(widen(w & 0xFFu), widen((w >> 8) & 0xFFu), widen((w >> 16) & 0xFFu),
                       widen(w >> 24));
  }
  // the byte pattern of a positive value that E4M3 represents exactly (a
  // widened E4M3 score); for positive values the byte order is the value order
  __device__ static __forceinline__ int32_t pattern_of_positive(float v) {
    const uint32_t b = __float_as_uint(v);
    const int32_t e = (int32_t)(b >> 23) - 127;
    if (e < -6) return (int32_t)(v * 512.0f);  // exponent field 0: m = v * 2^9
    return ((e + 7) << 3) | (int32_t)((b >> 20) & 7u);
  }
};

}  // namespace tk
