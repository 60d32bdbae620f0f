// Shared device helpers of the lin_state library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lin_state.h"

namespace lin {

// ---- storage conversions --------------------------------------------------

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Load element i of an f32 or bf16 array.
__device__ __forceinline__ float load_elem(const void* p, int64_t i, int dtype) {
  if (dtype == LIN_BF16)
    return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}
__device__ __forceinline__ void store_elem(void* p, int64_t i, int dtype, float v) {
  if (dtype == LIN_BF16)
    reinterpret_cast<uint16_t*>(p)[i] = f32_to_bf16_bits(v);
  else
    reinterpret_cast<float*>(p)[i] = v;
}
// Round a value to what the storage dtype can hold (RNE), staying in fp32.
__device__ __forceinline__ float round_to_dtype(float v, int dtype) {
  return dtype == LIN_BF16 ? bf16_bits_to_f32(f32_to_bf16_bits(v)) : v;
}

// 8 consecutive elements (one 16-byte bf16 vector or two float4s).
template <int DT>
struct Vec8;

template <>
struct Vec8<LIN_F32> {
  static __device__ __forceinline__ void load(const void* p, float (&v)[8]) {
    const float4* q = reinterpret_cast<const float4*>(p);
    float4 a = q[0], b = q[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[8]) {
    float4* q = reinterpret_cast<float4*>(p);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  static __device__ __forceinline__ void round(float (&)[8]) {}
};

template <>
struct Vec8<LIN_BF16> {
  static __device__ __forceinline__ void load(const void* p, float (&v)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);  // .x = low half
      w[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void round(float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = bf16_bits_to_f32(f32_to_bf16_bits(v[i]));
  }
};

// ---- packed fp32 pairs (two lanes of fp32 arithmetic per instruction) ----
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2sum(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 8 consecutive elements as 4 packed fp32 pairs, element 2i in the low half.
template <int DT>
struct Pair8;

template <>
struct Pair8<LIN_F32> {
  static __device__ __forceinline__ void load(const void* p, uint64_t (&v)[4]) {
    const ulonglong2* q = reinterpret_cast<const ulonglong2*>(p);
    const ulonglong2 a = q[0], b = q[1];
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  }
  static __device__ __forceinline__ void store(void* p, const uint64_t (&v)[4]) {
    ulonglong2* q = reinterpret_cast<ulonglong2*>(p);
    q[0] = make_ulonglong2(v[0], v[1]);
    q[1] = make_ulonglong2(v[2], v[3]);
  }
};

template <>
struct Pair8<LIN_BF16> {
  static __device__ __forceinline__ void load(const void* p, uint64_t (&v)[4]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = f2pack(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  static __device__ __forceinline__ uint32_t pack(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));  // hi -> upper half
    return r;
  }
  static __device__ __forceinline__ void store(void* p, const uint64_t (&v)[4]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack(v[0]), pack(v[1]), pack(v[2]), pack(v[3]));
  }
};

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float silu(float y) { return __fdividef(y, 1.0f + __expf(-y)); }

// SiLU as (y/2)(1 + tanh(y/2)): one transcendental, relative error about 2^-11
__device__ __forceinline__ float silu_tanh(float y) {
  const float h = 0.5f * y;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}

}  // namespace lin
