// Device helpers of the selective-scan kernels: fast transcendentals, packed
// f32x2 arithmetic (sm_100 family) and element conversion.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace ss {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x with the MUFU ex2 unit (flush-to-zero: results below 2^-126 are 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- packed pairs: two fp32 lanes in one 64-bit register -------------------
struct f2 {
  unsigned long long v;
};

__device__ __forceinline__ f2 pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack(f2 p, float& lo, float& hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p.v));
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}
__device__ __forceinline__ f2 ex2x2(f2 x) {
  float lo, hi;
  unpack(x, lo, hi);
  return pack(ex2(lo), ex2(hi));
}

// ---- step size and gate -------------------------------------------------------
// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^-|x|); e^-|x| is in (0, 1],
// so neither term overflows and small results keep full relative precision.
__device__ __forceinline__ float softplus(float x) {
  const float e = ex2(-fabsf(x) * kLog2e);
  return fmaxf(x, 0.f) + log1pf(e);
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z)
__device__ __forceinline__ float silu(float z) {
  return __fdividef(z, 1.f + ex2(-z * kLog2e));
}

// ---- element types ---------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static float to_f32(float x) { return x; }
  __device__ __forceinline__ static float from_f32(float x) { return x; }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// 16-byte vector of V elements, loaded/stored whole.
template <typename T>
struct alignas(16) Vec16 {
  T e[Elem<T>::kVec];
};

template <typename T>
__device__ __forceinline__ Vec16<T> ldg_vec(const T* p) {
  Vec16<T> v;
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
  *reinterpret_cast<uint4*>(&v) = raw;
  return v;
}

template <typename T>
__device__ __forceinline__ void stg_vec(T* p, const Vec16<T>& v) {
  *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(&v);
}

// ---- asynchronous global -> shared copies (per-thread, 16 bytes) -------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace ss
