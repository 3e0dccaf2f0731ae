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

__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 splat(float x) { return pack(x, x); }
__device__ __forceinline__ float lo_of(f2 p) {
  float lo, hi;
  unpack(p, lo, hi);
  return lo;
}
__device__ __forceinline__ float hi_of(f2 p) {
  float lo, hi;
  unpack(p, lo, hi);
  return hi;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- step size and gate, two steps at a time ------------------------------------
// log1p(e) for e in [0, 1] as e * g(e), g a polynomial fitted by least squares
// on Chebyshev nodes of [0, 1] to log1p(e)/e (the fit is reproduced by
// softplus_fit.py beside the package).  Degree 8 for fp32 I/O: max relative
// error of the fp32 evaluation 1.7e-7 over (0, 1], tiny e included.
__device__ __forceinline__ f2 log1p_unit2(f2 e) {
  f2 g = splat(0.005253458f);
  g = fma2(g, e, splat(-0.029588507f));
  g = fma2(g, e, splat(0.07836167f));
  g = fma2(g, e, splat(-0.1367477f));
  g = fma2(g, e, splat(0.1911143f));
  g = fma2(g, e, splat(-0.2484437f));
  g = fma2(g, e, splat(0.3331927f));
  g = fma2(g, e, splat(-0.49999502f));
  g = fma2(g, e, splat(1.0f));
  return mul2(e, g);
}
// Degree 5 for bf16 I/O: max relative error 8.8e-6, far below what the bf16
// rounding of delta already puts into dt (2^-9 |delta| in the exponent).
__device__ __forceinline__ f2 log1p_unit2_d5(f2 e) {
  f2 g = splat(-0.023979573f);
  g = fma2(g, e, splat(0.10150005f));
  g = fma2(g, e, splat(-0.2102937f));
  g = fma2(g, e, splat(0.32529515f));
  g = fma2(g, e, splat(-0.4993726f));
  g = fma2(g, e, splat(0.99999183f));
  return mul2(e, g);
}

// softplus(x) = max(x, 0) + log1p(e^-|x|) on a pair of steps; e^-|x| is in
// (0, 1], so nothing overflows and small results keep their relative precision.
// BF16IO: the inputs are bf16, so the degree-5 log1p is accurate enough.
template <bool BF16IO = false>
__device__ __forceinline__ f2 softplus2(f2 x) {
  float x0, x1;
  unpack(x, x0, x1);
  const f2 e = pack(ex2(-fabsf(x0) * kLog2e), ex2(-fabsf(x1) * kLog2e));
  return add2(pack(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), BF16IO ? log1p_unit2_d5(e) : log1p_unit2(e));
}

// silu(z) = z / (1 + e^-z) on a pair of steps
__device__ __forceinline__ f2 silu2(f2 z) {
  const f2 e = ex2x2(mul2(z, splat(-kLog2e)));
  const f2 d = add2(e, splat(1.f));
  float d0, d1;
  unpack(d, d0, d1);
  return mul2(z, pack(rcp_approx(d0), rcp_approx(d1)));
}

// ---- step size and gate (scalar path) -------------------------------------------
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

// A 16-byte vector of V elements as V/2 fp32 pairs (consecutive steps).
template <typename T>
__device__ __forceinline__ void to_pairs(const uint4& raw, f2 (&out)[Elem<T>::kVec / 2]);
template <>
__device__ __forceinline__ void to_pairs<float>(const uint4& raw, f2 (&out)[2]) {
  out[0] = pack(__uint_as_float(raw.x), __uint_as_float(raw.y));
  out[1] = pack(__uint_as_float(raw.z), __uint_as_float(raw.w));
}
template <>
__device__ __forceinline__ void to_pairs<__nv_bfloat16>(const uint4& raw, f2 (&out)[4]) {
  const unsigned w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)  // low half is the earlier step
    out[i] = pack(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
// ... and back (bf16: round to nearest even)
template <typename T>
__device__ __forceinline__ uint4 from_pairs(const f2 (&in)[Elem<T>::kVec / 2]);
template <>
__device__ __forceinline__ uint4 from_pairs<float>(const f2 (&in)[2]) {
  float a, b, c, d;
  unpack(in[0], a, b);
  unpack(in[1], c, d);
  return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c),
                    __float_as_uint(d));
}
template <>
__device__ __forceinline__ uint4 from_pairs<__nv_bfloat16>(const f2 (&in)[4]) {
  unsigned w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    unpack(in[i], lo, hi);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(hi), "f"(lo));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

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
