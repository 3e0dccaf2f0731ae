// One decode step of the selective scan (the recurrent, token-by-token form
// that the Blelloch article, section 1, recommends for inference): for every
// (batch b, channel d)
//   dt   = softplus(dt_raw[b,d] + bias[d])          (or dt_raw + bias)
//   h[n] = exp(dt*A[d,n]) * h[n] + dt*B[b,n]*x[b,d]  for n < N
//   y    = (sum_n C[b,n]*h[n] + D[d]*x[b,d]) * silu(z[b,d])
// with the state h = state[b,d,:] (fp32) read and written in place.  It is the
// forward pass of ss_fwd_sched for one step from an initial state.
//
// The step is bound by the state traffic (8 bytes per state element: one read,
// one write), so each lane keeps up to kDecodeQuads quads of four states (64
// bytes) in flight: it issues all its loads before any arithmetic.  A group of
// S lanes (S a power of two) serves one row, S = 1 up to 16 states: lane j of
// the group holds the quads j, j+S, ... (one 16-byte load and store each when
// the row allows); the read-out is summed over the group by a butterfly of
// shuffles and lane 0 of the group stores y.  The grid's y axis is the batch
// row, so no thread divides an index.
#pragma once

#include "ss_device.cuh"

namespace ss {

struct DecodeParams {
  float* state;          // [b,d,N] fp32, in place
  const void* x;         // [b,d]
  const void* dt;        // [b,d]
  const float* A;        // [d,N]
  const void* B;         // [b,N]
  const void* C;         // [b,N]
  const float* D;        // [d] or null
  const void* z;         // [b,d] or null
  const float* bias;     // [d] or null
  void* y;               // [b,d]
  int64_t batch0;        // first batch row of this launch (grid.y = batch rows)
  int64_t dim, dstate;
  int softplus;
  int seg_shift;         // log2 of the lanes per row
  int quads;             // ceil(dstate / 4)
};

// Four consecutive elements n0..n0+3 of an fp32 or bf16 row as floats
// (VEC: one 16- or 8-byte load; the caller guarantees alignment and range).
template <typename T, bool VEC>
__device__ __forceinline__ void load4(const T* p, int64_t n0, int64_t N, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float, true>(const float* p, int64_t n0, int64_t, float (&v)[4]) {
  const float4 q = *reinterpret_cast<const float4*>(p + n0);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16, true>(const __nv_bfloat16* p, int64_t n0,
                                                           int64_t, float (&v)[4]) {
  const uint2 q = *reinterpret_cast<const uint2*>(p + n0);
  v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
  v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
}
template <>
__device__ __forceinline__ void load4<float, false>(const float* p, int64_t n0, int64_t N, float (&v)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = n0 + e < N ? p[n0 + e] : 0.f;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16, false>(const __nv_bfloat16* p, int64_t n0,
                                                            int64_t N, float (&v)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = n0 + e < N ? Elem<__nv_bfloat16>::to_f32(p[n0 + e]) : 0.f;
}

constexpr int kDecodeQuads = 4;  // state quads per lane

// grid = (ceil(dim * lanes / 256), batch rows of this launch), block = 256.
// VEC4: dstate % 4 == 0 and state, A (16 bytes) and B, C (4 elements) aligned.
template <typename T, bool VEC4>
__global__ void __launch_bounds__(256) ss_state_update(const DecodeParams p) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t d = t >> p.seg_shift;
  const int lane = (int)(t & ((1 << p.seg_shift) - 1));
  const int64_t b = p.batch0 + blockIdx.y;
  const bool active = d < p.dim;
  const int64_t N = p.dstate;
  const int64_t row = b * p.dim + d;

  float part = 0.f, xv = 0.f;
  if (active) {
    xv = Elem<T>::to_f32(static_cast<const T*>(p.x)[row]);
    float dtv = Elem<T>::to_f32(static_cast<const T*>(p.dt)[row]) + (p.bias ? p.bias[d] : 0.f);
    if (p.softplus) dtv = lo_of(softplus2(splat(dtv)));
    const float du = dtv * xv;
    float* __restrict__ h = p.state + row * N;
    const float* __restrict__ Ad = p.A + d * N;
    const T* __restrict__ Bb = static_cast<const T*>(p.B) + b * N;
    const T* __restrict__ Cb = static_cast<const T*>(p.C) + b * N;
    // every load of the lane first, then the arithmetic, then the stores
    float hv[kDecodeQuads][4], av[kDecodeQuads][4], bv[kDecodeQuads][4], cv[kDecodeQuads][4];
#pragma unroll
    for (int i = 0; i < kDecodeQuads; ++i) {
      const int q = lane + (i << p.seg_shift);
      const int64_t n0 = 4 * (int64_t)q;
      if (q < p.quads) {
        load4<float, VEC4>(h, n0, N, hv[i]);
        load4<float, VEC4>(Ad, n0, N, av[i]);
        load4<T, VEC4>(Bb, n0, N, bv[i]);
        load4<T, VEC4>(Cb, n0, N, cv[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kDecodeQuads; ++i) {
      const int q = lane + (i << p.seg_shift);
      if (q >= p.quads) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = ex2(dtv * av[i][e] * kLog2e);
        hv[i][e] = fmaf(a, hv[i][e], du * bv[i][e]);
        part = fmaf(cv[i][e], hv[i][e], part);  // zero C past dstate adds nothing
      }
    }
#pragma unroll
    for (int i = 0; i < kDecodeQuads; ++i) {
      const int q = lane + (i << p.seg_shift);
      const int64_t n0 = 4 * (int64_t)q;
      if (q >= p.quads) continue;
      if (VEC4) {
        *reinterpret_cast<float4*>(h + n0) = make_float4(hv[i][0], hv[i][1], hv[i][2], hv[i][3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (n0 + e < N) h[n0 + e] = hv[i][e];
      }
    }
  }
  // read-out over the row's lanes (groups of 2^seg_shift, aligned to their size)
  for (int off = (1 << p.seg_shift) >> 1; off > 0; off >>= 1)
    part += __shfl_xor_sync(0xffffffffu, part, off);
  if (active && lane == 0) {
    float yv = part + (p.D ? p.D[d] : 0.f) * xv;
    if (p.z) yv *= silu(Elem<T>::to_f32(static_cast<const T*>(p.z)[row]));
    static_cast<T*>(p.y)[row] = Elem<T>::from_f32(yv);
  }
}

}  // namespace ss
