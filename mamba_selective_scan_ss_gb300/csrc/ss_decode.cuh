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
// one write) and, being short, by how many DRAM round trips it takes.  A CTA
// owns a tile of channels and up to kDecodeRows batch rows; every thread
// issues the loads of all its rows (state quads, x, dt, z) before any
// arithmetic, so the launch is about one wave with one DRAM latency.  A of
// the thread's channel is read once for all its rows, and B, C of the CTA's
// rows (shared by every channel of a batch row) are staged in shared memory.
// A group of S lanes (S a power of two) serves one channel, S = 1 up to 16
// states: lane j of the group holds the quads j, j+S, ... (one 16-byte load
// and store each when the row allows); the read-out is summed over the group
// by a butterfly of shuffles and lane 0 of the group stores y.
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
  int64_t batch, dim, dstate;
  int64_t rows_per_cta;  // batch rows a CTA walks (grid.y = ceil(batch / rows_per_cta))
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

constexpr int kDecodeQuads = 4;    // state quads per lane
constexpr int kDecodeRows = 4;     // batch rows per CTA
constexpr int kDecodeThreads = 128;
constexpr int kDecodeMaxN = 256;   // dstate limit of the decode step

// grid = (ceil(dim * lanes / kDecodeThreads), ceil(batch / rows_per_cta)),
// block = kDecodeThreads, rows_per_cta <= kDecodeRows.  VEC4: dstate % 4 == 0
// and state, A 16-byte aligned.
template <typename T, bool VEC4>
__global__ void __launch_bounds__(kDecodeThreads, 4) ss_state_update(const DecodeParams p) {
  constexpr int R = kDecodeRows, Q = kDecodeQuads;
  __shared__ __align__(16) float bc[R][2][kDecodeMaxN];  // B, C of the CTA's batch rows
  const int tid = threadIdx.x;
  const int64_t t = (int64_t)blockIdx.x * kDecodeThreads + tid;
  const int64_t d = t >> p.seg_shift;
  const int lane = (int)(t & ((1 << p.seg_shift) - 1));
  const bool active = d < p.dim;
  const int64_t dc = active ? d : p.dim - 1;
  const int64_t N = p.dstate;
  const int64_t b0 = (int64_t)blockIdx.y * p.rows_per_cta;
  const int nb = (int)min((int64_t)R, min(p.rows_per_cta, p.batch - b0));
  const T* __restrict__ xs = static_cast<const T*>(p.x);
  const T* __restrict__ dts = static_cast<const T*>(p.dt);
  const T* __restrict__ zs = static_cast<const T*>(p.z);

  // every load first: the rows' state quads and scalars, A, then B/C into smem
  float hv[R][Q][4], xv[R], dtv[R], zv[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r >= nb) continue;
    const int64_t row = (b0 + r) * p.dim + dc;
    const float* hrow = p.state + row * N;
#pragma unroll
    for (int i = 0; i < Q; ++i) {
      const int q = lane + (i << p.seg_shift);
      if (q < p.quads) load4<float, VEC4>(hrow, 4 * (int64_t)q, N, hv[r][i]);
    }
    xv[r] = Elem<T>::to_f32(xs[row]);
    dtv[r] = Elem<T>::to_f32(dts[row]);
    zv[r] = p.z ? Elem<T>::to_f32(zs[row]) : 0.f;
  }
  float av[Q][4];
#pragma unroll
  for (int i = 0; i < Q; ++i) {
    const int q = lane + (i << p.seg_shift);
    if (q < p.quads) load4<float, VEC4>(p.A + dc * N, 4 * (int64_t)q, N, av[i]);
  }
  const float bias = p.bias ? p.bias[dc] : 0.f;
  const float Dd = p.D ? p.D[dc] : 0.f;
  {
    const T* Bs = static_cast<const T*>(p.B) + b0 * N;
    const T* Cs = static_cast<const T*>(p.C) + b0 * N;
    const int64_t nq = 4 * (int64_t)p.quads;  // states past dstate read B = C = 0
    for (int64_t i = tid; i < (int64_t)nb * nq; i += kDecodeThreads) {
      const int64_t r = i / nq, n = i - r * nq;
      bc[r][0][n] = n < N ? Elem<T>::to_f32(Bs[r * N + n]) : 0.f;
      bc[r][1][n] = n < N ? Elem<T>::to_f32(Cs[r * N + n]) : 0.f;
    }
  }
  __syncthreads();

#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r >= nb) continue;
    const int64_t row = (b0 + r) * p.dim + dc;
    float dt = dtv[r] + bias;
    if (p.softplus) dt = lo_of(softplus2(splat(dt)));
    const float du = dt * xv[r];
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < Q; ++i) {
      const int q = lane + (i << p.seg_shift);
      if (q >= p.quads) continue;
      const float4 bq = *reinterpret_cast<const float4*>(&bc[r][0][4 * q]);
      const float4 cq = *reinterpret_cast<const float4*>(&bc[r][1][4 * q]);
      const float bb[4] = {bq.x, bq.y, bq.z, bq.w}, cc[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = ex2(dt * av[i][e] * kLog2e);
        hv[r][i][e] = fmaf(a, hv[r][i][e], du * bb[e]);
        part = fmaf(cc[e], hv[r][i][e], part);  // C past dstate is zero: adds nothing
      }
    }
    if (active) {
      float* __restrict__ h = p.state + row * N;
#pragma unroll
      for (int i = 0; i < Q; ++i) {
        const int q = lane + (i << p.seg_shift);
        const int64_t n0 = 4 * (int64_t)q;
        if (q >= p.quads) continue;
        if (VEC4) {
          *reinterpret_cast<float4*>(h + n0) =
              make_float4(hv[r][i][0], hv[r][i][1], hv[r][i][2], hv[r][i][3]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n0 + e < N) h[n0 + e] = hv[r][i][e];
        }
      }
    }
    // read-out over the row's lanes (groups of 2^seg_shift, aligned to their size)
    for (int off = (1 << p.seg_shift) >> 1; off > 0; off >>= 1)
      part += __shfl_xor_sync(0xffffffffu, part, off);
    if (active && lane == 0) {
      float yv = part + Dd * xv[r];
      if (p.z) yv *= silu(zv[r]);
      static_cast<T*>(p.y)[row] = Elem<T>::from_f32(yv);
    }
  }
}

}  // namespace ss
