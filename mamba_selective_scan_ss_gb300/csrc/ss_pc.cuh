// Forward pass with B and C given per channel, [batch, dim, dstate, seqlen]:
// the layout of the task spec's base kernel signature ("ТЕХНИЧЕСКОЕ ЗАДАНИЕ:
// Реализовать selective scan (Mamba)", Этап 2 step 3, which indexes B and C
// by batch, channel and step with a single state), taken to dstate states,
// with the recurrence of the same page's Этап 1 and of "Mamba CUDA 实现解析"
// eq (4)-(7):
//   h[n] = exp(dt*A[d,n]) * h[n] + dt*B[b,d,n,t]*u,  y = sum_n C[b,d,n,t]*h[n] + D*u
//
// Nothing is shared between channels, so every state update reads its own B
// and C values: the pass is bound by HBM traffic (2*dstate B/C elements per
// row and step against four row streams).  A group of S lanes (S a power of
// two, dstate <= 4*S <= 128) serves one row; lane j holds states [4j, 4j+4)
// and streams their B and C rows 32 bytes (8 fp32 or 16 bf16 steps) at a
// time, a whole DRAM sector per row, with the next 32 bytes' loads in flight.
// Above 128 states a row takes 64 lanes (two warps of the CTA): each warp
// sums its read-out by shuffles and the second warp hands its sums for the
// iteration's steps to the first through shared memory (double-buffered, one
// CTA barrier per iteration).
// One CTA per SM: with 64 rows per SM the partly read L2 lines of all row
// streams (about 44 MB over the GPU) stay in L2 until they are used up, so
// DRAM delivers each byte once.  dt, du and
// the gate are computed by every lane of the row from the row's own vector
// loads (the same 32 bytes for all its lanes); the read-out is summed over the
// group by a butterfly of shuffles and lane 0 stores y.
#pragma once

#include "ss_device.cuh"

namespace ss {

struct PcParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;         // [b,d,N,L]
  const void* C;         // [b,d,N,L]
  const float* D;
  const void* z;
  const float* bias;
  int softplus;
  void* y;
  float* last_state;
  const float* h0;       // [b,d,N] state before step 0, or null (zero)
  int64_t rows, dim, dstate, seqlen;
  int seg_shift;         // log2 of the lanes per row
};

// Steps per iteration: 32 bytes of every stream (a whole DRAM sector), so
// each fetched sector is used at once.
template <typename T>
constexpr int kPcSteps = 2 * Elem<T>::kVec;

// 32 bytes (kPcSteps steps) of a row.  VEC: kept as the raw bytes and widened
// element by element when used (half the registers of floats for bf16);
// otherwise loaded element by element as floats, zero past the row's end.
template <typename T, bool VEC>
struct PcVec;
__device__ __forceinline__ unsigned word_of(const uint4& r, int i) {
  return i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
}
// One 32-byte load (a whole sector) of read-only data: a single L1 access per
// lane instead of two 16-byte ones (256-bit loads, sm_100 family; the address
// must be 32-byte aligned).
__device__ __forceinline__ void ld32B(const void* p, uint4 (&r)[2]) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0].x), "=r"(r[0].y), "=r"(r[0].z), "=r"(r[0].w), "=r"(r[1].x),
                 "=r"(r[1].y), "=r"(r[1].z), "=r"(r[1].w)
               : "l"(p));
}
template <>
struct PcVec<float, true> {
  uint4 r[2];
  __device__ __forceinline__ void load(const float* row, int64_t t, int64_t) { ld32B(row + t, r); }
  __device__ __forceinline__ float at(int e) const { return __uint_as_float(word_of(r[e >> 2], e & 3)); }
};
template <>
struct PcVec<__nv_bfloat16, true> {
  uint4 r[2];
  __device__ __forceinline__ void load(const __nv_bfloat16* row, int64_t t, int64_t) {
    ld32B(row + t, r);
  }
  __device__ __forceinline__ float at(int e) const {
    const unsigned w = word_of(r[e >> 3], (e >> 1) & 3);
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};
template <typename T>
struct PcVec<T, false> {
  float f[kPcSteps<T>];
  __device__ __forceinline__ void load(const T* row, int64_t t, int64_t L) {
#pragma unroll
    for (int e = 0; e < kPcSteps<T>; ++e) f[e] = t + e < L ? Elem<T>::to_f32(row[t + e]) : 0.f;
  }
  __device__ __forceinline__ float at(int e) const { return f[e]; }
};

// The streams of one vector for one lane: u, delta, z of the row and B, C of
// the lane's four states.
template <typename T, bool VEC, bool HAS_Z>
struct PcStep {
  PcVec<T, VEC> u, x, z, b[4], c[4];
};

// grid = ceil(rows * 2^seg_shift / block); block = 256 for WIDE (four rows of
// 64 lanes), else any multiple of 32 up to 256.  VEC: seqlen a multiple
// of kPcSteps and every input row 32-byte aligned (y 16-byte aligned).  WIDE:
// 64 lanes per row (seg_shift 6, dstate up to 256).
template <typename T, bool HAS_Z, bool VEC, bool WIDE>
__global__ void __launch_bounds__(256, 1) ss_fwd_pc(const PcParams p) {
  constexpr int V = kPcSteps<T>;
  __shared__ float s_half[WIDE ? 2 : 1][WIDE ? 4 : 1][V];  // [buffer][row of the CTA][step]
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = gid >> p.seg_shift;
  const int lane = (int)(gid & ((1 << p.seg_shift) - 1));
  const bool active = row < p.rows;
  const int64_t rc = active ? row : p.rows - 1;
  const int64_t d = rc % p.dim;
  const int64_t L = p.seqlen, N = p.dstate;
  const int n0 = 4 * lane;

  const T* __restrict__ ug = static_cast<const T*>(p.u) + rc * L;
  const T* __restrict__ dg = static_cast<const T*>(p.delta) + rc * L;
  const T* __restrict__ zg = static_cast<const T*>(p.z) + rc * L;
  const T* Bq[4];
  const T* Cq[4];
  float A2[4], h[4];
  bool has[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    has[e] = n0 + e < N;
    const int64_t n = has[e] ? n0 + e : N - 1;  // past dstate: a valid row, zero weight
    Bq[e] = static_cast<const T*>(p.B) + (rc * N + n) * L;
    Cq[e] = static_cast<const T*>(p.C) + (rc * N + n) * L;
    A2[e] = has[e] ? p.A[d * N + n] * kLog2e : 0.f;
    h[e] = (has[e] && p.h0) ? p.h0[rc * N + n] : 0.f;
  }
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.D ? p.D[d] : 0.f;

  auto load = [&](int64_t t, PcStep<T, VEC, HAS_Z>& v) {
    v.u.load(ug, t, L);
    v.x.load(dg, t, L);
    if (HAS_Z) v.z.load(zg, t, L);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v.b[e].load(Bq[e], t, L);
      v.c[e].load(Cq[e], t, L);
    }
  };
  // vector path: the next iteration's loads are in flight while this one is
  // used; the element-wise path (a correctness path) loads at each iteration
  PcStep<T, VEC, HAS_Z> cur, nxt;
  if (VEC) load(0, cur);
  const int warp_lanes = WIDE ? 32 : (1 << p.seg_shift);
  for (int64_t t0 = 0; t0 < L; t0 += V) {
    if (VEC) {
      if (t0 + V < L) load(t0 + V, nxt);
    } else {
      load(t0, cur);
    }
    float yv[V];  // the read-out of each step, summed over the warp's lanes of the row
#pragma unroll
    for (int s = 0; s < V; ++s) {
      yv[s] = 0.f;
      if (!VEC && t0 + s >= L) continue;  // padding past the row's end (warp-uniform)
      const float x = cur.x.at(s) + bias;
      const float dtv = p.softplus ? lo_of(softplus2(splat(x))) : x;
      const float du = dtv * cur.u.at(s);
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = ex2(dtv * A2[e]);
        h[e] = fmaf(a, h[e], du * (has[e] ? cur.b[e].at(s) : 0.f));
        part = fmaf(has[e] ? cur.c[e].at(s) : 0.f, h[e], part);
      }
      for (int off = warp_lanes >> 1; off > 0; off >>= 1)
        part += __shfl_xor_sync(0xffffffffu, part, off);
      yv[s] = part;
    }
    if constexpr (WIDE) {
      // the second warp of each row hands its sums to the first
      const int buf = (int)((t0 / V) & 1), crow = (int)(threadIdx.x >> 6);
      if (lane == 32) {
#pragma unroll
        for (int s = 0; s < V; ++s) s_half[buf][crow][s] = yv[s];
      }
      __syncthreads();
      if (lane == 0) {
#pragma unroll
        for (int s = 0; s < V; ++s) yv[s] += s_half[buf][crow][s];
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < V; ++s) {
        float y = fmaf(Dd, cur.u.at(s), yv[s]);
        if (HAS_Z) y *= silu(cur.z.at(s));
        yv[s] = y;
      }
    }
    if (active && lane == 0) {
      T* yo = static_cast<T*>(p.y) + rc * L + t0;
      if (VEC) {
        constexpr int H = V / 2;  // one 16-byte store per half
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          f2 pr[H / 2];
#pragma unroll
          for (int m = 0; m < H / 2; ++m) pr[m] = pack(yv[q * H + 2 * m], yv[q * H + 2 * m + 1]);
          *reinterpret_cast<uint4*>(yo + q * H) = from_pairs<T>(pr);
        }
      } else {
#pragma unroll
        for (int s = 0; s < V; ++s)
          if (t0 + s < L) yo[s] = Elem<T>::from_f32(yv[s]);
      }
    }
    if (VEC) cur = nxt;
  }
  if (active && p.last_state) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (has[e]) p.last_state[rc * N + n0 + e] = h[e];
  }
}

}  // namespace ss
