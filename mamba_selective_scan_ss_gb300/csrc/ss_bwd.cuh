// Backward pass of the selective-scan forward (up to 16 states, zero initial
// state): the gradients of u, delta, A, B, C, D, z and delta_bias for a loss
// whose gradient is dy on y (and dlast on last_state).  The task spec asks for
// a backward verified with gradcheck ("ТЕХНИЧЕСКОЕ ЗАДАНИЕ: Реализовать
// selective scan (Mamba)", Этап 3 step 4 and section 5); the formulas are the
// chain rule through the forward's definition:
//   dy'_t = dy_t silu(z_t),  dz_t = dy_t y'_t silu'(z_t),  dD += dy'_t u_t
//   g_t[n] = C[n,t] dy'_t + a_{t+1}[n] g_{t+1}[n]          (g = dL/dh)
//   dC[n,t] += dy'_t h_t[n],  dB[n,t] += g_t[n] dt_t u_t
//   dA[n] += g_t[n] dt_t a_t[n] h_{t-1}[n]
//   d(dt_t) = sum_n g_t[n] (A[n] a_t[n] h_{t-1}[n] + B[n,t] u_t)
//   du_t = dy'_t D + sum_n g_t[n] dt_t B[n,t]
//   ddelta_t = d(dt_t) sigmoid(delta_t + bias)   (1 without softplus),  dbias += ddelta_t
//
// Layout: one thread per row with all (up to 16) states in registers, as in
// the forward, so the row's scalars (dt, du, the gate) and its sums over the
// states (d(dt), du, the pre-gate read-out) stay inside the thread.  A CTA
// holds 64 rows; the B/C values of each block of kBwdBlock steps are staged
// once in shared memory and read as broadcasts.  The one exchange between
// threads is the sum of dB/dC over the rows, step by step and within each
// warp (no CTA barrier): every thread writes its 32 contributions to a padded
// table and lane k of the warp adds column k over the warp's 32 rows in order.
//
// Time: a forward pass stores the state every kBwdBlock steps (checkpoints in
// scratch); the reverse pass then, block by block from the end, recomputes the
// block's states from its checkpoint into shared memory and runs the reverse
// recurrence over them (decays recomputed with ex2).
//
// Reductions are deterministic: dB/dC per warp in row order, then
// ss_bwd_reduce_bc over the CTAs of a batch row and their warps in order; dA, dD and dbias
// per (batch, channel), then ss_bwd_reduce_rows over the batch in order.
#pragma once

#include "ss_device.cuh"

namespace ss {

constexpr int kBwdBlock = 8;       // steps per recomputed block (and checkpoint spacing)
constexpr int kBwdRows = 64;       // rows per CTA (one thread each)
constexpr int kBwdLanes = 16;      // states per group (dstate <= 16)
constexpr int kBwdThreads = kBwdRows;

struct BwdParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* bias;
  int softplus;
  const void* dy;
  const float* dlast;   // [b,d,N] or null
  void* du;             // [b,d,L] dtype
  void* ddelta;         // [b,d,L] dtype
  void* dz;             // [b,d,L] dtype (z present)
  float* ckpt;          // [ctas][nblk][16][64] states at the end of each block
  float* part_bc;       // [ctas][2][16][L] per-CTA sums of dB, dC
  float* part_a;        // [b][d][16] per-row sums of dA
  float* part_dd;       // [b][d][2] per-row sums of dD, dbias
  float* dA;            // [d,N]
  float* dB;            // [b,N,L]
  float* dC;            // [b,N,L]
  float* dD;            // [d] or null
  float* dbias;         // [d] or null
  int64_t batch, dim, dstate, seqlen;
  int64_t dtiles;       // CTAs per batch row: ceil(dim / 64)
  int64_t nblk;         // ceil(seqlen / kBwdBlock)
  int vec;              // rows 16-byte aligned: a block's row values load as 16-byte vectors
};

// Steps [t0, t0 + kBwdBlock) of one row as floats: 16-byte loads when the
// block is whole and the row aligned (vec), else one element at a time.
template <typename T>
__device__ __forceinline__ void load_block(const T* row, int64_t t0, int cnt, bool vec,
                                           float (&out)[kBwdBlock]) {
  constexpr int V = Elem<T>::kVec;  // elements per 16 bytes (4 or 8)
  if (vec && cnt == kBwdBlock) {
#pragma unroll
    for (int q = 0; q < kBwdBlock / V; ++q) {
      const Vec16<T> v = *reinterpret_cast<const Vec16<T>*>(row + t0 + q * V);
#pragma unroll
      for (int e = 0; e < V; ++e) out[q * V + e] = Elem<T>::to_f32(v.e[e]);
    }
  } else {
#pragma unroll
    for (int st = 0; st < kBwdBlock; ++st) out[st] = st < cnt ? Elem<T>::to_f32(row[t0 + st]) : 0.f;
  }
}

__device__ __forceinline__ float sigmoid_f(float x) { return rcp_approx(1.f + ex2(-x * kLog2e)); }

template <typename T, bool HAS_Z>
__global__ void __launch_bounds__(kBwdThreads, 6) ss_bwd_main(const BwdParams p) {
  constexpr int S = kBwdBlock, NT = kBwdLanes;
  __shared__ float bc[2][S][NT];                 // B, C of the block's steps
  __shared__ float hp[S][NT][kBwdRows];          // state before each step of the block
  __shared__ float red[kBwdRows][2 * NT + 1];    // one step's dC (0..15), dB (16..31) per row
  __shared__ float wpart[kBwdRows / 32][S][2 * NT];  // the block's per-warp dC/dB sums

  const int tid = threadIdx.x;
  const int64_t cta = blockIdx.x;
  const int64_t b = cta / p.dtiles;
  const int64_t d = (cta - b * p.dtiles) * kBwdRows + tid;
  const bool valid = d < p.dim;
  const int64_t dc = valid ? d : p.dim - 1;
  const int64_t L = p.seqlen, N = p.dstate;
  const int64_t row = b * p.dim + dc;

  const T* __restrict__ ug = static_cast<const T*>(p.u) + row * L;
  const T* __restrict__ dg = static_cast<const T*>(p.delta) + row * L;
  const T* __restrict__ zg = static_cast<const T*>(p.z) + row * L;
  const T* __restrict__ yg = static_cast<const T*>(p.dy) + row * L;
  const T* __restrict__ Bg = static_cast<const T*>(p.B) + b * N * L;
  const T* __restrict__ Cg = static_cast<const T*>(p.C) + b * N * L;
  float A2[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) A2[n] = n < N ? p.A[dc * N + n] * kLog2e : 0.f;
  const float bias = p.bias ? p.bias[dc] : 0.f;
  const float Dd = p.D ? p.D[dc] : 0.f;
  auto ck = [&](int64_t blk, int n) -> float& {
    return p.ckpt[((cta * p.nblk + blk) * NT + n) * kBwdRows + tid];
  };
  // B (and C) of steps [t0, t0 + cnt) into shared memory, zero past dstate
  auto stage = [&](int64_t t0, int cnt, int tensors) {
    for (int i = tid; i < tensors * NT * S; i += kBwdThreads) {
      const int m = i / (NT * S), n = (i / S) % NT, st = i % S;
      const T* src = m == 0 ? Bg : Cg;
      bc[m][st][n] = (st < cnt && n < N) ? Elem<T>::to_f32(src[(int64_t)n * L + t0 + st]) : 0.f;
    }
  };
  const bool vec = p.vec != 0;
  auto dt_of = [&](float x) { return p.softplus ? lo_of(softplus2(splat(x))) : x; };

  // ---- forward: checkpoints at the end of every block but the last ----
  {
    float h[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) h[n] = 0.f;
    for (int64_t blk = 0; blk < p.nblk; ++blk) {
      const int64_t t0 = blk * S;
      const int cnt = (int)min((int64_t)S, L - t0);
      stage(t0, cnt, 1);
      float xs[S], us[S];
      load_block<T>(dg, t0, cnt, vec, xs);
      load_block<T>(ug, t0, cnt, vec, us);
      __syncthreads();
#pragma unroll
      for (int st = 0; st < S; ++st) {
        if (st < cnt) {
          const float dtv = dt_of(xs[st] + bias);
          const float du = dtv * us[st];
#pragma unroll
          for (int n = 0; n < NT; ++n) h[n] = fmaf(ex2(dtv * A2[n]), h[n], du * bc[0][st][n]);
        }
      }
      if (blk + 1 < p.nblk) {
#pragma unroll
        for (int n = 0; n < NT; ++n) ck(blk, n) = h[n];
      }
      __syncthreads();  // bc is restaged by the next block
    }
  }

  // ---- reverse, block by block ----
  float g[NT], dA_acc[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    g[n] = (valid && n < N && p.dlast) ? p.dlast[row * N + n] : 0.f;
    dA_acc[n] = 0.f;
  }
  float dD_acc = 0.f, dbias_acc = 0.f;
  for (int64_t blk = p.nblk - 1; blk >= 0; --blk) {
    const int64_t t0 = blk * S;
    const int cnt = (int)min((int64_t)S, L - t0);
    stage(t0, cnt, 2);
    // the row's scalars of the block's steps
    float xs[S], dts[S], us[S], dys[S], zs[S];
    load_block<T>(dg, t0, cnt, vec, xs);
    load_block<T>(ug, t0, cnt, vec, us);
    load_block<T>(yg, t0, cnt, vec, dys);
    if (HAS_Z) load_block<T>(zg, t0, cnt, vec, zs);
#pragma unroll
    for (int st = 0; st < S; ++st) {
      xs[st] += bias;
      dts[st] = dt_of(xs[st]);
      if (!valid) dys[st] = 0.f;
      if (!HAS_Z) zs[st] = 0.f;
    }
    __syncthreads();
    // recompute the block's states from its checkpoint
    {
      float h[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) h[n] = blk > 0 ? ck(blk - 1, n) : 0.f;
#pragma unroll
      for (int st = 0; st < S; ++st) {
        if (st < cnt) {
          const float du = dts[st] * us[st];
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            hp[st][n][tid] = h[n];
            h[n] = fmaf(ex2(dts[st] * A2[n]), h[n], du * bc[0][st][n]);
          }
        }
      }
    }
    // reverse over the block's steps
#pragma unroll
    for (int st = S - 1; st >= 0; --st) {
      if (st >= cnt) continue;
      const int64_t t = t0 + st;
      float dyp = dys[st], sig = 0.f;
      if (HAS_Z) {
        sig = sigmoid_f(zs[st]);
        dyp = dys[st] * zs[st] * sig;
      }
      const float dtv = dts[st], u = us[st], du = dtv * u;
      float ddt_a[2] = {0.f, 0.f}, ddt_b[2] = {0.f, 0.f}, dsum[2] = {0.f, 0.f},
            ysum[2] = {0.f, 0.f};
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float prev = hp[st][n][tid];
        const float a = ex2(dtv * A2[n]);
        const float bb = bc[0][st][n], cc = bc[1][st][n];
        const float ap = a * prev;
        const float ht = fmaf(du, bb, ap);
        const float gn = fmaf(cc, dyp, g[n]);
        const float gd = gn * dtv;
        red[tid][n] = dyp * ht;           // dC
        red[tid][NT + n] = gd * u;        // dB
        dA_acc[n] = fmaf(gd, ap, dA_acc[n]);
        ddt_a[n & 1] = fmaf(gn * A2[n], ap, ddt_a[n & 1]);
        ddt_b[n & 1] = fmaf(gn, bb, ddt_b[n & 1]);
        dsum[n & 1] = fmaf(gd, bb, dsum[n & 1]);
        ysum[n & 1] = fmaf(cc, ht, ysum[n & 1]);
        g[n] = a * gn;
      }
      const float ddt = (ddt_a[0] + ddt_a[1]) * kLn2 + (ddt_b[0] + ddt_b[1]) * u;
      const float dx = p.softplus ? ddt * sigmoid_f(xs[st]) : ddt;
      dbias_acc += dx;
      dD_acc = fmaf(dyp, u, dD_acc);
      if (valid) {
        const int64_t xi = row * L + t;
        static_cast<T*>(p.ddelta)[xi] = Elem<T>::from_f32(dx);
        static_cast<T*>(p.du)[xi] = Elem<T>::from_f32(fmaf(dyp, Dd, dsum[0] + dsum[1]));
        if (HAS_Z) {
          const float yp = fmaf(Dd, u, ysum[0] + ysum[1]);
          const float dz = dys[st] * yp * sig * fmaf(zs[st], 1.f - sig, 1.f);
          static_cast<T*>(p.dz)[xi] = Elem<T>::from_f32(dz);
        }
      }
      // dB/dC of step t over the warp's 32 rows, in row order: lane k sums
      // column k (no CTA barrier); the two warps' sums meet once per block
      __syncwarp();
      {
        const int lane = tid & 31, w = tid >> 5;
        float acc = 0.f;
#pragma unroll 8
        for (int r = 0; r < 32; ++r) acc += red[w * 32 + r][lane];
        wpart[w][st][lane] = acc;
      }
      __syncwarp();
    }
    // the block's dB/dC: the two warps' sums added, step by step
    __syncthreads();
    for (int idx = tid; idx < S * 2 * NT; idx += kBwdThreads) {
      const int st = idx / (2 * NT), k = idx - st * (2 * NT);
      if (st < cnt) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kBwdRows / 32; ++w) v += wpart[w][st][k];
        const int m = k < NT ? 1 : 0, nn = k & (NT - 1);
        p.part_bc[((cta * 2 + m) * NT + nn) * L + t0 + st] = v;
      }
    }
  }
  if (valid) {
#pragma unroll
    for (int n = 0; n < NT; ++n) p.part_a[(b * p.dim + d) * NT + n] = dA_acc[n];
    p.part_dd[(b * p.dim + d) * 2 + 0] = dD_acc;
    p.part_dd[(b * p.dim + d) * 2 + 1] = dbias_acc;
  }
}

// dB, dC [b,N,L]: the per-CTA partials of each batch row added in CTA order.
__global__ void ss_bwd_reduce_bc(const BwdParams p) {
  const int64_t L = p.seqlen, N = p.dstate;
  const int64_t total = p.batch * N * L;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i % L, bn = i / L, nn = bn % N, b = bn / N;
    float sb = 0.f, sc = 0.f;
    for (int64_t k = 0; k < p.dtiles; ++k) {
      const int64_t cta = b * p.dtiles + k;
      sb += p.part_bc[((cta * 2 + 0) * kBwdLanes + nn) * L + t];
      sc += p.part_bc[((cta * 2 + 1) * kBwdLanes + nn) * L + t];
    }
    p.dB[i] = sb;
    p.dC[i] = sc;
  }
}

// dA [d,N], dD [d], dbias [d]: per-row partials added over the batch in order.
__global__ void ss_bwd_reduce_rows(const BwdParams p) {
  const int64_t N = p.dstate;
  const int64_t total = p.dim * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t d = i / N, nn = i - d * N;
    float s = 0.f, sd = 0.f, sbias = 0.f;
    for (int64_t b = 0; b < p.batch; ++b) {
      s += p.part_a[(b * p.dim + d) * kBwdLanes + nn];
      if (nn == 0) {
        sd += p.part_dd[(b * p.dim + d) * 2 + 0];
        sbias += p.part_dd[(b * p.dim + d) * 2 + 1];
      }
    }
    p.dA[i] = s;
    if (nn == 0) {
      if (p.dD) p.dD[d] = sd;
      if (p.dbias) p.dbias[d] = sbias;
    }
  }
}

}  // namespace ss
