// Selective-scan forward kernels for sm_103a.
//
// Method ("Реализовать selective scan (Mamba)", Этап 1; "Mamba CUDA 实现解析"
// eq (4)-(7)): per (batch b, channel d, state n) the diagonal recurrence
//   h = exp(dt*A[d,n]) * h + dt*B[b,n,t]*u[b,d,t],  dt = softplus(delta + bias)
// and the read-out y = sum_n C[b,n,t]*h + D[d]*u, gated by silu(z).
//
// Decomposition (GB300-first, not the pages' kernels):
//  * A thread owns R channel rows of one batch and NT states of each row, all
//    in registers, and walks time sequentially.  Work per state update is one
//    MUFU ex2 plus four FP32 lane-ops, issued as packed f32x2 instructions
//    over state pairs (n, n+1), so the FP32 pipe and not instruction issue is
//    the limit.
//  * The B/C rows of a batch are shared by every channel: a CTA stages them
//    for a tile of TS steps into shared memory, transposed to [t][n] and
//    widened to fp32, so one 128-bit broadcast load yields two state pairs
//    and serves all R rows of a thread.
//  * u, delta and z are streamed with 128-bit loads straight into registers
//    (each thread reads its own rows; the vector path needs 16-byte aligned
//    rows), and y is written the same way.
//  * Long sequences are split into chunks that run in parallel.  Chunks are
//    joined with the associative operator of "Mamba CUDA 实现解析" eq (10),
//    (P1, v1) (+) (P2, e2) = (P2*P1, P2*v1 + e2):
//      ss_chunk_aggregate  computes each chunk's (P, e) = (prod of a, state
//                          reached from zero), with P = 2^(A*log2e*sum dt);
//      ss_chunk_carry      folds them into the state entering every chunk
//                          (the exclusive prefix of eq (11)-(12));
//      ss_fwd_main         runs every chunk from its carry and writes y.
//  * dstate above NT is handled in state groups of NT: each group's read-out
//    is accumulated in an fp32 scratch row and the last group applies the
//    skip and the gate.
#pragma once

#include "ss_device.cuh"

namespace ss {

constexpr int kTileSteps = 64;  // steps of B/C staged per shared-memory tile

struct FwdParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* bias;
  const float* h0;    // [b,d,N] state before step 0 (null: zero)
  void* y;
  float* last_state;
  float* y_partial;   // fp32 [rows, L]: read-out of earlier state groups (dstate > NT)
  float2* agg;        // [nchunks-1][rows][ns]: (prod a, state from zero) per chunk
  float* carry;       // [nchunks][rows][ns]: state entering each chunk
  int64_t batch, dim, dstate, seqlen;
  int64_t chunk_len;  // steps per chunk, a multiple of kTileSteps
  int nchunks;
  int ns;             // padded state count (groups * NT)
  int group;          // state group of this launch (ss_fwd_main)
  int softplus;
  int accum_in;       // ss_fwd_main: add y_partial of earlier groups
  int final_group;    // ss_fwd_main: last group: skip, gate and write y
  // scheduled vector path (ss_fwd_sched)
  unsigned* ticket;   // next unit to hand out (zeroed before the launch)
  unsigned* flags;    // [nchunks][tiles] publication state of each unit (zeroed)
  float2* unit_agg;   // [nchunks][tiles][rows_per_cta][NT] (prod a, state from zero)
  float* unit_incl;   // [nchunks][tiles][rows_per_cta][NT] state at the unit's end
  int64_t tiles;      // row tiles: batch * dim_tiles
  int chained;        // 1: units wait for their predecessor; 0: decoupled look-back
  int y_pairs;        // 1: y rows 32-byte aligned (seqlen a multiple of two vectors, y aligned)
};

// Row bookkeeping shared by the kernels: thread tid of the CTA owns channels
// d = tile*TPB*R + r*TPB + tid (r < R) of batch b.  Rows past dim are clamped
// to a valid row for loads and never stored.
template <int R, int TPB>
struct RowSet {
  int64_t row[R];
  int64_t d[R];
  bool valid[R];
  int64_t b;

  __device__ __forceinline__ RowSet(int64_t tile_linear, int64_t dim) {
    const int64_t dtiles = (dim + TPB * R - 1) / (TPB * R);
    b = tile_linear / dtiles;
    const int64_t dt = tile_linear - b * dtiles;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t dd = dt * (TPB * R) + r * TPB + threadIdx.x;
      valid[r] = dd < dim;
      d[r] = valid[r] ? dd : dim - 1;
      row[r] = b * dim + d[r];
    }
  }
};

// Stage one tile of M (= B or C) for steps [t0, t0 + tlen) and states
// [n0, n0 + NT) into s[TS][NT] as fp32; padded states and steps are zero.
template <typename T, int NT, int TPB, bool VEC>
__device__ __forceinline__ void stage_tile(float (*s)[NT], const T* __restrict__ M,
                                          int64_t b, int64_t N, int64_t L, int n0,
                                          int64_t t0, int tlen) {
  constexpr int V = VEC ? Elem<T>::kVec : 1;
  constexpr int VPR = kTileSteps / V;  // vectors per state row
  for (int i = threadIdx.x; i < NT * VPR; i += TPB) {
    const int n = i / VPR;
    const int j = (i - n * VPR) * V;
    const int64_t ng = n0 + n;
    float vals[V];
    if (ng < N && j < tlen) {
      const T* src = M + (b * N + ng) * L + t0 + j;
      if constexpr (VEC) {
        const Vec16<T> v = ldg_vec(src);
#pragma unroll
        for (int e = 0; e < V; ++e) vals[e] = Elem<T>::to_f32(v.e[e]);
      } else {
        vals[0] = Elem<T>::to_f32(src[0]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) vals[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < V; ++e) s[j + e][n] = vals[e];
  }
}

// dt for one step: softplus(delta + bias) or delta + bias.
__device__ __forceinline__ float step_size(float delta, float bias, int use_softplus) {
  const float x = delta + bias;
  return use_softplus ? softplus(x) : x;
}

// ---------------------------------------------------------------------------
// Main kernel: every chunk from its carry; writes y (or the fp32 partial
// read-out) and, for the last chunk, last_state.
// grid = (batch * dim_tiles, nchunks), block = TPB.
template <typename T, int NT, int R, int TPB, bool VEC>
__global__ void __launch_bounds__(TPB) ss_fwd_main(const FwdParams p) {
  constexpr int V = VEC ? Elem<T>::kVec : 1;
  constexpr int NP = NT / 2;
  static_assert(NT % 4 == 0, "NT must be a multiple of 4");
  __shared__ __align__(16) float sB[kTileSteps][NT];
  __shared__ __align__(16) float sC[kTileSteps][NT];

  const int64_t L = p.seqlen, N = p.dstate;
  const RowSet<R, TPB> rs(blockIdx.x, p.dim);
  const int chunk = blockIdx.y;
  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = min(L, t_begin + p.chunk_len);
  const int n0 = p.group * NT;
  const int64_t rows = p.batch * p.dim;

  const T* __restrict__ u = static_cast<const T*>(p.u);
  const T* __restrict__ dl = static_cast<const T*>(p.delta);
  const T* __restrict__ zg = static_cast<const T*>(p.z);
  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  T* __restrict__ y = static_cast<T*>(p.y);

  f2 A2[R][NP], h[R][NP];
  float bias[R], Dd[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    bias[r] = p.bias ? p.bias[rs.d[r]] : 0.f;
    Dd[r] = p.D ? p.D[rs.d[r]] : 0.f;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      float a[2], h0[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t n = n0 + 2 * q + k;
        a[k] = n < N ? p.A[rs.d[r] * N + n] * kLog2e : 0.f;
        // a split row takes every chunk's carry from ss_chunk_carry (chunk 0's
        // is h0), so h0 is read before this launch and may alias last_state;
        // an unsplit row reads h0 here, in the thread that writes last_state
        h0[k] = n >= N ? 0.f
                : p.nchunks > 1 ? p.carry[((int64_t)chunk * rows + rs.row[r]) * p.ns + n]
                : (p.h0 ? p.h0[rs.row[r] * N + n] : 0.f);
      }
      A2[r][q] = pack(a[0], a[1]);
      h[r][q] = pack(h0[0], h0[1]);
    }
  }

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kTileSteps) {
    const int tlen = (int)min((int64_t)kTileSteps, t_end - t0);
    __syncthreads();
    stage_tile<T, NT, TPB, VEC>(sB, Bg, rs.b, N, L, n0, t0, tlen);
    stage_tile<T, NT, TPB, VEC>(sC, Cg, rs.b, N, L, n0, t0, tlen);
    __syncthreads();

    for (int j0 = 0; j0 < tlen; j0 += V) {
      float uu[R][V], dd[R][V];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t off = rs.row[r] * L + t0 + j0;
        if constexpr (VEC) {
          const Vec16<T> vu = ldg_vec(u + off), vd = ldg_vec(dl + off);
#pragma unroll
          for (int e = 0; e < V; ++e) {
            uu[r][e] = Elem<T>::to_f32(vu.e[e]);
            dd[r][e] = Elem<T>::to_f32(vd.e[e]);
          }
        } else {
          uu[r][0] = Elem<T>::to_f32(u[off]);
          dd[r][0] = Elem<T>::to_f32(dl[off]);
        }
      }

      float yv[R][V];
#pragma unroll
      for (int s = 0; s < V; ++s) {
        const int j = j0 + s;
        f2 dt2[R], du2[R], yacc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float dt = step_size(dd[r][s], bias[r], p.softplus);
          const float du = dt * uu[r][s];
          dt2[r] = pack(dt, dt);
          du2[r] = pack(du, du);
          yacc[r] = pack(0.f, 0.f);
        }
#pragma unroll
        for (int q4 = 0; q4 < NT / 4; ++q4) {
          const ulonglong2 bq = *reinterpret_cast<const ulonglong2*>(&sB[j][4 * q4]);
          const ulonglong2 cq = *reinterpret_cast<const ulonglong2*>(&sC[j][4 * q4]);
          const f2 bp[2] = {{bq.x}, {bq.y}};
          const f2 cp[2] = {{cq.x}, {cq.y}};
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int q = 2 * q4 + k;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const f2 a = ex2x2(mul2(dt2[r], A2[r][q]));
              const f2 c = mul2(du2[r], bp[k]);
              h[r][q] = fma2(a, h[r][q], c);
              yacc[r] = fma2(cp[k], h[r][q], yacc[r]);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float lo, hi;
          unpack(yacc[r], lo, hi);
          yv[r][s] = lo + hi;
        }
      }

      // epilogue for V steps: earlier groups' read-out, skip, gate, store
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t off = rs.row[r] * L + t0 + j0;
        if (p.accum_in) {
#pragma unroll
          for (int e = 0; e < V; ++e) yv[r][e] += p.y_partial[off + e];
        }
        if (!p.final_group) {
          if (rs.valid[r]) {
#pragma unroll
            for (int e = 0; e < V; ++e) p.y_partial[off + e] = yv[r][e];
          }
          continue;
        }
        float zz[V];
        if (zg) {
          if constexpr (VEC) {
            const Vec16<T> vz = ldg_vec(zg + off);
#pragma unroll
            for (int e = 0; e < V; ++e) zz[e] = Elem<T>::to_f32(vz.e[e]);
          } else {
            zz[0] = Elem<T>::to_f32(zg[off]);
          }
        }
        Vec16<T> out;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          float v = fmaf(Dd[r], uu[r][e], yv[r][e]);
          if (zg) v *= silu(zz[e]);
          out.e[e] = Elem<T>::from_f32(v);
        }
        if (rs.valid[r]) {
          if constexpr (VEC) {
            stg_vec(y + off, out);
          } else {
            y[off] = out.e[0];
          }
        }
      }
    }
  }

  if (chunk == p.nchunks - 1 && p.last_state) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (!rs.valid[r]) continue;
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        float hv[2];
        unpack(h[r][q], hv[0], hv[1]);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int64_t n = n0 + 2 * q + k;
          if (n < N) p.last_state[rs.row[r] * N + n] = hv[k];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Chunk aggregate: for chunks 0..nchunks-2, the state each chunk reaches from
// a zero state, e, and its total decay P = 2^(A*log2e * sum dt) = prod a.
// grid = (batch * dim_tiles, nchunks - 1, groups), block = TPB.
template <typename T, int NT, int R, int TPB, bool VEC>
__global__ void __launch_bounds__(TPB) ss_chunk_aggregate(const FwdParams p) {
  constexpr int V = VEC ? Elem<T>::kVec : 1;
  constexpr int NP = NT / 2;
  __shared__ __align__(16) float sB[kTileSteps][NT];

  const int64_t L = p.seqlen, N = p.dstate;
  const RowSet<R, TPB> rs(blockIdx.x, p.dim);
  const int chunk = blockIdx.y;
  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = min(L, t_begin + p.chunk_len);
  const int n0 = blockIdx.z * NT;
  const int64_t rows = p.batch * p.dim;

  const T* __restrict__ u = static_cast<const T*>(p.u);
  const T* __restrict__ dl = static_cast<const T*>(p.delta);
  const T* __restrict__ Bg = static_cast<const T*>(p.B);

  f2 A2[R][NP], h[R][NP];
  float bias[R], dt_sum[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    bias[r] = p.bias ? p.bias[rs.d[r]] : 0.f;
    dt_sum[r] = 0.f;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      float a[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t n = n0 + 2 * q + k;
        a[k] = n < N ? p.A[rs.d[r] * N + n] * kLog2e : 0.f;
      }
      A2[r][q] = pack(a[0], a[1]);
      h[r][q] = pack(0.f, 0.f);
    }
  }

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kTileSteps) {
    const int tlen = (int)min((int64_t)kTileSteps, t_end - t0);
    __syncthreads();
    stage_tile<T, NT, TPB, VEC>(sB, Bg, rs.b, N, L, n0, t0, tlen);
    __syncthreads();
    for (int j0 = 0; j0 < tlen; j0 += V) {
      float uu[R][V], dd[R][V];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t off = rs.row[r] * L + t0 + j0;
        if constexpr (VEC) {
          const Vec16<T> vu = ldg_vec(u + off), vd = ldg_vec(dl + off);
#pragma unroll
          for (int e = 0; e < V; ++e) {
            uu[r][e] = Elem<T>::to_f32(vu.e[e]);
            dd[r][e] = Elem<T>::to_f32(vd.e[e]);
          }
        } else {
          uu[r][0] = Elem<T>::to_f32(u[off]);
          dd[r][0] = Elem<T>::to_f32(dl[off]);
        }
      }
      float vec_sum[R];
#pragma unroll
      for (int r = 0; r < R; ++r) vec_sum[r] = 0.f;
#pragma unroll
      for (int s = 0; s < V; ++s) {
        const int j = j0 + s;
        f2 dt2[R], du2[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float dt = step_size(dd[r][s], bias[r], p.softplus);
          vec_sum[r] += dt;
          dt2[r] = pack(dt, dt);
          du2[r] = pack(dt * uu[r][s], dt * uu[r][s]);
        }
#pragma unroll
        for (int q4 = 0; q4 < NT / 4; ++q4) {
          const ulonglong2 bq = *reinterpret_cast<const ulonglong2*>(&sB[j][4 * q4]);
          const f2 bp[2] = {{bq.x}, {bq.y}};
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int q = 2 * q4 + k;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const f2 a = ex2x2(mul2(dt2[r], A2[r][q]));
              h[r][q] = fma2(a, h[r][q], mul2(du2[r], bp[k]));
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) dt_sum[r] += vec_sum[r];
    }
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!rs.valid[r]) continue;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const f2 P = ex2x2(mul2(pack(dt_sum[r], dt_sum[r]), A2[r][q]));
      float Pv[2], hv[2];
      unpack(P, Pv[0], Pv[1]);
      unpack(h[r][q], hv[0], hv[1]);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t n = n0 + 2 * q + k;
        p.agg[((int64_t)chunk * rows + rs.row[r]) * p.ns + n] = make_float2(Pv[k], hv[k]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Carry across chunks: for every (row, state) fold the chunk aggregates in
// order, carry[k] = (P_{k-1}, e_{k-1}) applied to carry[k-1], carry[0] = h0
// (zero without an initial state).
// One thread per (row, state); grid covers rows * ns.
__global__ void ss_chunk_carry(const FwdParams p) {
  const int64_t rows = p.batch * p.dim;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * p.ns) return;
  const int64_t row = i / p.ns, n = i - row * p.ns;
  float h = (p.h0 && n < p.dstate) ? p.h0[row * p.dstate + n] : 0.f;
  for (int k = 0; k < p.nchunks; ++k) {
    p.carry[(int64_t)k * rows * p.ns + i] = h;
    if (k + 1 < p.nchunks) {
      const float2 pe = p.agg[(int64_t)k * rows * p.ns + i];
      h = fmaf(pe.x, h, pe.y);
    }
  }
}

}  // namespace ss
