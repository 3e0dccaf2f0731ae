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
        h0[k] = (chunk > 0 && n < N)
                    ? p.carry[((int64_t)chunk * rows + rs.row[r]) * p.ns + n]
                    : 0.f;
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
// Vector path (16-byte aligned rows, seqlen a multiple of the vector width).
//
// Thread layout: groups of TGS adjacent lanes share two channel rows; lane q
// of a group holds states [q*G, (q+1)*G) (G = NT / TGS) of both rows, so the
// B/C values it loads serve two rows.  Row work (streaming u/delta/z, dt and
// du, the skip/gate epilogue) is split between the lanes of a group: with
// TGS = 1 the lane does both rows, with TGS = 2 lane q does row q and the
// partners swap dt, du and the partial read-outs with three shuffles a step.
// Splitting states doubles the resident warps, which hides the MUFU/FMA
// dependency latency of the recurrence.
//
// Latency of global memory is taken off the critical path by asynchronous
// copies:
//  * u, delta (and z) of a lane's own rows stream through a STAGES-deep ring
//    of per-lane shared-memory slots filled with cp.async; a lane only reads
//    the slots it filled, so the ring needs no barrier.
//  * B (and C) tiles of kTileSteps steps are copied raw with cp.async one
//    tile ahead, then widened and transposed to [t][n] fp32 at the tile
//    boundary (two barriers per tile).
// AGG = false: the main pass (y, last_state).  AGG = true: the chunk
// aggregate pass (prod a and the state reached from zero; no C, z or y).
// grid = (batch * dim_tiles, nchunks [- 1 for AGG], groups for AGG), block = TPB.
template <int TGS, int TPB>
struct PairRows {
  static constexpr int kRowsPerCta = 2 * TPB / TGS;
  static constexpr int kOwn = 2 / TGS;  // rows whose row work this lane does
  int64_t row[2];   // slot 0: own row; slot 1: the other row of the group
  int64_t d[2];
  bool valid[2];
  int64_t b;
  int q;            // lane in group

  __device__ __forceinline__ PairRows(int64_t tile_linear, int64_t dim) {
    const int64_t dtiles = (dim + kRowsPerCta - 1) / kRowsPerCta;
    b = tile_linear / dtiles;
    const int64_t base = (tile_linear - b * dtiles) * kRowsPerCta;
    const int g = threadIdx.x / TGS;
    q = threadIdx.x % TGS;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int which = TGS == 1 ? s : (s == 0 ? q : 1 - q);
      const int64_t dd = base + (int64_t)which * (TPB / TGS) + g;
      valid[s] = dd < dim;
      d[s] = valid[s] ? dd : dim - 1;
      row[s] = b * dim + d[s];
    }
  }
};

template <typename T, int NT, int TGS, int TPB, int STAGES, bool AGG>
__global__ void __launch_bounds__(TPB) ss_fwd_pipe(const FwdParams p) {
  constexpr int V = Elem<T>::kVec;
  constexpr int G = NT / TGS;       // states per lane
  constexpr int GP = G / 2;         // state pairs per lane
  constexpr int OWN = 2 / TGS;      // own rows (row work) per lane
  constexpr int NX = AGG ? 2 : 3;   // streamed row tensors: u, delta (, z)
  constexpr int NM = AGG ? 1 : 2;   // staged state tensors: B (, C)
  constexpr int VPT = kTileSteps / V;
  constexpr int CPR = kTileSteps * (int)sizeof(T) / 16;  // 16-byte chunks per state row
  constexpr int RAW = kTileSteps + 16 / (int)sizeof(T);  // padded raw row (bank spread)
  static_assert(TGS == 1 || TGS == 2, "two lanes per group at most");
  static_assert(G % 4 == 0, "a lane holds a multiple of four states");
  static_assert(STAGES >= 2 && STAGES <= VPT, "pipeline depth must fit in a tile");
  __shared__ __align__(16) uint4 sX[STAGES][NX][OWN][TPB];
  __shared__ __align__(16) T sRaw[NM][NT][RAW];
  __shared__ __align__(16) float sM[NM][kTileSteps][NT];

  const int tid = threadIdx.x;
  const int64_t L = p.seqlen, N = p.dstate;
  const PairRows<TGS, TPB> rs(blockIdx.x, p.dim);
  const int chunk = blockIdx.y;
  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = min(L, t_begin + p.chunk_len);
  const int ng0 = (AGG ? (int)blockIdx.z : p.group) * NT;  // first state of the group
  const int nl0 = rs.q * G;                                 // first state of this lane
  const int64_t rows = p.batch * p.dim;
  const int64_t nvec = (t_end - t_begin) / V;

  const T* __restrict__ ug = static_cast<const T*>(p.u);
  const T* __restrict__ dg = static_cast<const T*>(p.delta);
  const T* __restrict__ zg = AGG ? nullptr : static_cast<const T*>(p.z);
  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  T* __restrict__ y = static_cast<T*>(p.y);

  f2 A2[2][GP], h[2][GP];
  float bias[OWN], Dd[OWN], dt_sum[OWN];
#pragma unroll
  for (int o = 0; o < OWN; ++o) {
    bias[o] = p.bias ? p.bias[rs.d[o]] : 0.f;
    Dd[o] = (!AGG && p.D) ? p.D[rs.d[o]] : 0.f;
    dt_sum[o] = 0.f;
  }
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int k = 0; k < GP; ++k) {
      float a[2], h0[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t n = ng0 + nl0 + 2 * k + e;
        a[e] = n < N ? p.A[rs.d[s] * N + n] * kLog2e : 0.f;
        h0[e] = (!AGG && chunk > 0 && n < N)
                    ? p.carry[((int64_t)chunk * rows + rs.row[s]) * p.ns + n]
                    : 0.f;
      }
      A2[s][k] = pack(a[0], a[1]);
      h[s][k] = pack(h0[0], h0[1]);
    }
  }

  // copies of the own-row vectors of vector index j (one commit group per call)
  auto issue_vec = [&](int64_t j) {
    if (j < nvec) {
      const int slot = (int)(j % STAGES);
      const int64_t t = t_begin + j * V;
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        const int64_t off = rs.row[o] * L + t;
        cp_async16(&sX[slot][0][o][tid], ug + off);
        cp_async16(&sX[slot][1][o][tid], dg + off);
        if (!AGG && zg) cp_async16(&sX[slot][NX - 1][o][tid], zg + off);
      }
    }
    cp_async_commit();
  };
  // raw copies of the B (and C) tile starting at t0; they join the next commit group
  auto issue_tile = [&](int64_t t0) {
    if (t0 >= t_end) return;
    const int tlen = (int)min((int64_t)kTileSteps, t_end - t0);
    for (int i = tid; i < NM * NT * CPR; i += TPB) {
      const int m = i / (NT * CPR);
      const int rem = i - m * NT * CPR;
      const int n = rem / CPR;
      const int j = (rem - n * CPR) * (16 / (int)sizeof(T));
      const int64_t ng = ng0 + n;
      if (ng < N && j < tlen)
        cp_async16(&sRaw[m][n][j], (m == 0 ? Bg : Cg) + (rs.b * N + ng) * L + t0 + j);
    }
  };

  issue_tile(t_begin);
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) issue_vec(s);

  for (int64_t j = 0; j < nvec; ++j) {
    issue_vec(j + STAGES - 1);
    cp_async_wait<STAGES - 1>();  // this lane's copies of vector j (and older) landed
    const int jt = (int)(j % VPT) * V;
    if (jt == 0) {
      // tile boundary: widen + transpose the raw tile, then prefetch the next one
      const int64_t t0 = t_begin + j * V;
      const int tlen = (int)min((int64_t)kTileSteps, t_end - t0);
      __syncthreads();  // every lane's raw copies landed; the previous tile is consumed
      constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte chunk
      for (int i = tid; i < NM * NT * CPR; i += TPB) {
        const int n = i % NT;  // state fastest: conflict-free transposed stores
        const int c = (i / NT) % CPR;
        const int m = i / (NT * CPR);
        const Vec16<T> v = *reinterpret_cast<const Vec16<T>*>(&sRaw[m][n][c * EPC]);
        const bool nok = ng0 + n < N;
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
          const int t = c * EPC + e;
          sM[m][t][n] = (nok && t < tlen) ? Elem<T>::to_f32(v.e[e]) : 0.f;
        }
      }
      __syncthreads();
      issue_tile(t0 + kTileSteps);
    }

    const int slot = (int)(j % STAGES);
    Vec16<T> xu[OWN], xd[OWN];
#pragma unroll
    for (int o = 0; o < OWN; ++o) {
      *reinterpret_cast<uint4*>(&xu[o]) = sX[slot][0][o][tid];
      *reinterpret_cast<uint4*>(&xd[o]) = sX[slot][1][o][tid];
    }

    float yv[OWN][V];
#pragma unroll
    for (int s = 0; s < V; ++s) {
      const int t = jt + s;
      f2 dt2[2], du2[2], yacc[2];
      {
        float dt[OWN], du[OWN];
#pragma unroll
        for (int o = 0; o < OWN; ++o) {
          dt[o] = step_size(Elem<T>::to_f32(xd[o].e[s]), bias[o], p.softplus);
          du[o] = dt[o] * Elem<T>::to_f32(xu[o].e[s]);
          if (AGG) dt_sum[o] += dt[o];
        }
        if constexpr (TGS == 1) {
          dt2[0] = pack(dt[0], dt[0]);
          du2[0] = pack(du[0], du[0]);
          dt2[1] = pack(dt[1], dt[1]);
          du2[1] = pack(du[1], du[1]);
        } else {
          const float dto = __shfl_xor_sync(0xffffffffu, dt[0], 1);
          const float duo = __shfl_xor_sync(0xffffffffu, du[0], 1);
          dt2[0] = pack(dt[0], dt[0]);
          du2[0] = pack(du[0], du[0]);
          dt2[1] = pack(dto, dto);
          du2[1] = pack(duo, duo);
        }
        yacc[0] = pack(0.f, 0.f);
        yacc[1] = pack(0.f, 0.f);
      }
#pragma unroll
      for (int k4 = 0; k4 < G / 4; ++k4) {
        const ulonglong2 bq = *reinterpret_cast<const ulonglong2*>(&sM[0][t][nl0 + 4 * k4]);
        const f2 bp[2] = {{bq.x}, {bq.y}};
        f2 cp[2];
        if (!AGG) {
          const ulonglong2 cq =
              *reinterpret_cast<const ulonglong2*>(&sM[NM - 1][t][nl0 + 4 * k4]);
          cp[0].v = cq.x;
          cp[1].v = cq.y;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 2 * k4 + e;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const f2 a = ex2x2(mul2(dt2[r], A2[r][k]));
            h[r][k] = fma2(a, h[r][k], mul2(du2[r], bp[e]));
            if (!AGG) yacc[r] = fma2(cp[e], h[r][k], yacc[r]);
          }
        }
      }
      if (!AGG) {
        float part[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float lo, hi;
          unpack(yacc[r], lo, hi);
          part[r] = lo + hi;
        }
        if constexpr (TGS == 1) {
          yv[0][s] = part[0];
          yv[1][s] = part[1];
        } else {
          yv[0][s] = part[0] + __shfl_xor_sync(0xffffffffu, part[1], 1);
        }
      }
    }

    if constexpr (!AGG) {
      // epilogue for V steps of the own rows: earlier groups' read-out, skip, gate, store
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        const int64_t off = rs.row[o] * L + t_begin + j * V;
        if (p.accum_in) {
#pragma unroll
          for (int e = 0; e < V; ++e) yv[o][e] += p.y_partial[off + e];
        }
        if (!p.final_group) {
          if (rs.valid[o]) {
#pragma unroll
            for (int e = 0; e < V; ++e) p.y_partial[off + e] = yv[o][e];
          }
          continue;
        }
        float zz[V];
        if (zg) {
          const uint4 rz = sX[slot][NX - 1][o][tid];
          const T* ez = reinterpret_cast<const T*>(&rz);
#pragma unroll
          for (int e = 0; e < V; ++e) zz[e] = Elem<T>::to_f32(ez[e]);
        }
        Vec16<T> out;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          float v = fmaf(Dd[o], Elem<T>::to_f32(xu[o].e[e]), yv[o][e]);
          if (zg) v *= silu(zz[e]);
          out.e[e] = Elem<T>::from_f32(v);
        }
        if (rs.valid[o]) stg_vec(y + off, out);
      }
    }
  }
  cp_async_wait<0>();

  if constexpr (AGG) {
    float sum[2];
    sum[0] = dt_sum[0];
    if constexpr (TGS == 1) {
      sum[1] = dt_sum[1];
    } else {
      sum[1] = __shfl_xor_sync(0xffffffffu, dt_sum[0], 1);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!rs.valid[r]) continue;
#pragma unroll
      for (int k = 0; k < GP; ++k) {
        const f2 P = ex2x2(mul2(pack(sum[r], sum[r]), A2[r][k]));
        float Pv[2], hv[2];
        unpack(P, Pv[0], Pv[1]);
        unpack(h[r][k], hv[0], hv[1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t n = ng0 + nl0 + 2 * k + e;
          p.agg[((int64_t)chunk * rows + rs.row[r]) * p.ns + n] = make_float2(Pv[e], hv[e]);
        }
      }
    }
  } else if (chunk == p.nchunks - 1 && p.last_state) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!rs.valid[r]) continue;
#pragma unroll
      for (int k = 0; k < GP; ++k) {
        float hv[2];
        unpack(h[r][k], hv[0], hv[1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t n = ng0 + nl0 + 2 * k + e;
          if (n < N) p.last_state[rs.row[r] * N + n] = hv[e];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Carry across chunks: for every (row, state) fold the chunk aggregates in
// order, carry[k] = (P_{k-1}, e_{k-1}) applied to carry[k-1], carry[0] = 0.
// One thread per (row, state); grid covers rows * ns.
__global__ void ss_chunk_carry(const FwdParams p) {
  const int64_t rows = p.batch * p.dim;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * p.ns) return;
  float h = 0.f;
  for (int k = 0; k < p.nchunks; ++k) {
    p.carry[(int64_t)k * rows * p.ns + i] = h;
    if (k + 1 < p.nchunks) {
      const float2 pe = p.agg[(int64_t)k * rows * p.ns + i];
      h = fmaf(pe.x, h, pe.y);
    }
  }
}

}  // namespace ss
