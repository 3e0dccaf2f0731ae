// Vector path of the selective-scan forward: one persistent kernel per call
// that hands out (row tile, sequence chunk) units in order and joins the
// chunks of a row tile with the associative operator of "Mamba CUDA 实现解析"
// eq (10): (P1, v1) (+) (P2, e2) = (P2*P1, P2*v1 + e2), where a chunk's
// aggregate is P = prod of its decays a = exp(dt*A) and e = the state it
// reaches from zero.  The state entering chunk k is the prefix
// s_0 (+) E_1 (+) ... (+) E_{k-1} of eq (11)-(12).
//
// Scheduling.  CTAs take tickets from a global counter; ticket t is unit
// (chunk k = t / tiles, tile i = t % tiles), so every unit's predecessor
// (k-1, i) was handed out earlier to a CTA that is running or done, and
// every wait below ends.  The mode of a launch is fixed by the host:
//  * chained (at least as many row tiles as CTAs): a unit waits for the
//    state its predecessor reached, runs its single pass from it and
//    publishes its own end state; the predecessor was handed out a full
//    round of tickets earlier, so the wait is normally over at once and no
//    work is repeated.
//  * decoupled (fewer row tiles than CTAs): every unit after the first of
//    its tile computes its own aggregate (a pass without C, z or y) and
//    publishes it, then looks back to the nearest predecessor whose end
//    state is published (one warp polls 32 predecessors at a time) and
//    folds the aggregates in between forward, in chunk order; that gives
//    its carry, it publishes its own end state P*carry + e at once and runs
//    the main pass from the carry.
// Both modes evaluate every carry by the same sequence of operations whatever
// the timing, so results are bitwise reproducible from run to run.
// Every wait polls with back-off and gives up after kSpinLimit polls: it then
// sets the device error word (ss_selective_scan_check reports SS_ERR_TIMEOUT),
// uses a zero carry and carries on, so no call can hang the device.
//
// Thread layout inside a unit: groups of TGS adjacent lanes share two channel
// rows; lane q of a group holds states [q*G, (q+1)*G) (G = NT / TGS) of both
// rows, so every B/C value it loads serves two rows.  Row work (streaming
// u/delta/z, dt and du, the skip/gate epilogue) is split between the lanes of
// a group: with TGS = 1 the lane does both rows, with TGS = 2 lane q does row
// q and the partners swap dt, du and the partial read-outs by shuffle.
//
// Memory latency is taken off the critical path by asynchronous copies: u,
// delta (and z) of a lane's own rows stream through a STAGES-deep ring of
// per-lane shared-memory slots filled with cp.async (a lane only reads the
// slots it filled, so the ring needs no barrier); B (and C) tiles of
// kTileSteps steps are copied raw one tile ahead and widened/transposed to
// [t][n] fp32 at the tile boundary (two barriers per tile).
#pragma once

#include <type_traits>

#include "ss_fwd.cuh"

namespace ss {

// Error word of the device-side waits (one per device context).
__device__ unsigned int g_ss_device_error = 0;

constexpr unsigned kUnitAgg = 1u;             // unit aggregate published
constexpr unsigned kUnitIncl = 2u;            // state at the unit's end published
constexpr long long kSpinLimit = 1LL << 20;   // polls before a wait gives up (~0.3 s)
constexpr unsigned kErrTimeout = 1u;

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Thread 0 waits until *flag >= want (bounded); returns the flag value seen,
// or 0 after giving up (the device error word is then set).
__device__ __forceinline__ unsigned wait_flag(const unsigned* flag, unsigned want) {
  unsigned v = ld_acquire(flag);
  long long polls = 0;
  while (v < want) {
    if (++polls > kSpinLimit) {
      atomicOr(&g_ss_device_error, kErrTimeout);
      return 0u;
    }
    __nanosleep(polls < 64 ? 32 : 256);
    v = ld_acquire(flag);
  }
  return v;
}

// Decoupled look-back of unit (chunk k, tile) by one warp: lane i inspects
// chunk base - i, so one poll covers 32 predecessors.  The search ends when
// the nearest predecessor whose end state is published (flag kUnitIncl) and
// every chunk after it have at least their aggregates published; a window of
// aggregates only moves the search 32 chunks back.  Chunk 0 always publishes
// its end state, so the search ends.  Returns j0 + 1 for the chunk j0 found,
// or 0 after kSpinLimit polls (the device error word is then set).  Called by
// all 32 lanes of one warp.
__device__ __forceinline__ unsigned look_back(const unsigned* flags, int64_t M, int64_t tile,
                                              int k, int lane) {
  int base = k - 1;
  long long polls = 0;
  for (;;) {
    const int j = base - lane;
    const unsigned f = j >= 0 ? ld_acquire(&flags[(int64_t)j * M + tile]) : 0u;
    const unsigned incl = __ballot_sync(0xffffffffu, j >= 0 && f >= kUnitIncl);
    const unsigned ready = __ballot_sync(0xffffffffu, j < 0 || f >= kUnitAgg);
    if (incl != 0u) {
      const int fi = __ffs(incl) - 1;  // nearest published end state
      const unsigned need = fi == 31 ? 0xffffffffu : (2u << fi) - 1u;
      if ((ready & need) == need) return (unsigned)(base - fi) + 1u;
    } else if (ready == 0xffffffffu) {
      base -= 32;  // aggregates only: search further back
      continue;
    }
    if (++polls > kSpinLimit) {
      if (lane == 0) atomicOr(&g_ss_device_error, kErrTimeout);
      return 0u;
    }
    __nanosleep(polls < 64 ? 32 : 256);
  }
}

#ifdef SS_TEST_HOOKS
// Test hook of the host (test build only): start a launch's ticket counter at
// `first`, so units below it are never handed out and the waits of their
// successors run out (bounded; the device error word reports it).
__global__ void ss_set_ticket(unsigned* ticket, unsigned first) { *ticket = first; }
#endif

// Two lanes per row pair (8 or 16 states) stream u, delta and z through
// per-warp segments (below); four states per row pair through per-lane slots.
template <typename T, int TGS>
constexpr bool kSegStream = TGS == 2;
// vectors per segment: fp32 4 (64 bytes of each of 32 rows), bf16 2 (32
// bytes); segments in a warp's ring: 4.  (The bf16 tile of B/C holds 8
// vectors, and a tile's raw copies ride in a segment's copy group, which bounds
// (slots - 1) x vectors by the tile.)
template <typename T>
constexpr int kSegVecs = sizeof(T) == 4 ? 4 : 2;
constexpr int kSegSlots = 4;

// WARP_ROWS: a warp's rows are the contiguous rows [32 w, 32 w + 32) of the
// tile, lane l owning row 32 w + l (the segment stream copies a warp's rows as
// one block); otherwise lane pair g owns rows g and g + TPB / TGS.
template <int TGS, int TPB, bool WARP_ROWS = false>
struct PairRows {
  static constexpr int kRowsPerCta = 2 * TPB / TGS;
  static_assert(!WARP_ROWS || TGS == 2, "warp rows need two lanes per row pair");
  int64_t row[2];  // slot 0: own row; slot 1: the other row of the group
  int64_t d[2];
  int rc[2];       // row index inside the tile
  bool valid[2];
  int64_t b;
  int64_t d0;      // first channel of the tile
  int q;           // lane in group

  __device__ __forceinline__ PairRows(int64_t tile, int64_t dim) {
    const int64_t dtiles = (dim + kRowsPerCta - 1) / kRowsPerCta;
    b = tile / dtiles;
    const int64_t base = (tile - b * dtiles) * kRowsPerCta;
    d0 = base;
    const int g = threadIdx.x / TGS;
    q = threadIdx.x % TGS;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int which = TGS == 1 ? s : (s == 0 ? q : 1 - q);
      rc[s] = WARP_ROWS ? (int)(threadIdx.x & ~31u) + 2 * ((int)(threadIdx.x & 31u) / 2) + which
                        : which * (TPB / TGS) + g;
      const int64_t dd = base + rc[s];
      valid[s] = dd < dim;
      d[s] = valid[s] ? dd : dim - 1;
      row[s] = b * dim + d[s];
    }
  }
};

template <typename T, int NT, int TGS, int TPB, int STAGES, bool SEG = kSegStream<T, TGS>>
struct PipeSmem {
  static constexpr int kOwn = 2 / TGS;
  static constexpr int kRaw = kTileSteps + 16 / (int)sizeof(T);  // padded raw row
  uint4 x[STAGES][3][kOwn][TPB];      // u, delta, z ring of the own rows
  T raw[2][NT][kRaw];                 // raw B, C tile
  float m[2][kTileSteps][NT];         // widened, transposed B, C tile
};

// Segment stream: per warp, a ring of kSegSlots segments; a segment holds
// kSegVecs vectors of the warp's 32 rows for u, delta and z, each row 64 (fp32)
// or 32 (bf16) bytes whose 16-byte vectors are XOR-permuted by (row / 2) % 4 or
// (row / 4) % 2, so that both the copies (two or four rows per 8 lanes) and
// the reads (8 rows per 8 lanes, one vector each) touch every bank once.
template <typename T, int NT, int TGS, int TPB, int STAGES>
struct PipeSmem<T, NT, TGS, TPB, STAGES, true> {
  static constexpr int kRaw = kTileSteps + 16 / (int)sizeof(T);
  uint4 xs[TPB / 32][kSegSlots][3][32][kSegVecs<T>];
  T raw[2][NT][kRaw];
  float m[2][kTileSteps][NT];
};

// The kernel's pipeline buffers, declared in a function of their own rather
// than at kernel scope (measured: 1-2.5% faster on every workload, the fp32
// ones most; the placement of the CTA's shared variables is the only change).
// The segment-stream layout is larger than the 48 KB of static shared memory
// and lives in dynamic shared memory (the launch passes its size).
template <class S, bool DYN>
__device__ __forceinline__ S& pipe_smem() {
  if constexpr (DYN) {
    extern __shared__ __align__(1024) unsigned char ss_dyn_smem[];
    return *reinterpret_cast<S*>(ss_dyn_smem);
  } else {
    __shared__ __align__(16) S sm;
    return sm;
  }
}

// Dynamic shared memory of one ss_fwd_sched instantiation (0: static only).
template <typename T, int NT, int TGS, int TPB, int STAGES>
constexpr int fwd_sched_dyn_smem() {
  return kSegStream<T, TGS> ? (int)sizeof(PipeSmem<T, NT, TGS, TPB, STAGES>) : 0;
}

// One pass over steps [t_begin, t_end) of a unit: AGG = false runs the
// recurrence from h and writes y; AGG = true runs it from h (zero) without C,
// z or y and accumulates sum dt of the lane's own steps (for the aggregate's
// decay).  HAS_Z: the gate input is present.  MULTI: dstate spans several
// state groups (read-out accumulated in the fp32 partial row).
//
// The loop over 16-byte vectors is software-pipelined: the row work of
// vector j+1 (its shared-memory reads, softplus and the dt/du exchange,
// ~150 cycles of latency) is issued before the recurrence of vector j, so
// that latency overlaps the recurrence instead of stalling it.
//
// u, delta and z reach shared memory one of two ways.  Per-lane slots: each
// lane copies the next vectors of its own row (one 16-byte copy per row and
// tensor, 32 rows per warp instruction).  Segment stream (two lanes per row
// pair): every kSegVecs vectors the warp copies a whole segment of its 32
// rows, 8 rows x 64 bytes (fp32) or 16 rows x 32 bytes (bf16) per
// instruction, kSegSlots - 2 segments ahead, and a __syncwarp hands it to the
// lanes.  The per-lane form made the fp32 sweep's copies cost ~17% of its time
// (measured by leaving them out); the segments, with the same instruction
// count, cut the fp32 sweep by 7-8% and the bf16 layers by about 2%.
template <typename T, int NT, int TGS, int TPB, int STAGES, bool AGG, bool HAS_Z, bool MULTI>
__device__ __forceinline__ void scan_pass(const FwdParams& p,
                                          PipeSmem<T, NT, TGS, TPB, STAGES>& sm,
                                          const PairRows<TGS, TPB, kSegStream<T, TGS>>& rs,
                                          int64_t t_begin,
                                          int64_t t_end, f2 (&h)[2][NT / TGS / 2],
                                          const f2 (&A2)[2][NT / TGS / 2],
                                          const float (&bias)[2 / TGS],
                                          const float (&Dd)[2 / TGS],
                                          float (&dt_sum)[2 / TGS]) {
  constexpr int V = Elem<T>::kVec;
  constexpr int VP = V / 2;            // step pairs in a vector
  constexpr int G = NT / TGS;          // states per lane
  constexpr int OWN = 2 / TGS;         // own rows (row work) per lane
  constexpr int NM = AGG ? 1 : 2;      // staged state tensors: B (, C)
  constexpr bool GATE = !AGG && HAS_Z;
  constexpr int VPT = kTileSteps / V;  // vectors per tile
  constexpr int CPR = kTileSteps * (int)sizeof(T) / 16;  // 16-byte chunks per state row
  constexpr int EPC = 16 / (int)sizeof(T);                // elements per 16-byte chunk
  static_assert(STAGES >= 3 && STAGES <= VPT + 1, "pipeline depth must fit in a tile");
  constexpr bool SEG = kSegStream<T, TGS>;
  constexpr int SV = kSegVecs<T>, SR = kSegSlots;
  // the raw B/C copies of a tile join the copy group of the first segment
  // issued after the tile boundary, which is waited for (SR - 1) * SV vectors
  // later: that must come before the next tile boundary
  static_assert(!SEG || ((SR - 1) * SV <= VPT && SR >= 3), "segment ring too deep for the B/C tile");

  const int tid = threadIdx.x;
  const int64_t L = p.seqlen, N = p.dstate;
  const int ng0 = p.group * NT;  // first state of this launch's group
  const int nl0 = rs.q * G;      // first state of this lane within the group
  const int64_t nvec = (t_end - t_begin) / V;
  const T* __restrict__ ug = static_cast<const T*>(p.u);
  const T* __restrict__ dg = static_cast<const T*>(p.delta);
  const T* __restrict__ zg = static_cast<const T*>(p.z);
  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  T* __restrict__ y = static_cast<T*>(p.y);
  const bool use_softplus = p.softplus != 0;

  auto issue_vec = [&](int64_t j) {
    if constexpr (!SEG) {
    if (j < nvec) {
      const int slot = (int)(j % STAGES);
      const int64_t t = t_begin + j * V;
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        const int64_t off = rs.row[o] * L + t;
        cp_async16(&sm.x[slot][0][o][tid], ug + off);
        cp_async16(&sm.x[slot][1][o][tid], dg + off);
        if (GATE) cp_async16(&sm.x[slot][2][o][tid], zg + off);
      }
    }
    cp_async_commit();
    }
  };
  // segment stream: lane l copies vector l % SV of rows (32 i + l) / SV of the
  // warp (i < SV); rows past dim read the last channel (never stored)
  const int lane = tid & 31, wp = tid >> 5;
  int64_t seg_row[SEG ? SV : 1];
  if constexpr (SEG) {
#pragma unroll
    for (int i = 0; i < SV; ++i) {
      const int64_t dd = rs.d0 + wp * 32 + (i * 32 + lane) / SV;
      seg_row[i] = (rs.b * p.dim + (dd < p.dim ? dd : p.dim - 1)) * L;
    }
  }
  auto seg_pos = [](int row, int c) {  // 16-byte slot of vector c in row's segment
    return SV == 4 ? (c ^ ((row >> 1) & 3)) : (c ^ ((row >> 2) & 1));
  };
  auto issue_seg = [&](int64_t sg) {
    if constexpr (SEG) {
      const int64_t v0 = sg * SV;
      if (v0 < nvec) {
        const int slot = (int)(sg % SR);
        const int64_t t = t_begin + v0 * V;
        const int c = lane % SV;
#pragma unroll
        for (int i = 0; i < SV; ++i) {
          const int r = (i * 32 + lane) / SV;
          if (v0 + c < nvec) {
            const int64_t off = seg_row[i] + t + c * V;
            const int pc = seg_pos(r, c);
            cp_async16(&sm.xs[wp][slot][0][r][pc], ug + off);
            cp_async16(&sm.xs[wp][slot][1][r][pc], dg + off);
            if (GATE) cp_async16(&sm.xs[wp][slot][2][r][pc], zg + off);
          }
        }
      }
      cp_async_commit();
    }
  };
  auto issue_tile = [&](int64_t t0) {
    if (t0 >= t_end) return;
    const int tlen = (int)min((int64_t)kTileSteps, t_end - t0);
    for (int i = tid; i < NM * NT * CPR; i += TPB) {
      const int m = i / (NT * CPR);
      const int rem = i - m * NT * CPR;
      const int n = rem / CPR;
      const int j = (rem - n * CPR) * EPC;
      const int64_t ng = ng0 + n;
      if (ng < N && j < tlen)
        cp_async16(&sm.raw[m][n][j], (m == 0 ? Bg : Cg) + (rs.b * N + ng) * L + t0 + j);
    }
  };

  // bf16 I/O: y leaves as 32-byte stores of vector pairs (one L1 access for two
  // vectors; measured -5% on the Mamba-2.8B layer, but slower for fp32 I/O at
  // one warp per scheduler), when the host found rows and y 32-byte aligned
  const bool pair_store = std::is_same<T, __nv_bfloat16>::value && p.y_pairs != 0;
  uint4 ypend[OWN];
  // row work of vector j, kept in registers until its recurrence and epilogue
  float dts[2][V], dus[2][V];   // dt and du of both row slots of the group
  f2 up[OWN][VP], zp[OWN][VP];  // own u (skip) and z (gate)
  auto rowwork = [&](int64_t j, float (&dt_o)[2][V], float (&du_o)[2][V], f2 (&u_o)[OWN][VP],
                     f2 (&z_o)[OWN][VP]) {
#pragma unroll
    for (int o = 0; o < OWN; ++o) {
      f2 dp[VP];
      if constexpr (SEG) {
        const int slot = (int)((j / SV) % SR), c = seg_pos(lane, (int)(j % SV));
        to_pairs<T>(sm.xs[wp][slot][0][lane][c], u_o[o]);
        to_pairs<T>(sm.xs[wp][slot][1][lane][c], dp);
        if (GATE) to_pairs<T>(sm.xs[wp][slot][2][lane][c], z_o[o]);
      } else {
        const int slot = (int)(j % STAGES);
        to_pairs<T>(*reinterpret_cast<const uint4*>(&sm.x[slot][0][o][tid]), u_o[o]);
        to_pairs<T>(*reinterpret_cast<const uint4*>(&sm.x[slot][1][o][tid]), dp);
        if (GATE) to_pairs<T>(*reinterpret_cast<const uint4*>(&sm.x[slot][2][o][tid]), z_o[o]);
      }
#pragma unroll
      for (int m = 0; m < VP; ++m) {
        const f2 x = add2(dp[m], splat(bias[o]));
        const f2 sp = softplus2<std::is_same<T, __nv_bfloat16>::value>(x);
        f2 dtm;
        dtm.v = use_softplus ? sp.v : x.v;
        const f2 dum = mul2(dtm, u_o[o][m]);
        unpack(dtm, dt_o[o][2 * m], dt_o[o][2 * m + 1]);
        unpack(dum, du_o[o][2 * m], du_o[o][2 * m + 1]);
      }
    }
    if constexpr (TGS == 2) {
#pragma unroll
      for (int e = 0; e < V; ++e) {
        dt_o[1][e] = __shfl_xor_sync(0xffffffffu, dt_o[0][e], 1);
        du_o[1][e] = __shfl_xor_sync(0xffffffffu, du_o[0][e], 1);
      }
    }
  };

  issue_tile(t_begin);
  if constexpr (SEG) {
#pragma unroll
    for (int sg = 0; sg < SR - 1; ++sg) issue_seg(sg);
    cp_async_wait<SR - 2>();  // this lane's copies of segment 0 landed
    __syncwarp();             // ... and every lane's
  } else {
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) issue_vec(s);
    cp_async_wait<STAGES - 2>();  // vector 0 landed
  }
  rowwork(0, dts, dus, up, zp);

  // unrolled by two so that the hand-over of the next vector's row work
  // (dts_n -> dts, ...) becomes register renaming instead of moves
#pragma unroll 2
  for (int64_t j = 0; j < nvec; ++j) {
    if constexpr (SEG) {
      if ((j % SV) == SV - 1 && j + 1 < nvec) {
        // vector j+1 opens segment ns: copy segment ns + SR - 2 into the slot of
        // segment ns - 2 (every lane passed the last __syncwarp after reading
        // it), then wait for segment ns and hand it to the lanes
        const int64_t ns = (j + 1) / SV;
        issue_seg(ns + SR - 2);
        cp_async_wait<SR - 2>();
        __syncwarp();
      }
    } else {
      issue_vec(j + STAGES - 1);
      cp_async_wait<STAGES - 2>();  // this lane's copies of vector j+1 (and older) landed
    }
    const int jt = (int)(j % VPT) * V;
    if (jt == 0) {
      // tile boundary: widen + transpose the raw tile, then prefetch the next one
      const int64_t t0 = t_begin + j * V;
      const int tlen = (int)min((int64_t)kTileSteps, t_end - t0);
      __syncthreads();  // every lane's raw copies landed; the previous tile is consumed
      for (int i = tid; i < NM * NT * CPR; i += TPB) {
        const int n = i % NT;  // state fastest: conflict-free transposed stores
        const int c = (i / NT) % CPR;
        const int m = i / (NT * CPR);
        const Vec16<T> v = *reinterpret_cast<const Vec16<T>*>(&sm.raw[m][n][c * EPC]);
        const bool nok = ng0 + n < N;
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
          const int t = c * EPC + e;
          sm.m[m][t][n] = (nok && t < tlen) ? Elem<T>::to_f32(v.e[e]) : 0.f;
        }
      }
      __syncthreads();
      issue_tile(t0 + kTileSteps);
    }

    // row work of the next vector (the last vector repeats itself: unused)
    float dts_n[2][V], dus_n[2][V];
    f2 up_n[OWN][VP], zp_n[OWN][VP];
    rowwork(j + 1 < nvec ? j + 1 : j, dts_n, dus_n, up_n, zp_n);

    // the recurrence over the V steps of vector j, one group of two state pairs
    // at a time: inside a group the decays and inputs of all V steps depend only
    // on dt and du, not on the state, so their MUFU and FMUL work issues as a
    // batch while the state's own dependency chain (one FFMA2 per step) runs
    float part[2][V];  // read-out over this lane's states, per row slot and step
    f2 yac[2][V];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int s = 0; s < V; ++s) yac[r][s] = splat(0.f);
#pragma unroll
    for (int k4 = 0; k4 < G / 4; ++k4) {
#pragma unroll
      for (int s = 0; s < V; ++s) {
        const ulonglong2 bq = *reinterpret_cast<const ulonglong2*>(&sm.m[0][jt + s][nl0 + 4 * k4]);
        ulonglong2 cq = bq;
        if (!AGG) cq = *reinterpret_cast<const ulonglong2*>(&sm.m[NM - 1][jt + s][nl0 + 4 * k4]);
        const f2 bp[2] = {{bq.x}, {bq.y}};
        const f2 cp[2] = {{cq.x}, {cq.y}};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 2 * k4 + e;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const f2 a = ex2x2(mul2(splat(dts[r][s]), A2[r][k]));
            h[r][k] = fma2(a, h[r][k], mul2(splat(dus[r][s]), bp[e]));
            if (!AGG) yac[r][s] = fma2(cp[e], h[r][k], yac[r][s]);
          }
        }
      }
    }
    if (!AGG) {
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int s = 0; s < V; ++s) part[r][s] = lo_of(yac[r][s]) + hi_of(yac[r][s]);
    }

    if constexpr (AGG) {
#pragma unroll
      for (int o = 0; o < OWN; ++o)
#pragma unroll
        for (int e = 0; e < V; ++e) dt_sum[o] += dts[o][e];
    } else {
      float yv[OWN][V];
#pragma unroll
      for (int s = 0; s < V; ++s) {
        if constexpr (TGS == 1) {
          yv[0][s] = part[0][s];
          yv[1][s] = part[1][s];
        } else {
          yv[0][s] = part[0][s] + __shfl_xor_sync(0xffffffffu, part[1][s], 1);
        }
      }
      // epilogue for V steps of the own rows: earlier groups' read-out, skip, gate, store
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        const int64_t off = rs.row[o] * L + t_begin + j * V;
        if constexpr (MULTI) {
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
        }
        f2 yp[VP];
#pragma unroll
        for (int m = 0; m < VP; ++m)
          yp[m] = fma2(splat(Dd[o]), up[o][m], pack(yv[o][2 * m], yv[o][2 * m + 1]));
        if constexpr (GATE) {
#pragma unroll
          for (int m = 0; m < VP; ++m) yp[m] = mul2(yp[m], silu2(zp[o][m]));
        }
        {
          const uint4 w = from_pairs<T>(yp);
          if (pair_store) {  // vectors j-1, j of the pass as one 32-byte store
            if ((j & 1) == 0) {
              ypend[o] = w;
              if (j + 1 == nvec && rs.valid[o]) *reinterpret_cast<uint4*>(y + off) = w;
            } else if (rs.valid[o]) {
              const uint4 a = ypend[o];
              asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(y + off - V),
                           "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(w.x), "r"(w.y), "r"(w.z),
                           "r"(w.w)
                           : "memory");
            }
          } else if (rs.valid[o]) {
            *reinterpret_cast<uint4*>(y + off) = w;
          }
        }
      }
    }

    // the next vector's row work becomes the current one
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int e = 0; e < V; ++e) {
        dts[r][e] = dts_n[r][e];
        dus[r][e] = dus_n[r][e];
      }
#pragma unroll
    for (int o = 0; o < OWN; ++o)
#pragma unroll
      for (int m = 0; m < VP; ++m) {
        up[o][m] = up_n[o][m];
        zp[o][m] = zp_n[o][m];
      }
  }
  cp_async_wait<0>();
}

// The persistent, ticketed kernel.  grid = resident CTAs (at most the unit
// count), block = TPB; one launch per state group of NT states.
template <typename T, int NT, int TGS, int TPB, int STAGES, bool HAS_Z, bool MULTI>
__global__ void __launch_bounds__(TPB) ss_fwd_sched(const FwdParams p) {
  constexpr int G = NT / TGS;
  constexpr int GP = G / 2;
  constexpr int OWN = 2 / TGS;
  constexpr bool SEG = kSegStream<T, TGS>;
  constexpr int RPC = PairRows<TGS, TPB, SEG>::kRowsPerCta;
  static_assert(TGS == 1 || TGS == 2, "one or two lanes per row pair");
  static_assert(G % 4 == 0, "a lane holds a multiple of four states");
  PipeSmem<T, NT, TGS, TPB, STAGES>& sm = pipe_smem<PipeSmem<T, NT, TGS, TPB, STAGES>, SEG>();
  __shared__ unsigned s_ticket, s_flag;

  const int tid = threadIdx.x;
  const int64_t L = p.seqlen, N = p.dstate;
  const int64_t M = p.tiles;
  const int64_t units = M * p.nchunks;
  const int ng0 = p.group * NT;

  for (;;) {
    if (tid == 0) s_ticket = atomicAdd(p.ticket, 1u);
    __syncthreads();
    const int64_t t = s_ticket;
    __syncthreads();
    if (t >= units) break;
    const int k = (int)(t / M);
    const int64_t tile = t - (int64_t)k * M;
    const PairRows<TGS, TPB, SEG> rs(tile, p.dim);
    const int nl0 = rs.q * G;
    const int64_t t_begin = (int64_t)k * p.chunk_len;
    const int64_t t_end = min(L, t_begin + p.chunk_len);
    auto rec = [&](int kk, int s, int n) -> int64_t {  // record index of (unit kk of this tile)
      return (((int64_t)kk * M + tile) * RPC + rs.rc[s]) * NT + n;
    };

    f2 A2[2][GP], h[2][GP];
    float bias[OWN], Dd[OWN], dt_sum[OWN];
#pragma unroll
    for (int o = 0; o < OWN; ++o) {
      bias[o] = p.bias ? p.bias[rs.d[o]] : 0.f;
      Dd[o] = p.D ? p.D[rs.d[o]] : 0.f;
      dt_sum[o] = 0.f;
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
#pragma unroll
      for (int kk = 0; kk < GP; ++kk) {
        float a[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t n = ng0 + nl0 + 2 * kk + e;
          a[e] = n < N ? p.A[rs.d[s] * N + n] * kLog2e : 0.f;
        }
        A2[s][kk] = pack(a[0], a[1]);
        h[s][kk] = splat(0.f);
      }
    }
    // the state before step 0 (chunk 0 only)
    auto load_h0 = [&]() {
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int kk = 0; kk < GP; ++kk) {
          float v[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int64_t n = ng0 + nl0 + 2 * kk + e;
            v[e] = (p.h0 && n < N) ? p.h0[rs.row[s] * N + n] : 0.f;
          }
          h[s][kk] = pack(v[0], v[1]);
        }
    };
    if (k == 0) load_h0();

    // ---- carry into this unit ----
    bool published = false;  // this unit's end state already published
    if (k > 0 && p.chained) {
      if (tid == 0) s_flag = wait_flag(&p.flags[(int64_t)(k - 1) * M + tile], kUnitIncl);
      __syncthreads();
      const bool ok = s_flag >= kUnitIncl;
      __syncthreads();
      if (ok) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int kk = 0; kk < GP; ++kk)
            h[s][kk] = pack(__ldcg(&p.unit_incl[rec(k - 1, s, nl0 + 2 * kk)]),
                            __ldcg(&p.unit_incl[rec(k - 1, s, nl0 + 2 * kk + 1)]));
      }
    } else if (k == 0 && !p.chained && p.nchunks > 1) {
      // decoupled, first chunk: its carry is h0, so the state its first pass
      // reaches from h0 is its end state; publishing that before the main
      // pass lets the look-backs of the later chunks finish early.  h0 is read
      // again for the main pass before the flag is released, so a successor
      // that writes last_state over h0 (in-place update) cannot come first.
      scan_pass<T, NT, TGS, TPB, STAGES, true, HAS_Z, MULTI>(p, sm, rs, t_begin, t_end, h, A2, bias, Dd,
                                               dt_sum);
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int kk = 0; kk < GP; ++kk) {
          float hv[2];
          unpack(h[s][kk], hv[0], hv[1]);
          p.unit_incl[rec(0, s, nl0 + 2 * kk)] = hv[0];
          p.unit_incl[rec(0, s, nl0 + 2 * kk + 1)] = hv[1];
        }
      load_h0();
      __threadfence();
      __syncthreads();
      if (tid == 0) st_release(&p.flags[tile], kUnitIncl);
      published = true;
    } else if (k > 0) {
      // decoupled: own aggregate first, published for successors
      scan_pass<T, NT, TGS, TPB, STAGES, true, HAS_Z, MULTI>(p, sm, rs, t_begin, t_end, h, A2, bias, Dd,
                                               dt_sum);
      float sum[2];
      if constexpr (TGS == 1) {
        sum[0] = dt_sum[0];
        sum[1] = dt_sum[1];
      } else {
        sum[0] = dt_sum[0];
        sum[1] = __shfl_xor_sync(0xffffffffu, sum[0], 1);
      }
      f2 Pk[2][GP], ek[2][GP];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
#pragma unroll
        for (int kk = 0; kk < GP; ++kk) {
          Pk[s][kk] = ex2x2(mul2(splat(sum[s]), A2[s][kk]));
          ek[s][kk] = h[s][kk];
          float pv[2], ev[2];
          unpack(Pk[s][kk], pv[0], pv[1]);
          unpack(ek[s][kk], ev[0], ev[1]);
          p.unit_agg[rec(k, s, nl0 + 2 * kk)] = make_float2(pv[0], ev[0]);
          p.unit_agg[rec(k, s, nl0 + 2 * kk + 1)] = make_float2(pv[1], ev[1]);
        }
      }
      __threadfence();
      __syncthreads();
      if (tid < 32) {
        if (tid == 0) st_release(&p.flags[(int64_t)k * M + tile], kUnitAgg);
        const unsigned r = look_back(p.flags, M, tile, k, tid);
        if (tid == 0) s_flag = r;  // 0: a wait gave up
      }
      __syncthreads();
      const unsigned found = s_flag;
      __syncthreads();
      // carry into unit k: the end state of chunk j0, then the aggregates of
      // chunks j0+1 .. k-1 applied in chunk order
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int kk = 0; kk < GP; ++kk) h[s][kk] = splat(0.f);
      if (found != 0u) {
        const int j0 = (int)found - 1;
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int kk = 0; kk < GP; ++kk)
            h[s][kk] = pack(__ldcg(&p.unit_incl[rec(j0, s, nl0 + 2 * kk)]),
                            __ldcg(&p.unit_incl[rec(j0, s, nl0 + 2 * kk + 1)]));
        // two chunks' records are loaded before either is applied, so their
        // loads overlap; the fold itself stays in chunk order
        auto fold = [&](int jj, auto count) {
          constexpr int NC = decltype(count)::value;
          float2 r[NC][2][GP][2];
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
              for (int kk = 0; kk < GP; ++kk)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                  r[c][s][kk][e] = __ldcg(&p.unit_agg[rec(jj + c, s, nl0 + 2 * kk + e)]);
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
              for (int kk = 0; kk < GP; ++kk)
                h[s][kk] = fma2(pack(r[c][s][kk][0].x, r[c][s][kk][1].x), h[s][kk],
                                pack(r[c][s][kk][0].y, r[c][s][kk][1].y));
        };
        int jj = j0 + 1;
        for (; jj + 1 < k; jj += 2) fold(jj, std::integral_constant<int, 2>{});
        if (jj < k) fold(jj, std::integral_constant<int, 1>{});
      }
      // own end state = own aggregate applied to the carry, published before the main pass
      if (k + 1 < p.nchunks) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int kk = 0; kk < GP; ++kk) {
            const f2 hend = fma2(Pk[s][kk], h[s][kk], ek[s][kk]);
            float hv[2];
            unpack(hend, hv[0], hv[1]);
            p.unit_incl[rec(k, s, nl0 + 2 * kk)] = hv[0];
            p.unit_incl[rec(k, s, nl0 + 2 * kk + 1)] = hv[1];
          }
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(&p.flags[(int64_t)k * M + tile], kUnitIncl);
      }
      published = true;
    }

    // ---- main pass from the carry ----
    scan_pass<T, NT, TGS, TPB, STAGES, false, HAS_Z, MULTI>(p, sm, rs, t_begin, t_end, h, A2, bias, Dd,
                                              dt_sum);

    if (k + 1 < p.nchunks) {
      if (!published) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
          for (int kk = 0; kk < GP; ++kk) {
            float hv[2];
            unpack(h[s][kk], hv[0], hv[1]);
            p.unit_incl[rec(k, s, nl0 + 2 * kk)] = hv[0];
            p.unit_incl[rec(k, s, nl0 + 2 * kk + 1)] = hv[1];
          }
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(&p.flags[(int64_t)k * M + tile], kUnitIncl);
      }
    } else if (p.last_state) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!rs.valid[s]) continue;
#pragma unroll
        for (int kk = 0; kk < GP; ++kk) {
          float hv[2];
          unpack(h[s][kk], hv[0], hv[1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int64_t n = ng0 + nl0 + 2 * kk + e;
            if (n < N) p.last_state[rs.row[s] * N + n] = hv[e];
          }
        }
      }
    }
    __syncthreads();  // shared buffers are reused by the next unit
  }
}

}  // namespace ss
