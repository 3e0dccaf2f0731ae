// Mamba-2 forward (one scalar decay per head) on the 5th-generation tensor
// cores: the chunked evaluation that the Mamba-2 cuTile news page ("Прорыв в
// оптимизации SSM-моделей", sections "Три оптимизированных ядра" and
// "Технические детали оптимизации") splits into chunk_cumsum, fwd_pass_state
// and compute_out, here fused into one kernel per (batch, head):
//
//   h_t = exp(A dt_t) h_{t-1} + dt_t x_t B_t^T   (state [P, N])
//   y_t = h_t C_t + D x_t
//
// One CTA walks the chunks of its (b, h) in order and keeps the state across
// them in registers (fp32).  For a chunk of Q = 128 steps starting at t0, with
// cum_t the decay accumulated inside the chunk up to t (in log2 units):
//
//   CB    = C B^T                                        [Q x Q]  tensor cores
//   Y_in  = C H^T  (H the state entering the chunk)      [Q x P]  tensor cores
//   M     = CB . exp(cum_t - cum_s) dt_s  for s <= t, else 0
//   Y_dg  = M X                                          [Q x P]  tensor cores
//   S     = B^T (w . X),  w_s = exp(cum_end - cum_s) dt_s [N x P] tensor cores
//   y_t   = exp(cum_t) Y_in[t] + Y_dg[t] + D x_t
//   H    <- exp(cum_end) H + S^T                          (the jump formula)
//
// The four products are tcgen05.mma kind::f16 (bf16 operands from shared
// memory, fp32 accumulators in tensor memory), issued by one thread and
// completed through an mbarrier; threads own tensor-memory lanes (rows t of CB
// and Y, rows n of S).  Every operand uses the 128-byte-swizzle layout: rows of
// 64 elements (128 bytes) whose 16-byte chunks are XOR-permuted by the row
// index mod 8, 8-row groups 1024 bytes apart, which is what TMA writes for a
// 64 x 128 box and what lets a warp write a chunk of 32 rows without bank
// conflicts.  B serves as the CB operand (K-major, K = n) and as the state
// product's A operand (MN-major, K = s) from the same bytes.
#pragma once

#include <cuda.h>

#include "ss_device.cuh"
#include "ss_sched.cuh"

namespace ss {

constexpr int kSsdQ = 128;  // steps per chunk (the MMA's M)
constexpr int kSsdP = 64;   // head dim
constexpr int kSsdN = 128;  // dstate
constexpr int kSsdThreads = 256;

// shared-memory map (bytes from the 1024-aligned dynamic base)
constexpr uint32_t kSsdOffC = 0;           // C [t][n], then M [t][s]: two 64-column halves
constexpr uint32_t kSsdOffB = 32768;       // B [s][n]: two 64-column halves
constexpr uint32_t kSsdOffX = 65536;       // x [s][p]
constexpr uint32_t kSsdOffH = 81920;       // H [n][p], then w.x [s][p]
constexpr uint32_t kSsdHalf = 16384;       // bytes of a 64-column half of a 128-row tile
// per-step tables of two chunks (this one and the next): fp32 [2][Q] each
constexpr uint32_t kSsdOffCum = 98304;     // decay sums cum
constexpr uint32_t kSsdOffDt = 99328;      // dt
constexpr uint32_t kSsdOffG = 100352;      // block factors
constexpr uint32_t kSsdOffMisc = 101376;   // warp sums, mbarriers, tensor-memory address
constexpr uint32_t kSsdSmemBytes = 101376 + 64;
constexpr uint32_t kSsdTmemCols = 256;     // CB / S [0,128), Y_in [128,192), Y_dg [192,256)

struct SsdParams {
  // TMA descriptors (3-D: columns, steps, batch; 128-byte-swizzled boxes of
  // 64 columns x 128 steps, zero past the sequence's end) of x [b,L,H*P] and
  // B, C [b,L,G*N]
  CUtensorMap tx, tb, tc;
  const __nv_bfloat16* x;   // [b,L,H,P]
  const __nv_bfloat16* dt;  // [b,L,H]
  const float* A;           // [H]
  const __nv_bfloat16* B;   // [b,L,G,N]
  const __nv_bfloat16* C;   // [b,L,G,N]
  const float* D;           // [H] or null
  const float* bias;        // [H] or null
  int softplus;
  __nv_bfloat16* y;         // [b,L,H,P]
  float* final_state;       // [b,H,P,N] or null
  int64_t batch, seqlen, nheads, ngroups;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start,
// leading byte offset (MN-major: between 64-element atoms along M or N; unused
// by K-major), stride byte offset (between 8-row groups: 1024), version 1,
// layout 2 (128-byte swizzle).  A K-major operand steps through K inside an
// atom by moving the start 32 bytes per 16 elements.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// start of K step ks (16 elements) of a K-major tile whose K = 128 is split in
// two 64-column halves
__device__ __forceinline__ uint32_t kmajor_step(uint32_t base, int ks) {
  return base + (ks >> 2) * kSsdHalf + (ks & 3) * 32;
}
// byte offset of 16-byte chunk c (columns 8c..8c+7 of a 64-column half) of row r
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, M = 128,
// the given N; a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t umma_idesc(int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
      bar));
}

// Wait for the mbarrier phase with the given parity; false after kSpinLimit
// polls (the device error word is then set).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (long long i = 0; i < kSpinLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  atomicOr(&g_ss_device_error, kErrTimeout);
  return false;
}

// Start reading 32 consecutive fp32 columns of this warp's 32 tensor-memory
// lanes; the values are valid after tmem_wait on the same array.
__device__ __forceinline__ void tmem_ld32_async(uint32_t addr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(addr));
}
// Wait for this thread's tensor-memory reads; the array is an operand so that
// no use of it is scheduled before the wait.
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ float fu(uint32_t v) { return __uint_as_float(v); }

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One TMA box (64 columns x 128 steps of one batch row) into shared memory:
// 128 rows of 128 bytes, 128-byte swizzled (16 KB).
__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                          int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// grid = batch * nheads CTAs (one per (b, h)), block = 256, dynamic shared
// memory kSsdSmemBytes.  Requires P = 64, N = 128 and 16-byte aligned rows.
//
// Thread i works on row r = 32 (w % 4) + lane of every Q x * matrix (warp w
// may read only tensor-memory lanes 32 (w % 4) ..), half hf = w / 4 of its
// columns.  The next chunk's copies are issued as soon as the second pair of
// products has consumed the shared operands, so they overlap the epilogue.
__global__ void __launch_bounds__(kSsdThreads, 2) ss_ssd_fwd(const __grid_constant__ SsdParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int Q = kSsdQ, P = kSsdP, N = kSsdN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hf = warp >> 2;
  const int r = q4 * 32 + lane;  // row (t, s or n) of this thread
  const int64_t H = p.nheads, G = p.ngroups, L = p.seqlen;
  const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
  const int64_t g = h / (H / G);

  unsigned char* sC = smem + kSsdOffC;
  unsigned char* sX = smem + kSsdOffX;
  unsigned char* sH = smem + kSsdOffH;
  float* cum2 = reinterpret_cast<float*>(smem + kSsdOffCum);
  float* dts2 = reinterpret_cast<float*>(smem + kSsdOffDt);
  float* gs2 = reinterpret_cast<float*>(smem + kSsdOffG);
  float* wsum = reinterpret_cast<float*>(smem + kSsdOffMisc);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kSsdOffMisc + 32);   // products
  uint64_t* lbar = reinterpret_cast<uint64_t*>(smem + kSsdOffMisc + 40);  // copies
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kSsdOffMisc + 48);
  const uint32_t uC = smem_u32(sC), uB = smem_u32(smem + kSsdOffB), uX = smem_u32(sX),
                 uH = smem_u32(sH);
  const uint32_t ubar = smem_u32(bar), ulbar = smem_u32(lbar);

  if (smem_u32(smem) & 1023u) {  // the swizzled TMA boxes need a 1024-byte aligned base
    if (tid == 0) atomicOr(&g_ss_device_error, kErrTimeout);
    return;
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ubar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ulbar));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tslot)),
                 "r"(kSsdTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  const uint32_t tlane = tm + ((uint32_t)(q4 * 32) << 16);  // this warp's lanes

  const float A2 = p.A[h] * kLog2e;
  const float bias = p.bias ? p.bias[h] : 0.f;
  const float Dh = p.D ? p.D[h] : 0.f;
  float hs[P / 2];  // state row n = r, columns p in [32 hf, 32 hf + 32)
#pragma unroll
  for (int i = 0; i < P / 2; ++i) hs[i] = 0.f;

  // chunk c's rows of C, B and x by TMA (thread 0; completes on lbar), and
  // its dt (warps 0-3, row r)
  const unsigned short* dt_bits = reinterpret_cast<const unsigned short*>(p.dt);
  auto load_dt = [&](int64_t c) -> uint32_t {  // raw bf16 bits of chunk c's dt (warps 0-3)
    const int64_t t = c * Q + r;
    return (hf == 0 && t < L) ? (uint32_t)dt_bits[(b * L + t) * H + h] : 0u;
  };
  // (lane 0 of warps 0-4 each issue one box; warp 0 also posts the byte count)
  auto issue = [&](int64_t c) {
    const int t0 = (int)(c * Q);
    if (lane == 0 && warp < 5) {
      if (warp == 0) mbar_expect_tx(ulbar, (2 * (N / 64) + P / 64) * kSsdHalf);
      if (warp < 4) {
        const int a = warp & 1;
        tma_load3((warp < 2 ? uC : uB) + a * kSsdHalf, warp < 2 ? &p.tc : &p.tb,
                  (int)(g * N + 64 * a), t0, (int)b, ulbar);
      } else {
        tma_load3(uX, &p.tx, (int)(h * P), t0, (int)b, ulbar);
      }
    }
  };
  // decay sums, dt and block factors of chunk cc into table buf (warps 0-3,
  // row s = r): cum_s = sum_{r<=s} dt_r A log2e, and the factors of the
  // below-diagonal 32 x 32 blocks: exp2(cum_t - cum_s) = exp2(cum_t - cum_e)
  // exp2(cum_e - cum_s), e the block's last column; both exponents are <= 0
  // there (the decay only shrinks), so neither overflows
  auto scan_chunk = [&](int64_t cc, uint32_t bits, int buf) {
    float dtv = 0.f;
    if (cc * Q + r < L) {
      const float xdt = __uint_as_float(bits << 16) + bias;
      dtv = p.softplus ? lo_of(softplus2(splat(xdt))) : xdt;
    }
    float run = dtv * A2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += v;
    }
    if (lane == 31) wsum[warp] = run;
    dts2[buf * Q + r] = dtv;
    asm volatile("bar.sync 1, 128;" ::: "memory");  // warps 0-3 only
#pragma unroll
    for (int w = 0; w < 3; ++w)
      if (w < warp) run += wsum[w];
    cum2[buf * Q + r] = run;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    gs2[buf * Q + r] = ex2(cum2[buf * Q + (r | 31)] - run) * dtv;
  };

  constexpr uint32_t kIdCB = umma_idesc(128, 0, 0);
  constexpr uint32_t kIdY = umma_idesc(64, 0, 1);
  constexpr uint32_t kIdS = umma_idesc(64, 1, 1);
  uint32_t parity = 0, lparity = 0;
  bool ok = true;
  const int64_t nchunks = (L + Q - 1) / Q;
  issue(0);
  // the tables of chunk 0 now; those of chunk c + 1 while the tensor cores run
  // chunk c's second pair of products (dt is loaded a chunk before it is used)
  if (hf == 0) scan_chunk(0, load_dt(0), 0);
  uint32_t dt_nxt = load_dt(1);
  for (int64_t c = 0; c < nchunks && ok; ++c) {
    const int64_t t0 = c * Q;
    const int len = (int)(L - t0 < Q ? L - t0 : Q);
    const int buf = (int)(c & 1);
    const float* cum = cum2 + buf * Q;
    const float* dts = dts2 + buf * Q;
    const float* gs = gs2 + buf * Q;

    ok = __syncthreads_and(mbar_wait(ulbar, lparity));  // chunk c's copies have landed
    lparity ^= 1;
    if (!ok) break;

    // ---- CB = C B^T, Y_in = C H^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks)
        umma(tm + 0, umma_desc(kmajor_step(uC, ks), 16), umma_desc(kmajor_step(uB, ks), 16), kIdCB,
             ks > 0);
      if (c > 0) {
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
          umma(tm + 128, umma_desc(kmajor_step(uC, ks), 16), umma_desc(uH + ks * 2048, 16), kIdY,
               ks > 0);
      }
      umma_commit(ubar);
    }
    ok = __syncthreads_and(mbar_wait(ubar, parity));
    parity ^= 1;
    tc_fence_after();
    if (!ok) break;

    // ---- M (row t = r) into C's buffer: D on the diagonal, zero above it
    {
      const int t = r;
      const float ct = cum[t];
      auto store8 = [&](int jb, const float (&m)[8]) {  // columns 8 jb .. 8 jb + 7
        *reinterpret_cast<uint4*>(sC + (jb >> 3) * kSsdHalf + sw128(t, jb & 7)) =
            make_uint4(bf16x2(m[0], m[1]), bf16x2(m[2], m[3]), bf16x2(m[4], m[5]),
                       bf16x2(m[6], m[7]));
      };
      // block q (columns 32 q .. 32 q + 31) below the diagonal, from its CB values
      auto full_block = [&](int q, const uint32_t (&cb)[32]) {
        const float et = ex2(ct - cum[q * 32 + 31]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float m[8], gv[8];
          *reinterpret_cast<float4*>(gv) = *reinterpret_cast<const float4*>(gs + q * 32 + k * 8);
          *reinterpret_cast<float4*>(gv + 4) = *reinterpret_cast<const float4*>(gs + q * 32 + k * 8 + 4);
#pragma unroll
          for (int e = 0; e < 8; ++e) m[e] = fu(cb[k * 8 + e]) * et * gv[e];
          store8(q * 4 + k, m);
        }
      };
      if (hf == 0) {  // the diagonal block q4: exp2(cum_t - cum_s) per element
        uint32_t cb[32];
        tmem_ld32_async(tlane + q4 * 32, cb);
        tmem_wait(cb);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float m[8], cv[8], dv[8];
          const int s0 = q4 * 32 + k * 8;
          *reinterpret_cast<float4*>(cv) = *reinterpret_cast<const float4*>(cum + s0);
          *reinterpret_cast<float4*>(cv + 4) = *reinterpret_cast<const float4*>(cum + s0 + 4);
          *reinterpret_cast<float4*>(dv) = *reinterpret_cast<const float4*>(dts + s0);
          *reinterpret_cast<float4*>(dv + 4) = *reinterpret_cast<const float4*>(dts + s0 + 4);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = s0 + e;
            const float v = fu(cb[k * 8 + e]) * ex2(ct - cv[e]) * dv[e];
            m[e] = s < t ? v : (s == t ? v + Dh : 0.f);
          }
          store8(q4 * 4 + k, m);
        }
      } else {  // blocks q < q4 factorised, blocks q > q4 zero
#pragma unroll
        for (int q = 0; q < Q / 32 - 1; ++q) {
          if (q < q4) {
            uint32_t cb[32];
            tmem_ld32_async(tlane + q * 32, cb);
            tmem_wait(cb);
            full_block(q, cb);
          }
        }
#pragma unroll
        for (int q = 1; q < Q / 32; ++q) {
          if (q > q4) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<uint4*>(sC + ((q * 4 + k) >> 3) * kSsdHalf + sw128(t, (q * 4 + k) & 7)) =
                  make_uint4(0, 0, 0, 0);
          }
        }
      }
      // w.x (row s = r, columns [32 hf, 32 hf + 32)) into H's buffer
      const int s = r;
      const float ws = ex2(cum[Q - 1] - cum[s]) * dts[s];
#pragma unroll
      for (int jj = 0; jj < P / 16; ++jj) {
        const int j = hf * (P / 16) + jj;
        const uint4 v = *reinterpret_cast<const uint4*>(sX + sw128(s, j));
        *reinterpret_cast<uint4*>(sH + sw128(s, j)) =
            make_uint4(bf16x2(bf_lo(v.x) * ws, bf_hi(v.x) * ws), bf16x2(bf_lo(v.y) * ws, bf_hi(v.y) * ws),
                       bf16x2(bf_lo(v.z) * ws, bf_hi(v.z) * ws), bf16x2(bf_lo(v.w) * ws, bf_hi(v.w) * ws));
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- Y_dg = M X (with the skip), S = B^T (w.x)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < Q / 16; ++ks) {
        umma(tm + 192, umma_desc(kmajor_step(uC, ks), 16), umma_desc(uX + ks * 2048, 16), kIdY,
             ks > 0);
        umma(tm + 0, umma_desc(uB + ks * 2048, kSsdHalf), umma_desc(uH + ks * 2048, 16), kIdS,
             ks > 0);
      }
      umma_commit(ubar);
    }
    if (hf == 0 && c + 1 < nchunks) scan_chunk(c + 1, dt_nxt, buf ^ 1);
    ok = __syncthreads_and(mbar_wait(ubar, parity));
    parity ^= 1;
    tc_fence_after();
    if (!ok) break;
    // the shared operands are consumed: the next chunk's copies overlap the epilogue
    if (c + 1 < nchunks) issue(c + 1);
    dt_nxt = load_dt(c + 2);

    // ---- state (row n = r): H <- exp(cum_end) H + S^T, then its bf16 copy
    uint32_t sv[32], yd[32];
    tmem_ld32_async(tlane + hf * 32, sv);
    tmem_ld32_async(tlane + 192 + hf * 32, yd);  // Y_dg, for the output below
    {
      const int n = r;
      const float decay = ex2(cum[Q - 1]);
      tmem_wait(sv);
#pragma unroll
      for (int i = 0; i < 32; ++i) hs[i] = fmaf(decay, hs[i], fu(sv[i]));
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        *reinterpret_cast<uint4*>(sH + sw128(n, hf * 4 + jj)) =
            make_uint4(bf16x2(hs[jj * 8 + 0], hs[jj * 8 + 1]), bf16x2(hs[jj * 8 + 2], hs[jj * 8 + 3]),
                       bf16x2(hs[jj * 8 + 4], hs[jj * 8 + 5]), bf16x2(hs[jj * 8 + 6], hs[jj * 8 + 7]));
    }
    // ---- output (row t = r, columns [32 hf, 32 hf + 32)): y = exp(cum_t) Y_in + Y_dg
    {
      const int t = r;
      tmem_wait(yd);
      float yv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) yv[i] = fu(yd[i]);
      if (c > 0) {
        uint32_t yi[32];
        tmem_ld32_async(tlane + 128 + hf * 32, yi);
        const float et = ex2(cum[t]);
        tmem_wait(yi);
#pragma unroll
        for (int i = 0; i < 32; ++i) yv[i] = fmaf(et, fu(yi[i]), yv[i]);
      }
      if (t < len) {
        __nv_bfloat16* yrow = p.y + ((b * L + t0 + t) * H + h) * P + hf * 32;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(yrow + k * 8) =
              make_uint4(bf16x2(yv[k * 8 + 0], yv[k * 8 + 1]), bf16x2(yv[k * 8 + 2], yv[k * 8 + 3]),
                         bf16x2(yv[k * 8 + 4], yv[k * 8 + 5]), bf16x2(yv[k * 8 + 6], yv[k * 8 + 7]));
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
  }

  if (ok && p.final_state) {
    float* fs = p.final_state + (b * H + h) * P * N + (int64_t)(hf * 32) * N;
#pragma unroll
    for (int i = 0; i < P / 2; ++i) fs[i * N + r] = hs[i];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm),
                 "r"(kSsdTmemCols));
}

}  // namespace ss
