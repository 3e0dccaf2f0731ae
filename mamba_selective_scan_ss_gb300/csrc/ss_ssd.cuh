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
//   M     = CB . exp(cum_t - cum_s) dt_s  for s <= t, else 0; + D on the diagonal
//   Y_dg  = M X                                          [Q x P]  tensor cores
//   S     = B^T (w . X),  w_s = exp(cum_end - cum_s) dt_s [N x P] tensor cores
//   y_t   = exp(cum_t) Y_in[t] + Y_dg[t]
//   H    <- exp(cum_end) H + S^T                          (the jump formula)
//
// The CTA is warp-specialised and pipelined over chunks: a producer warp
// issues the TMA copies (C and B double-buffered, so chunk c+1's arrive
// while chunk c is computed), an MMA warp issues the tcgen05.mma products
// (bf16 operands from shared memory, fp32 accumulators in tensor memory; C.B^T
// double-buffered, so chunk c+1's runs while the threads finish chunk c),
// eight prep warps build M and w.x of chunk c+1 while four epilogue warps
// finish chunk c (the state update and y).  They meet on mbarriers; every
// wait is bounded.  Every operand uses the 128-byte-swizzle
// layout: rows of 64 elements (128 bytes) whose 16-byte chunks are
// XOR-permuted by the row index mod 8, 8-row groups 1024 bytes apart, which is
// what TMA writes for a 64 x 128 box and what lets a warp write a chunk of 32
// rows without bank conflicts.  B serves as the CB operand (K-major, K = n)
// and as the state product's A operand (MN-major, K = s) from the same bytes.
#pragma once

#include <cuda.h>

#include "ss_device.cuh"
#include "ss_sched.cuh"

namespace ss {

constexpr int kSsdQ = 128;  // steps per chunk (the MMA's M)
constexpr int kSsdP = 64;   // head dim
constexpr int kSsdN = 128;  // dstate
constexpr int kSsdPrepWarps = 8;  // M and w.x, two threads per row
constexpr int kSsdEpiWarps = 4;   // state update and y, one thread per row
constexpr int kSsdProducerWarp = kSsdPrepWarps + kSsdEpiWarps, kSsdMmaWarp = kSsdProducerWarp + 1;
constexpr int kSsdThreads = 32 * (kSsdMmaWarp + 1);

// shared-memory map (bytes from the 1024-aligned dynamic base)
constexpr uint32_t kSsdHalf = 16384;       // bytes of a 64-column half of a 128-row tile
constexpr uint32_t kSsdSlot = 65536;       // one copy slot: C [t][n] then B [s][n]
constexpr uint32_t kSsdOffX = 131072;      // x [s][p]
constexpr uint32_t kSsdOffM = 147456;      // M [t][s]: two 64-column halves
constexpr uint32_t kSsdOffW = 180224;      // w.x [s][p]
constexpr uint32_t kSsdOffH = 196608;      // H [n][p] (bf16 copy of the state)
// per-step tables of three chunks (the epilogue's, the prep warps' and the
// next): fp32 [3][Q] each
constexpr uint32_t kSsdOffCum = 212992;    // decay sums cum
constexpr uint32_t kSsdOffDt = 214528;     // dt
constexpr uint32_t kSsdOffG = 216064;      // block factors
constexpr uint32_t kSsdOffMisc = 217600;   // warp sums, mbarriers, abort flag, tensor-memory address
constexpr uint32_t kSsdSmemBytes = 217600 + 256;
// tensor memory: C.B^T of two chunks [0,128) [128,256), Y_dg [256,320),
// S [320,384), Y_in [384,448)
constexpr uint32_t kSsdTmemCols = 512;
constexpr uint32_t kTmYdg = 256, kTmS = 320, kTmYin = 384;

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
  const float* h0;          // [b,H,P,N] state before step 0, or null (zero)
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
// polls (the device error word and the CTA's abort flag are then set), or at
// once when another wait of the CTA has already given up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  for (long long i = 0; i < kSpinLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (*abort) return false;
  }
  *abort = 1;
  atomicOr(&g_ss_device_error, kErrTimeout);
  return false;
}
// OR of a predicate over the threads of named barrier `id` (count threads),
// which it also synchronises: the same answer in every thread.
template <int ID, int COUNT>
__device__ __forceinline__ bool bar_any(bool v) {
  uint32_t res;
  asm volatile(
      "{\n.reg .pred q, r;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred r, %2, %3, q;\n"
      "selp.u32 %0, 1, 0, r;\n}\n"
      : "=r"(res)
      : "r"((uint32_t)v), "n"(ID), "n"(COUNT)
      : "memory");
  return res != 0;
}
// Non-blocking: has the mbarrier phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// The same for 16 columns.
__device__ __forceinline__ void tmem_ld16_async(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
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

// grid = batch * nheads CTAs (one per (b, h)), block = kSsdThreads, dynamic
// shared memory kSsdSmemBytes (one CTA per SM).  Requires P = 64, N = 128 and
// 16-byte aligned rows.
//
// A prep thread (warps 0-7) works on row r = 32 (w % 4) + lane of every
// Q x * matrix (warp w may read only tensor-memory lanes 32 (w % 4) ..), half
// hf = w / 4 of its columns; an epilogue thread (warps 8-11) on the whole of
// row r.  Warp 12 is the producer, warp 13 the MMA issuer.
// HAS_H0: the sequence starts from p.h0 (else from zero); a template
// parameter so that the zero-state kernel carries none of its bookkeeping.
template <bool HAS_H0>
__global__ void __launch_bounds__(kSsdThreads, 1) ss_ssd_fwd(const __grid_constant__ SsdParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int Q = kSsdQ, P = kSsdP, N = kSsdN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hf = (warp >> 2) & 1;
  const int r = q4 * 32 + lane;  // row (t, s or n) of a compute thread
  const int64_t H = p.nheads, G = p.ngroups, L = p.seqlen;
  const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
  const int64_t g = h / (H / G);
  const int64_t nchunks = (L + Q - 1) / Q;

  unsigned char* sX = smem + kSsdOffX;
  unsigned char* sM = smem + kSsdOffM;
  unsigned char* sW = smem + kSsdOffW;
  unsigned char* sH = smem + kSsdOffH;
  float* cum2 = reinterpret_cast<float*>(smem + kSsdOffCum);
  float* dts2 = reinterpret_cast<float*>(smem + kSsdOffDt);
  float* gs2 = reinterpret_cast<float*>(smem + kSsdOffG);
  float* wsum = reinterpret_cast<float*>(smem + kSsdOffMisc);
  const uint32_t ubar0 = smem_u32(smem + kSsdOffMisc + 64);  // 17 mbarriers, 8 bytes each
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kSsdOffMisc + 208);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kSsdOffMisc + 216);
  const uint32_t uS0 = smem_u32(smem), uX = smem_u32(sX), uM = smem_u32(sM), uW = smem_u32(sW),
                 uH = smem_u32(sH);
  // mbarriers: copies of C and B of slot 0/1 (tx), copy of x (tx), C.B^T of
  // slot 0/1 done, M and w.x written (prep warps), Y_dg and S done, Y_in
  // done, H written and the chunk's accumulators read (epilogue warps), slot
  // 0/1 free, and the ring of step tables: buffer k written (warps 0-3) and
  // read (epilogue warps).  Every barrier's next phase depends on each of its
  // waiters having passed the current one, so parity waits cannot alias.
  const uint32_t bFullCB = ubar0, bFullX = ubar0 + 16, bCB = ubar0 + 24, bMready = ubar0 + 40,
                 bMma2 = ubar0 + 48, bYin = ubar0 + 56, bHready = ubar0 + 64,
                 bSlotFree = ubar0 + 72, bTFull = ubar0 + 88, bTEmpty = ubar0 + 112;

  if (smem_u32(smem) & 1023u) {  // the swizzled TMA boxes need a 1024-byte aligned base
    if (tid == 0) atomicOr(&g_ss_device_error, kErrTimeout);
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bFullCB + 8 * i, 1);
      mbar_init(bCB + 8 * i, 1);
      mbar_init(bSlotFree + 8 * i, 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(bTFull + 8 * i, 128);
      mbar_init(bTEmpty + 8 * i, 32 * kSsdEpiWarps);
    }
    mbar_init(bFullX, 1);
    mbar_init(bMready, 32 * kSsdPrepWarps);
    mbar_init(bMma2, 1);
    mbar_init(bYin, 1);
    mbar_init(bHready, 32 * kSsdEpiWarps);
    *abort = 0;
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

  if (warp == kSsdProducerWarp) {
    // ---------------- producer: C, B (two slots) and x of every chunk
    if (lane == 0) {
      for (int64_t c = 0; c < nchunks; ++c) {
        const int sl = (int)(c & 1);
        const int t0 = (int)(c * Q);
        const uint32_t uC = uS0 + sl * kSsdSlot, uB = uC + 2 * kSsdHalf;
        if (c >= 2 && !mbar_wait(bSlotFree + 8 * sl, (uint32_t)(((c - 2) >> 1) & 1), abort)) break;
        mbar_expect_tx(bFullCB + 8 * sl, 4 * kSsdHalf);
        for (int a = 0; a < 2; ++a) {
          tma_load3(uC + a * kSsdHalf, &p.tc, (int)(g * N + 64 * a), t0, (int)b, bFullCB + 8 * sl);
          tma_load3(uB + a * kSsdHalf, &p.tb, (int)(g * N + 64 * a), t0, (int)b, bFullCB + 8 * sl);
        }
        // x is single-buffered: free once the previous chunk's Y_dg is done
        if (c >= 1 && !mbar_wait(bMma2, (uint32_t)((c - 1) & 1), abort)) break;
        mbar_expect_tx(bFullX, kSsdHalf);
        tma_load3(uX, &p.tx, (int)(h * P), t0, (int)b, bFullX);
      }
    }
  } else if (warp == kSsdMmaWarp) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdCB = umma_idesc(128, 0, 0);
      constexpr uint32_t kIdY = umma_idesc(64, 0, 1);
      constexpr uint32_t kIdS = umma_idesc(64, 1, 1);
      // Three streams of products, each issued as soon as its inputs are ready
      // (tested without blocking), in chunk order within a stream:
      //   CB(c)      = C B^T      needs C, B of chunk c copied; its tensor-memory
      //                           buffer was read by M(c-2), so c <= (MMA2 issued) + 1
      //   Y_in(c)    = C H_c^T    needs H_c written (the epilogue of chunk c-1,
      //                           which has also read the accumulators reused here)
      //   Y_dg, S(c) = M X, B^T w.x  needs M, w.x and x of chunk c, and Y_in(c)
      //                           issued (so that the slot release covers it)
      // Y_in(0) exists only when the sequence starts from a given state; the
      // k-th Y_in issued waits for the k-th phase of bHready
      constexpr int64_t yin0 = HAS_H0 ? 0 : 1;
      int64_t ncb = 0, nyin = yin0, nmm = 0;  // next chunk of each stream
      long long idle = 0;
      while (nmm < nchunks) {
        bool progress = false;
        if (ncb < nchunks && ncb <= nmm + 1 &&
            mbar_test(bFullCB + 8 * (int)(ncb & 1), (uint32_t)((ncb >> 1) & 1))) {
          const int sl = (int)(ncb & 1);
          const uint32_t uC = uS0 + sl * kSsdSlot, uB = uC + 2 * kSsdHalf;
          tc_fence_after();
          for (int ks = 0; ks < N / 16; ++ks)
            umma(tm + sl * 128, umma_desc(kmajor_step(uC, ks), 16),
                 umma_desc(kmajor_step(uB, ks), 16), kIdCB, ks > 0);
          umma_commit(bCB + 8 * sl);
          ++ncb;
          progress = true;
        }
        if (nyin < nchunks && nyin <= nmm && nyin < ncb &&
            mbar_test(bHready, (uint32_t)((nyin - yin0) & 1))) {
          const uint32_t uC = uS0 + (int)(nyin & 1) * kSsdSlot;
          tc_fence_after();
          for (int ks = 0; ks < N / 16; ++ks)
            umma(tm + kTmYin, umma_desc(kmajor_step(uC, ks), 16), umma_desc(uH + ks * 2048, 16),
                 kIdY, ks > 0);
          umma_commit(bYin);
          ++nyin;
          progress = true;
        }
        if ((nmm < yin0 || nyin > nmm) && nmm < ncb && mbar_test(bMready, (uint32_t)(nmm & 1)) &&
            mbar_test(bFullX, (uint32_t)(nmm & 1))) {
          const int sl = (int)(nmm & 1);
          const uint32_t uB = uS0 + sl * kSsdSlot + 2 * kSsdHalf;
          tc_fence_after();
          for (int ks = 0; ks < Q / 16; ++ks) {
            umma(tm + kTmYdg, umma_desc(kmajor_step(uM, ks), 16), umma_desc(uX + ks * 2048, 16),
                 kIdY, ks > 0);
            umma(tm + kTmS, umma_desc(uB + ks * 2048, kSsdHalf), umma_desc(uW + ks * 2048, 16),
                 kIdS, ks > 0);
          }
          umma_commit(bMma2);
          umma_commit(bSlotFree + 8 * sl);  // C and B of this slot are read by now
          ++nmm;
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else if (*abort) {
          break;
        } else if (++idle > kSpinLimit * 4) {  // nothing became ready: give up
          *abort = 1;
          atomicOr(&g_ss_device_error, kErrTimeout);
          break;
        }
      }
    }
  } else if (warp >= kSsdPrepWarps) {
    // ---------------- epilogue warps 8-11 (row r, all columns)
    const uint32_t tlane = tm + ((uint32_t)(q4 * 32) << 16);  // this warp's lanes
    float hs[P];  // state row n = r: hs[p] = H[p][n]
    constexpr bool has_h0 = HAS_H0;
    auto store_h_copy = [&]() {  // bf16 copy of row n = r of H, the Y_in operand
#pragma unroll
      for (int j = 0; j < P / 8; ++j)
        *reinterpret_cast<uint4*>(sH + sw128(r, j)) =
            make_uint4(bf16x2(hs[j * 8 + 0], hs[j * 8 + 1]), bf16x2(hs[j * 8 + 2], hs[j * 8 + 3]),
                       bf16x2(hs[j * 8 + 4], hs[j * 8 + 5]), bf16x2(hs[j * 8 + 6], hs[j * 8 + 7]));
    };
    if constexpr (has_h0) {  // the given state enters as H of chunk 0 (phase 0 of bHready)
      const float* h0 = p.h0 + (b * H + h) * P * N;
#pragma unroll
      for (int i = 0; i < P; ++i) hs[i] = h0[i * N + r];
      store_h_copy();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bHready);
    } else {
#pragma unroll
      for (int i = 0; i < P; ++i) hs[i] = 0.f;
    }
    constexpr bool yin_c0 = has_h0;  // chunk 0 has a Y_in product
    bool ok = true;
    for (int64_t c = 0; c < nchunks; ++c) {
      const int64_t t0 = c * Q;
      const int len = (int)(L - t0 < Q ? L - t0 : Q);
      const int tb = (int)(c % 3);
      const float* cum = cum2 + tb * Q;
      // chunk c's tables, then Y_dg, S and Y_in of chunk c
      ok = ok && mbar_wait(bTFull + 8 * tb, (uint32_t)((c / 3) & 1), abort);
      const float decay = ok ? ex2(cum[Q - 1]) : 0.f;
      const float et = ok ? ex2(cum[r]) : 0.f;
      mbar_arrive(bTEmpty + 8 * tb);  // the table buffer is read
      ok = ok && mbar_wait(bMma2, (uint32_t)(c & 1), abort);
      const bool has_yin = c > 0 || yin_c0;
      if (ok && has_yin) ok = mbar_wait(bYin, (uint32_t)((c - (yin_c0 ? 0 : 1)) & 1), abort);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      if (ok) {
        {  // state (row n = r): H <- exp(cum_end) H + S^T, then its bf16 copy
          uint32_t sa[16], sb[16];  // the next 16 columns are read while these are used
          tmem_ld16_async(tlane + kTmS, sa);
#pragma unroll
          for (int q = 0; q < P / 16; ++q) {
            uint32_t(&sv)[16] = (q & 1) ? sb : sa;
            uint32_t(&sn)[16] = (q & 1) ? sa : sb;
            tmem_wait(sv);
            if (q + 1 < P / 16) tmem_ld16_async(tlane + kTmS + (q + 1) * 16, sn);
#pragma unroll
            for (int i = 0; i < 16; ++i) hs[q * 16 + i] = fmaf(decay, hs[q * 16 + i], fu(sv[i]));
          }
          store_h_copy();
        }
        // output (row t = r), 16 columns at a time: y = exp(cum_t) Y_in + Y_dg
        const int t = r;
        __nv_bfloat16* yrow = p.y + ((b * L + t0 + t) * H + h) * P;
#pragma unroll
        for (int q = 0; q < P / 16; ++q) {
          uint32_t yd[16], yi[16];
          tmem_ld16_async(tlane + kTmYdg + q * 16, yd);
          if (has_yin) tmem_ld16_async(tlane + kTmYin + q * 16, yi);
          tmem_wait(yd);
          if (has_yin) {
            tmem_wait(yi);
#pragma unroll
            for (int i = 0; i < 16; ++i) yd[i] = __float_as_uint(fmaf(et, fu(yi[i]), fu(yd[i])));
          }
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = bf16x2(fu(yd[2 * i]), fu(yd[2 * i + 1]));
          if (t < len) {
            *reinterpret_cast<uint4*>(yrow + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(yrow + q * 16 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        fence_async_smem();  // H's copy, for Y_in of the next chunk
        tc_fence_before();
        mbar_arrive(bHready);
      }
      if (bar_any<3, 32 * kSsdEpiWarps>(!ok || *abort)) {
        ok = false;
        break;
      }
    }
    if (ok && p.final_state) {
      float* fs = p.final_state + (b * H + h) * P * N;
#pragma unroll
      for (int i = 0; i < P; ++i) fs[i * N + r] = hs[i];
    }
  } else {
    // ---------------- prep warps 0-7
    const uint32_t tlane = tm + ((uint32_t)(q4 * 32) << 16);  // this warp's lanes
    const float A2 = p.A[h] * kLog2e;
    const float bias = p.bias ? p.bias[h] : 0.f;
    const float Dh = p.D ? p.D[h] : 0.f;

    bool ok = true;
    const unsigned short* dt_bits = reinterpret_cast<const unsigned short*>(p.dt);
    auto load_dt = [&](int64_t c) -> uint32_t {  // raw bf16 bits of chunk c's dt (warps 0-3)
      const int64_t t = c * Q + r;
      return (hf == 0 && t < L) ? (uint32_t)dt_bits[(b * L + t) * H + h] : 0u;
    };
    // decay sums, dt and block factors of chunk cc into table buf (warps 0-3,
    // row s = r): cum_s = sum_{r<=s} dt_r A log2e, and the factors of the
    // below-diagonal 32 x 32 blocks: exp2(cum_t - cum_s) = exp2(cum_t - cum_e)
    // exp2(cum_e - cum_s), e the block's last column; both exponents are <= 0
    // there (the decay only shrinks), so neither overflows
    auto scan_chunk = [&](int64_t cc, uint32_t bits, int buf) {
      // the buffer's previous chunk (cc - 3) must have been read by the epilogue
      if (cc >= 3) ok = mbar_wait(bTEmpty + 8 * buf, (uint32_t)(((cc - 3) / 3) & 1), abort) && ok;
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
      mbar_arrive(bTFull + 8 * buf);
    };

    if (hf == 0) scan_chunk(0, load_dt(0), 0);
    uint32_t dt_nxt = load_dt(1);  // dt is loaded a chunk before its tables are built
    asm volatile("bar.sync 2, 256;" ::: "memory");  // prep warps: tables of chunk 0
    // A wait that gives up only skips work: every prep warp still passes the
    // named barriers of the iteration, and all leave the loop together.
    for (int64_t c = 0; c < nchunks; ++c) {
      const int buf = (int)(c & 1);  // C.B^T buffer
      const int tb = (int)(c % 3);   // table buffer
      const float* cum = cum2 + tb * Q;
      const float* dts = dts2 + tb * Q;
      const float* gs = gs2 + tb * Q;

      // ---- M (row t = r) from CB: D on the diagonal, zero above it.  The two
      // warps of a lane quarter split every 32-column block in 16-column halves
      // (this warp: half hf of blocks 0..3), so the causal work is shared
      // evenly.  M's buffer is free once chunk c-1's products are done.
      ok = __all_sync(0xffffffffu, ok && mbar_wait(bCB + 8 * buf, (uint32_t)((c >> 1) & 1), abort));
      if (c > 0)
        ok = __all_sync(0xffffffffu, ok && mbar_wait(bMma2, (uint32_t)((c - 1) & 1), abort));
      tc_fence_after();
      if (ok) {
        const int t = r;
        const float ct = cum[t];
        const uint32_t tcb = tlane + buf * 128 + hf * 16;  // column 32 i + 16 hf of block i
        auto store8 = [&](int jb, const float (&m)[8]) {  // columns 8 jb .. 8 jb + 7
          *reinterpret_cast<uint4*>(sM + (jb >> 3) * kSsdHalf + sw128(t, jb & 7)) =
              make_uint4(bf16x2(m[0], m[1]), bf16x2(m[2], m[3]), bf16x2(m[4], m[5]),
                         bf16x2(m[6], m[7]));
        };
        // one 32-column block at a time; the loop is not unrolled, which keeps
        // this role's code small (measured: the unrolled form, a tensor-memory
        // read of the next block in flight, was 6% slower, the roles' code
        // contending for the instruction cache)
#pragma unroll 1
        for (int i = 0; i <= q4; ++i) {  // at and below the diagonal
          uint32_t cur[16];
          tmem_ld16_async(tcb + 32 * i, cur);
          tmem_wait(cur);
          const int s0 = 32 * i + 16 * hf;  // first column of this half
          if (i < q4) {  // below the diagonal: exp2(cum_t - cum_e) exp2(cum_e - cum_s) dt_s
            const float et = ex2(ct - cum[32 * i + 31]);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              float m[8], gv[8];
              *reinterpret_cast<float4*>(gv) = *reinterpret_cast<const float4*>(gs + s0 + 8 * kk);
              *reinterpret_cast<float4*>(gv + 4) =
                  *reinterpret_cast<const float4*>(gs + s0 + 8 * kk + 4);
#pragma unroll
              for (int e = 0; e < 8; ++e) m[e] = fu(cur[8 * kk + e]) * et * gv[e];
              store8(s0 / 8 + kk, m);
            }
          } else {  // the diagonal block: exp2(cum_t - cum_s) dt_s per element, masked
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              float m[8], cv[8], dv[8];
              const int sb = s0 + 8 * kk;
              *reinterpret_cast<float4*>(cv) = *reinterpret_cast<const float4*>(cum + sb);
              *reinterpret_cast<float4*>(cv + 4) = *reinterpret_cast<const float4*>(cum + sb + 4);
              *reinterpret_cast<float4*>(dv) = *reinterpret_cast<const float4*>(dts + sb);
              *reinterpret_cast<float4*>(dv + 4) = *reinterpret_cast<const float4*>(dts + sb + 4);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int sc = sb + e;
                const float v = fu(cur[8 * kk + e]) * ex2(ct - cv[e]) * dv[e];
                m[e] = sc < t ? v : (sc == t ? v + Dh : 0.f);
              }
              store8(sb / 8, m);
            }
          }
        }
#pragma unroll 1
        for (int i = q4 + 1; i < Q / 32; ++i) {  // above the diagonal
          const int s0 = 32 * i + 16 * hf;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            *reinterpret_cast<uint4*>(sM + ((s0 / 8 + kk) >> 3) * kSsdHalf +
                                      sw128(t, (s0 / 8 + kk) & 7)) = make_uint4(0, 0, 0, 0);
        }
      }
      // ---- w.x (row s = r, columns [32 hf, 32 hf + 32)) once x has arrived
      ok = __all_sync(0xffffffffu, ok && mbar_wait(bFullX, (uint32_t)(c & 1), abort));
      if (ok) {
        const int s = r;
        const float ws = ex2(cum[Q - 1] - cum[s]) * dts[s];
#pragma unroll
        for (int jj = 0; jj < P / 16; ++jj) {
          const int j = hf * (P / 16) + jj;
          const uint4 v = *reinterpret_cast<const uint4*>(sX + sw128(s, j));
          *reinterpret_cast<uint4*>(sW + sw128(s, j)) =
              make_uint4(bf16x2(bf_lo(v.x) * ws, bf_hi(v.x) * ws), bf16x2(bf_lo(v.y) * ws, bf_hi(v.y) * ws),
                         bf16x2(bf_lo(v.z) * ws, bf_hi(v.z) * ws), bf16x2(bf_lo(v.w) * ws, bf_hi(v.w) * ws));
        }
      }
      fence_async_smem();
      tc_fence_before();
      if (ok) mbar_arrive(bMready);

      // ---- the next chunk's tables
      if (hf == 0 && c + 1 < nchunks) scan_chunk(c + 1, dt_nxt, (int)((c + 1) % 3));
      dt_nxt = load_dt(c + 2);
      if (bar_any<2, 32 * kSsdPrepWarps>(!ok || *abort)) {
        ok = false;
        break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm),
                 "r"(kSsdTmemCols));
}

}  // namespace ss
