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
// completed through an mbarrier; thread i of the CTA owns tensor-memory lane i
// (row t of CB and Y, row n of S).  Operands use the no-swizzle canonical
// layouts: 16-byte rows of 8 elements, a row block of 8 rows at 128 bytes, so
// a thread that owns a row writes one 16-byte chunk per 8 columns and a warp's
// chunks are contiguous.  B serves as the CB operand (K-major, K = n) and as
// the state product's A operand (MN-major, K = s) from the same bytes.
#pragma once

#include "ss_device.cuh"
#include "ss_sched.cuh"

namespace ss {

constexpr int kSsdQ = 128;  // steps per chunk (the MMA's M)
constexpr int kSsdP = 64;   // head dim
constexpr int kSsdN = 128;  // dstate
constexpr int kSsdThreads = 128;

// shared-memory map (bytes from the 1024-aligned dynamic base)
constexpr uint32_t kSsdOffC = 0;           // C [t][n] K-major, then M [t][s] K-major
constexpr uint32_t kSsdOffB = 32768;       // B [s][n]
constexpr uint32_t kSsdOffX = 65536;       // x [s][p] MN-major
constexpr uint32_t kSsdOffH = 81920;       // H [n][p] MN-major, then w.x [s][p]
constexpr uint32_t kSsdOffCum = 98304;     // cum [Q] fp32
constexpr uint32_t kSsdOffDt = 98816;      // dt [Q] fp32
constexpr uint32_t kSsdOffMisc = 99328;    // warp sums, mbarrier, tensor-memory address
constexpr uint32_t kSsdSmemBytes = 99328 + 64;
constexpr uint32_t kSsdTmemCols = 256;     // CB / S [0,128), Y_in [128,192), Y_dg [192,256)

struct SsdParams {
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

// Shared-memory matrix descriptor, no swizzle: start, leading-dimension byte
// offset (between 8-element blocks along K), stride byte offset (between
// 8-row blocks along M or N), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
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

// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 bytes global -> shared, zero-filled when !valid (the source is then not read).
__device__ __forceinline__ void cp_async16_zfill(uint32_t smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// grid = batch * nheads CTAs (one per (b, h)), block = 128, dynamic shared
// memory kSsdSmemBytes.  Requires P = 64, N = 128 and 16-byte aligned rows.
__global__ void __launch_bounds__(kSsdThreads, 2) ss_ssd_fwd(const SsdParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int Q = kSsdQ, P = kSsdP, N = kSsdN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t H = p.nheads, G = p.ngroups, L = p.seqlen;
  const int64_t b = blockIdx.x / H, h = blockIdx.x % H;
  const int64_t g = h / (H / G);

  unsigned char* sC = smem + kSsdOffC;
  unsigned char* sB = smem + kSsdOffB;
  unsigned char* sX = smem + kSsdOffX;
  unsigned char* sH = smem + kSsdOffH;
  float* cum = reinterpret_cast<float*>(smem + kSsdOffCum);
  float* dts = reinterpret_cast<float*>(smem + kSsdOffDt);
  float* wsum = reinterpret_cast<float*>(smem + kSsdOffMisc);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kSsdOffMisc + 32);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kSsdOffMisc + 48);
  const uint32_t uC = smem_u32(sC), uB = smem_u32(sB), uX = smem_u32(sX), uH = smem_u32(sH);
  const uint32_t ubar = smem_u32(bar);

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ubar));
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
  const uint32_t tlane = tm + ((uint32_t)(warp * 32) << 16);  // this warp's lanes

  const float A2 = p.A[h] * kLog2e;
  const float bias = p.bias ? p.bias[h] : 0.f;
  const float Dh = p.D ? p.D[h] : 0.f;
  float hs[P];  // state row n = tid: hs[p] = H[p][n]
#pragma unroll
  for (int i = 0; i < P; ++i) hs[i] = 0.f;

  constexpr uint32_t kIdCB = umma_idesc(128, 0, 0);
  constexpr uint32_t kIdY = umma_idesc(64, 0, 1);
  constexpr uint32_t kIdS = umma_idesc(64, 1, 1);
  uint32_t parity = 0;
  bool ok = true;
  const int64_t nchunks = (L + Q - 1) / Q;
  for (int64_t c = 0; c < nchunks && ok; ++c) {
    const int64_t t0 = c * Q;
    const int len = (int)(L - t0 < Q ? L - t0 : Q);
    const int s = tid;  // the row this thread stages: step t0 + s
    const bool valid = s < len;
    const int64_t tok = b * L + t0 + (valid ? s : 0);

    // ---- stage: x, B, C rows (zero past the end) and the in-chunk decay sums
    {
      const __nv_bfloat16* crow = p.C + (tok * G + g) * N;
      const __nv_bfloat16* brow = p.B + (tok * G + g) * N;
      const __nv_bfloat16* xrow = p.x + (tok * H + h) * P;
#pragma unroll
      for (int j = 0; j < N / 8; ++j) {
        cp_async16_zfill(uC + j * (Q * 16) + s * 16, crow + j * 8, valid);
        cp_async16_zfill(uB + j * (Q * 16) + s * 16, brow + j * 8, valid);
      }
#pragma unroll
      for (int j = 0; j < P / 8; ++j) cp_async16_zfill(uX + j * (Q * 16) + s * 16, xrow + j * 8, valid);
      cp_async_commit();
    }
    float dtv = 0.f;
    if (valid) {
      const float xdt = __bfloat162float(p.dt[tok * H + h]) + bias;
      dtv = p.softplus ? softplus(xdt) : xdt;
    }
    float run = dtv * A2;  // inclusive scan of dt*A*log2e over the chunk's steps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += v;
    }
    if (lane == 31) wsum[warp] = run;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (w < warp) run += wsum[w];
    cum[s] = run;
    dts[s] = dtv;
    cp_async_wait<0>();
    fence_async_smem();
    __syncthreads();

    // ---- CB = C B^T, Y_in = C H^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks)
        umma(tm + 0, umma_desc(uC + ks * 2 * (Q * 16), Q * 16, 128),
             umma_desc(uB + ks * 2 * (Q * 16), Q * 16, 128), kIdCB, ks > 0);
      if (c > 0) {
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
          umma(tm + 128, umma_desc(uC + ks * 2 * (Q * 16), Q * 16, 128),
               umma_desc(uH + ks * 2 * 128, 128, N / 8 * 128), kIdY, ks > 0);
      }
      umma_commit(ubar);
    }
    ok = __syncthreads_and(mbar_wait(ubar, parity));
    parity ^= 1;
    tc_fence_after();
    if (!ok) break;

    // ---- M from CB (row t = tid) into C's buffer; w.x (row s = tid) into H's
    {
      const int t = tid;
      const float ct = cum[t];
#pragma unroll
      for (int q = 0; q < Q / 32; ++q) {
        float cb[32];
        tmem_ld32(tlane + q * 32, cb);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int s0 = q * 32 + k * 8 + e;
            const float m0 = s0 <= t ? cb[k * 8 + e] * ex2(ct - cum[s0]) * dts[s0] : 0.f;
            const float m1 = s0 + 1 <= t ? cb[k * 8 + e + 1] * ex2(ct - cum[s0 + 1]) * dts[s0 + 1] : 0.f;
            w4[e / 2] = bf16x2(m0, m1);
          }
          *reinterpret_cast<uint4*>(sC + (q * 4 + k) * (Q * 16) + t * 16) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      const float ws = ex2(cum[Q - 1] - cum[s]) * dts[s];
#pragma unroll
      for (int j = 0; j < P / 8; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(sX + j * (Q * 16) + s * 16);
        *reinterpret_cast<uint4*>(sH + j * (Q * 16) + s * 16) =
            make_uint4(bf16x2(bf_lo(v.x) * ws, bf_hi(v.x) * ws), bf16x2(bf_lo(v.y) * ws, bf_hi(v.y) * ws),
                       bf16x2(bf_lo(v.z) * ws, bf_hi(v.z) * ws), bf16x2(bf_lo(v.w) * ws, bf_hi(v.w) * ws));
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- Y_dg = M X, S = B^T (w.x)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < Q / 16; ++ks) {
        umma(tm + 192, umma_desc(uC + ks * 2 * (Q * 16), Q * 16, 128),
             umma_desc(uX + ks * 2 * 128, 128, Q / 8 * 128), kIdY, ks > 0);
        umma(tm + 0, umma_desc(uB + ks * 2 * 128, 128, Q / 8 * 128),
             umma_desc(uH + ks * 2 * 128, 128, Q / 8 * 128), kIdS, ks > 0);
      }
      umma_commit(ubar);
    }
    ok = __syncthreads_and(mbar_wait(ubar, parity));
    parity ^= 1;
    tc_fence_after();
    if (!ok) break;

    // ---- state (row n = tid): H <- exp(cum_end) H + S^T, then its bf16 copy
    {
      const int n = tid;
      const float decay = ex2(cum[Q - 1]);
#pragma unroll
      for (int q = 0; q < P / 32; ++q) {
        float sv[32];
        tmem_ld32(tlane + q * 32, sv);
#pragma unroll
        for (int i = 0; i < 32; ++i) hs[q * 32 + i] = fmaf(decay, hs[q * 32 + i], sv[i]);
      }
#pragma unroll
      for (int j = 0; j < P / 8; ++j)
        *reinterpret_cast<uint4*>(sH + j * (N / 8 * 128) + n * 16) =
            make_uint4(bf16x2(hs[j * 8 + 0], hs[j * 8 + 1]), bf16x2(hs[j * 8 + 2], hs[j * 8 + 3]),
                       bf16x2(hs[j * 8 + 4], hs[j * 8 + 5]), bf16x2(hs[j * 8 + 6], hs[j * 8 + 7]));
    }
    // ---- output (row t = tid): y = exp(cum_t) Y_in + Y_dg + D x
    {
      const int t = tid;
      const float et = ex2(cum[t]);
      __nv_bfloat16* yrow = p.y + ((b * L + t0 + t) * H + h) * P;
#pragma unroll
      for (int q = 0; q < P / 32; ++q) {
        float yd[32], yi[32];
        tmem_ld32(tlane + 192 + q * 32, yd);
        if (c > 0) {
          tmem_ld32(tlane + 128 + q * 32, yi);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) yi[i] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = q * 4 + k;  // p block of 8
          const uint4 xv = *reinterpret_cast<const uint4*>(sX + j * (Q * 16) + t * 16);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i0 = k * 8 + 2 * e;
            const float y0 = fmaf(et, yi[i0], fmaf(Dh, bf_lo(xw[e]), yd[i0]));
            const float y1 = fmaf(et, yi[i0 + 1], fmaf(Dh, bf_hi(xw[e]), yd[i0 + 1]));
            o[e] = bf16x2(y0, y1);
          }
          if (t < len) *reinterpret_cast<uint4*>(yrow + j * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
  }

  if (ok && p.final_state) {
    float* fs = p.final_state + (b * H + h) * P * N;
#pragma unroll
    for (int i = 0; i < P; ++i) fs[i * N + tid] = hs[i];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm),
                 "r"(kSsdTmemCols));
}

}  // namespace ss
