// Unit-throughput microbenchmarks for the roofline of the selective-scan
// forward kernel.
//
// The selective-scan update is bound by arithmetic issue rather than by a
// dense contraction, so the roofline needs three per-SM unit rates that the
// public specifications do not state for this part:
//   * MUFU ex2 results per clock per SM   (the decay exp(dt*A) of every update)
//   * FP32 FMA lane-ops per clock per SM  (scalar FFMA)
//   * FP32 FMA lane-ops per clock per SM  (packed f32x2 FFMA, sm_100 family)
// plus one probe of the update body itself with all operands on chip, which
// bounds what any kernel built around that body can reach.
//
// Each probe keeps several independent dependency chains per thread so that
// latency is hidden and the unit, not the chain, is the limit.  Clocks are
// measured inside the kernel (clock64 against globaltimer) so the per-clock
// figures are independent of whatever SM clock the part runs at.
//
// This file is built into its own shared library (libss_peaks.so); the
// selective-scan library does not link it.

#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>

namespace {

constexpr int kChains = 8;

struct ClockRec {
  unsigned long long clk0, clk1, ns0, ns1;
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void record_start(ClockRec* rec) {
  if (threadIdx.x == 0) {
    rec[blockIdx.x].clk0 = clock64();
    rec[blockIdx.x].ns0 = globaltimer_ns();
  }
}
__device__ __forceinline__ void record_end(ClockRec* rec) {
  __syncthreads();
  if (threadIdx.x == 0) {
    rec[blockIdx.x].clk1 = clock64();
    rec[blockIdx.x].ns1 = globaltimer_ns();
  }
}

// x <- 2^(-x) stays inside [0.5, 1] for x in [0, 1]: no overflow, no denormals.
__global__ void k_ex2(float* out, int iters, ClockRec* rec) {
  float x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) x[j] = 1e-3f * (threadIdx.x + 7 * j);
  __syncthreads();
  record_start(rec);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = ex2_approx(-x[j]);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += x[j];
  record_end(rec);
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// x <- x*a + b with |a| < 1 converges: the chains stay finite.
__global__ void k_ffma(float* out, int iters, float a, float b, ClockRec* rec) {
  float x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) x[j] = 1e-3f * (threadIdx.x + 7 * j);
  __syncthreads();
  record_start(rec);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = fmaf(x[j], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += x[j];
  record_end(rec);
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Same chains as k_ffma, two lanes-ops per instruction (fma.rn.f32x2).
__global__ void k_ffma2(float* out, int iters, float a, float b, ClockRec* rec) {
  unsigned long long x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j)
    x[j] = pack2(1e-3f * (threadIdx.x + 7 * j), 2e-3f * (threadIdx.x + 5 * j));
  const unsigned long long A = pack2(a, a), B = pack2(b, b);
  __syncthreads();
  record_start(rec);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j)
      asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[j]) : "l"(A), "l"(B));
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) {
    float lo, hi;
    unpack2(x[j], lo, hi);
    s += lo + hi;
  }
  record_end(rec);
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// The pipe mix of one state update with nothing else: per chain step two
// packed FFMA2 (the four FP32 lane-ops of an update on a state pair count as
// two instructions per update) and one MUFU ex2, in independent chains.  The
// rate it reaches is the ceiling of any kernel whose updates cost one ex2 and
// four FP32 lane-ops, before loads, row work or bookkeeping.
__global__ void k_mix(float* out, int iters, float a, float b, ClockRec* rec) {
  unsigned long long x[kChains], w[kChains];
  float e[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) {
    x[j] = pack2(1e-3f * (threadIdx.x + 7 * j), 2e-3f * (threadIdx.x + 5 * j));
    w[j] = pack2(3e-3f * (threadIdx.x + 3 * j), 4e-3f * (threadIdx.x + 2 * j));
    e[j] = 1e-3f * (threadIdx.x + 11 * j);
  }
  const unsigned long long A = pack2(a, a), B = pack2(b, b);
  __syncthreads();
  record_start(rec);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) {
      asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[j]) : "l"(A), "l"(B));
      asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(w[j]) : "l"(A), "l"(B));
      e[j] = ex2_approx(-e[j]);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) {
    float lo, hi, lo2, hi2;
    unpack2(x[j], lo, hi);
    unpack2(w[j], lo2, hi2);
    s += lo + hi + lo2 + hi2 + e[j];
  }
  record_end(rec);
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// The selective-scan update body with every operand on chip.  Per time step a
// thread owning one channel row and all 16 states does, for each state n,
//   a = 2^(dt*A2[n]); h[n] = a*h[n] + du*B[n]; y += C[n]*h[n]
// with dt, du and the B/C rows read from shared memory as the real kernel
// does.  kPacked = false: one row and all 16 states per thread, scalar FP32,
// `steps` time steps.  kPacked = true: the scan kernel's own layout (below),
// `steps` vectors of 8 time steps.
template <bool kPacked>
__global__ void k_update(float* out, int steps, ClockRec* rec) {
  constexpr int N = 16;
  constexpr int T = 64;
  __shared__ __align__(16) float sB[T][N];
  __shared__ __align__(16) float sC[T][N];
  __shared__ __align__(16) float sDt[T][32];
  __shared__ __align__(16) float sDu[T][32];
  for (int i = threadIdx.x; i < T * N; i += blockDim.x) {
    (&sB[0][0])[i] = 0.01f * ((i * 37) % 101) - 0.5f;
    (&sC[0][0])[i] = 0.01f * ((i * 53) % 97) - 0.5f;
  }
  for (int i = threadIdx.x; i < T * 32; i += blockDim.x) {
    (&sDt[0][0])[i] = 1e-3f + 1e-4f * (i % 89);
    (&sDu[0][0])[i] = 0.01f * ((i * 29) % 83) - 0.4f;
  }
  float A2[N];
#pragma unroll
  for (int n = 0; n < N; ++n) A2[n] = -1.4426950f * (n + 1);
  __syncthreads();
  record_start(rec);
  const int lane = threadIdx.x & 31;
  float ysum = 0.f;
  if (!kPacked) {
    float h[N];
#pragma unroll
    for (int n = 0; n < N; ++n) h[n] = 0.f;
    for (int s = 0; s < steps; ++s) {
      const int t = s & (T - 1);
      const float dt = sDt[t][lane];
      const float du = sDu[t][lane];
      float y = 0.f;
#pragma unroll
      for (int q = 0; q < N / 4; ++q) {
        const float4 b4 = *reinterpret_cast<const float4*>(&sB[t][4 * q]);
        const float4 c4 = *reinterpret_cast<const float4*>(&sC[t][4 * q]);
        const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
        const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int n = 4 * q + r;
          const float a = ex2_approx(dt * A2[n]);
          h[n] = fmaf(a, h[n], du * bb[r]);
          y = fmaf(cc[r], h[n], y);
        }
      }
      ysum += y;
    }
#pragma unroll
    for (int n = 0; n < N; ++n) ysum += h[n];
  } else {
    // the scan kernel's lane layout: two rows x 8 states per lane as f32x2
    // state pairs, dt/du of both rows per 8-step vector, B/C quads of the
    // lane's states per step, states outer and steps inner
    constexpr int V = 8, G = 8;
    const int nl0 = (threadIdx.x & 1) * G;
    unsigned long long h[2][G / 2], A2p[2][G / 2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int k = 0; k < G / 2; ++k) {
        h[r][k] = 0ull;
        A2p[r][k] = pack2(A2[nl0 + 2 * k] * (1 + r), A2[nl0 + 2 * k + 1] * (1 + r));
      }
    for (int j = 0; j < steps; ++j) {  // steps counts vectors of V steps here
      const int jt = (j & (T / V - 1)) * V;
      float dts[2][V], dus[2][V];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int q = 0; q < V; q += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(&sDt[jt + r][(lane & 3) * 8 + q]);
          const float4 b4 = *reinterpret_cast<const float4*>(&sDu[jt + r][(lane & 3) * 8 + q]);
          dts[r][q] = a4.x; dts[r][q + 1] = a4.y; dts[r][q + 2] = a4.z; dts[r][q + 3] = a4.w;
          dus[r][q] = b4.x; dus[r][q + 1] = b4.y; dus[r][q + 2] = b4.z; dus[r][q + 3] = b4.w;
        }
      unsigned long long yac[2][V];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) yac[r][v] = 0ull;
#pragma unroll
      for (int k4 = 0; k4 < G / 4; ++k4) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const ulonglong2 b4 = *reinterpret_cast<const ulonglong2*>(&sB[jt + v][nl0 + 4 * k4]);
          const ulonglong2 c4 = *reinterpret_cast<const ulonglong2*>(&sC[jt + v][nl0 + 4 * k4]);
          const unsigned long long bb[2] = {b4.x, b4.y};
          const unsigned long long cc[2] = {c4.x, c4.y};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = 2 * k4 + e;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              unsigned long long x2, c2;
              const unsigned long long dt2 = pack2(dts[r][v], dts[r][v]);
              const unsigned long long du2 = pack2(dus[r][v], dus[r][v]);
              asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(x2) : "l"(dt2), "l"(A2p[r][k]));
              float x0, x1;
              unpack2(x2, x0, x1);
              const unsigned long long a2 = pack2(ex2_approx(x0), ex2_approx(x1));
              asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(c2) : "l"(du2), "l"(bb[e]));
              asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(h[r][k]) : "l"(a2), "l"(c2));
              asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(yac[r][v]) : "l"(cc[e]), "l"(h[r][k]));
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) {
          float lo, hi;
          unpack2(yac[r][v], lo, hi);
          ysum += lo + hi;
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int k = 0; k < G / 2; ++k) {
        float lo, hi;
        unpack2(h[r][k], lo, hi);
        ysum += lo + hi;
      }
  }
  record_end(rec);
  out[blockIdx.x * blockDim.x + threadIdx.x] = ysum;
}

// Shared-memory loads as the scan kernel issues them for B and C: 16 bytes per
// lane.  MODE 0: every lane of a warp reads the same 16 bytes (a broadcast, as
// the B/C quads are); MODE 1: each lane its own 16 bytes, conflict-free; MODE
// 2: 4-byte broadcast loads, for comparison.  Eight independent loads per
// iteration, each folded into a running sum by one FADD.  Counts lane-loads.
template <int MODE>
__global__ void k_lds(float* out, int iters, ClockRec* rec) {
  __shared__ __align__(16) float buf[4096];
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) buf[i] = 1e-3f * (i % 97);
  const int lane = threadIdx.x & 31;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  __syncthreads();
  record_start(rec);
  for (int i = 0; i < iters; ++i) {
    const int base = (i * 256) & 4095;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (MODE == 2) {
        acc[j] += buf[(base + 4 * j) & 4095];
      } else {
        const int idx = MODE == 0 ? ((base + 32 * j) & 4095) : ((base + 128 * j + 4 * lane) & 4095);
        const float4 v = *reinterpret_cast<const float4*>(&buf[idx]);
        acc[j] += v.x + v.w;
      }
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += acc[j];
  record_end(rec);
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

// which: 0 = ex2, 1 = ffma, 2 = ffma2 (packed), 3 = update body scalar,
//        4 = update body packed, 5 = pipe mix of one update (2 FFMA2 + 1 ex2),
//        6 / 7 / 8 = 16-byte broadcast / 16-byte distinct / 4-byte broadcast
//        shared-memory loads (lane-loads).
// result[0] = lane-ops (or state updates) per second over the whole GPU
// result[1] = lane-ops (or updates) per clock per SM
// result[2] = mean SM clock during the run, MHz
// result[3] = number of SMs
// result[4] = elapsed milliseconds
// Returns 0 on success, a cudaError_t value otherwise.
extern "C" __attribute__((visibility("default"))) int ss_peaks_measure(int which, int iters, int blocks_per_sm, int threads,
                                double* result) {
  cudaDeviceProp prop;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return (int)e;
  const int sms = prop.multiProcessorCount;
  const int blocks = sms * blocks_per_sm;
  float* out = nullptr;
  ClockRec* rec = nullptr;
  e = cudaMalloc(&out, sizeof(float) * (size_t)blocks * threads);
  if (e != cudaSuccess) return (int)e;
  e = cudaMalloc(&rec, sizeof(ClockRec) * blocks);
  if (e != cudaSuccess) { cudaFree(out); return (int)e; }
  cudaEvent_t ev0, ev1;
  cudaEventCreate(&ev0);
  cudaEventCreate(&ev1);
  auto launch = [&]() {
    switch (which) {
      case 0: k_ex2<<<blocks, threads>>>(out, iters, rec); break;
      case 1: k_ffma<<<blocks, threads>>>(out, iters, 0.999f, 1e-3f, rec); break;
      case 2: k_ffma2<<<blocks, threads>>>(out, iters, 0.999f, 1e-3f, rec); break;
      case 3: k_update<false><<<blocks, threads>>>(out, iters, rec); break;
      case 4: k_update<true><<<blocks, threads>>>(out, iters, rec); break;
      case 5: k_mix<<<blocks, threads>>>(out, iters, 0.999f, 1e-3f, rec); break;
      case 6: k_lds<0><<<blocks, threads>>>(out, iters, rec); break;
      case 7: k_lds<1><<<blocks, threads>>>(out, iters, rec); break;
      case 8: k_lds<2><<<blocks, threads>>>(out, iters, rec); break;
      default: break;
    }
  };
  launch();  // warm-up
  cudaEventRecord(ev0);
  launch();
  cudaEventRecord(ev1);
  e = cudaEventSynchronize(ev1);
  if (e == cudaSuccess) e = cudaGetLastError();
  float ms = 0.f;
  cudaEventElapsedTime(&ms, ev0, ev1);
  ClockRec* h = new ClockRec[blocks];
  if (e == cudaSuccess) e = cudaMemcpy(h, rec, sizeof(ClockRec) * blocks, cudaMemcpyDeviceToHost);
  double mhz = 0.0;
  int cnt = 0;
  for (int i = 0; i < blocks; ++i) {
    const double dc = (double)(h[i].clk1 - h[i].clk0);
    const double dn = (double)(h[i].ns1 - h[i].ns0);
    if (dn > 0) { mhz += 1e3 * dc / dn; ++cnt; }
  }
  delete[] h;
  if (cnt) mhz /= cnt;
  double per_thread = 0.0;
  switch (which) {
    case 0: case 1: case 5: per_thread = (double)iters * kChains; break;
    case 2: per_thread = 2.0 * iters * kChains; break;
    case 3: per_thread = 16.0 * iters; break;
    case 4: per_thread = 128.0 * iters; break;  // iters vectors of 8 steps x 16 updates
    case 6: case 7: case 8: per_thread = 8.0 * iters; break;
    default: break;
  }
  const double total = per_thread * blocks * threads;
  const double per_s = total / (ms * 1e-3);
  result[0] = per_s;
  result[1] = (mhz > 0) ? per_s / (mhz * 1e6 * sms) : 0.0;
  result[2] = mhz;
  result[3] = sms;
  result[4] = ms;
  cudaEventDestroy(ev0);
  cudaEventDestroy(ev1);
  cudaFree(out);
  cudaFree(rec);
  return (int)e;
}
