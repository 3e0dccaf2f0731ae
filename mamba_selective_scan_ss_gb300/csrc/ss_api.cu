// C ABI of the selective-scan forward (declared in ss_selective_scan.h).
//
// Host side of one call: validate every argument (nothing is launched or
// written on error), pick the launch configuration from the sizes and the
// device, allocate stream-ordered scratch for chunk carries when the sequence
// is split, and enqueue the kernels on the caller's stream.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>

#include "ss_fwd.cuh"
#include "ss_selective_scan.h"

namespace {

constexpr int kThreads = 64;  // threads per CTA
constexpr int kRows = 2;      // channel rows per thread
constexpr int kMaxChunks = 1024;
constexpr int kStages = 4;    // depth of the per-thread u/delta/z copy ring

// Error word of the device-side waits (one per device context).
__device__ unsigned int g_ss_device_error = 0;

bool range_overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  if (!a || !b || a_bytes <= 0 || b_bytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }

struct Sizes {
  int64_t rows, x_elems, x_bytes, bc_bytes, a_elems, st_elems;
};

// Byte sizes of the operands; false if any of them overflows int64 (the fp32
// partial read-out of dstate > 16 is the largest: rows * seqlen * 4).
bool sizes_ok(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t elt,
              Sizes* s) {
  int64_t tmp, bc_elems;
  return mul_ok(batch, dim, &s->rows) && mul_ok(s->rows, seqlen, &s->x_elems) &&
         mul_ok(s->x_elems, elt, &s->x_bytes) && mul_ok(batch, dstate, &tmp) &&
         mul_ok(tmp, seqlen, &bc_elems) && mul_ok(bc_elems, elt, &s->bc_bytes) &&
         mul_ok(dim, dstate, &s->a_elems) && mul_ok(s->rows, dstate, &s->st_elems) &&
         mul_ok(s->x_elems, 4, &tmp) && mul_ok(s->rows, 256 * 1024 * 8, &tmp);
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

struct LaunchPlan {
  int nt;              // states per thread group (4, 8 or 16)
  int groups;          // state groups
  bool vec;            // 16-byte vector path
  int64_t dim_tiles;
  int64_t base_ctas;   // batch * dim_tiles
  int nchunks;
  int64_t chunk_len;
  int64_t agg_bytes, carry_bytes, part_bytes;  // scratch
  int launches;
};

// Number of sequence chunks: enough CTAs to fill the GPU about four CTAs deep,
// each chunk at least one B/C tile long.  SS_NCHUNKS overrides (tuning aid).
int choose_chunks(int64_t base_ctas, int64_t seqlen, int sms) {
  const int64_t max_by_len = std::max<int64_t>(1, seqlen / ss::kTileSteps);
  int64_t want = 1;
  if (const char* env = std::getenv("SS_NCHUNKS")) {
    want = std::atoll(env);
  } else {
    const int64_t target = (int64_t)std::max(sms, 1) * 4;
    want = (target + base_ctas - 1) / base_ctas;
  }
  want = std::max<int64_t>(1, std::min<int64_t>({want, max_by_len, kMaxChunks}));
  return (int)want;
}

// Launch plan shared by ss_selective_scan_fwd and ss_selective_scan_plan.
bool make_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t elt,
               bool aligned16, int sms, LaunchPlan* plan) {
  plan->nt = dstate <= 4 ? 4 : (dstate <= 8 ? 8 : 16);
  plan->groups = (int)((dstate + plan->nt - 1) / plan->nt);
  plan->vec = aligned16 && seqlen % (16 / elt) == 0;
  // rows per CTA: the vector kernel splits the states of a row pair over two
  // lanes when a group holds 8 or 16 states; the scalar kernel gives each
  // thread two rows with all their states
  const int64_t rows_per_cta = (plan->vec && plan->nt >= 8) ? kThreads : kThreads * kRows;
  plan->dim_tiles = (dim + rows_per_cta - 1) / rows_per_cta;
  if (plan->dim_tiles > INT_MAX / std::max<int64_t>(batch, 1)) return false;
  plan->base_ctas = batch * plan->dim_tiles;
  if (plan->base_ctas > INT_MAX) return false;
  plan->nchunks = choose_chunks(plan->base_ctas, seqlen, sms);
  const int64_t per = (seqlen + plan->nchunks - 1) / plan->nchunks;
  plan->chunk_len = (per + ss::kTileSteps - 1) / ss::kTileSteps * ss::kTileSteps;
  plan->nchunks = (int)((seqlen + plan->chunk_len - 1) / plan->chunk_len);
  const int64_t rows = batch * dim;
  const int64_t ns = (int64_t)plan->groups * plan->nt;
  plan->agg_bytes = 0;
  plan->carry_bytes = 0;
  plan->part_bytes = 0;
  if (plan->nchunks > 1) {
    plan->agg_bytes = (int64_t)(plan->nchunks - 1) * rows * ns * 8;
    plan->carry_bytes = (int64_t)plan->nchunks * rows * ns * 4;
  }
  if (plan->groups > 1) plan->part_bytes = rows * seqlen * 4;
  plan->launches = plan->groups + (plan->nchunks > 1 ? 2 : 0);
  return true;
}

template <typename T, int NT, bool VEC>
cudaError_t enqueue(ss::FwdParams p, const LaunchPlan& plan, cudaStream_t st) {
  constexpr int kTgs = NT >= 8 ? 2 : 1;  // lanes sharing a row pair
  const dim3 block(kThreads);
  if (plan.nchunks > 1) {
    const dim3 grid_agg((unsigned)plan.base_ctas, (unsigned)(plan.nchunks - 1),
                        (unsigned)plan.groups);
    if constexpr (VEC) {
      ss::ss_fwd_pipe<T, NT, kTgs, kThreads, kStages, true><<<grid_agg, block, 0, st>>>(p);
    } else {
      ss::ss_chunk_aggregate<T, NT, kRows, kThreads, false><<<grid_agg, block, 0, st>>>(p);
    }
    const int64_t n = p.batch * p.dim * p.ns;
    const unsigned cblocks = (unsigned)((n + 255) / 256);
    ss::ss_chunk_carry<<<cblocks, 256, 0, st>>>(p);
  }
  const dim3 grid((unsigned)plan.base_ctas, (unsigned)plan.nchunks);
  for (int g = 0; g < plan.groups; ++g) {
    p.group = g;
    p.accum_in = g > 0;
    p.final_group = g == plan.groups - 1;
    if constexpr (VEC) {
      ss::ss_fwd_pipe<T, NT, kTgs, kThreads, kStages, false><<<grid, block, 0, st>>>(p);
    } else {
      ss::ss_fwd_main<T, NT, kRows, kThreads, false><<<grid, block, 0, st>>>(p);
    }
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const ss::FwdParams& p, const LaunchPlan& plan, cudaStream_t st) {
  switch (plan.nt) {
    case 4: return plan.vec ? enqueue<T, 4, true>(p, plan, st) : enqueue<T, 4, false>(p, plan, st);
    case 8: return plan.vec ? enqueue<T, 8, true>(p, plan, st) : enqueue<T, 8, false>(p, plan, st);
    default: return plan.vec ? enqueue<T, 16, true>(p, plan, st) : enqueue<T, 16, false>(p, plan, st);
  }
}

}  // namespace

extern "C" {

SS_API const char* ss_status_string(ss_status_t status) {
  switch (status) {
    case SS_OK: return "SS_OK";
    case SS_ERR_INVALID_ARGUMENT: return "SS_ERR_INVALID_ARGUMENT";
    case SS_ERR_UNSUPPORTED: return "SS_ERR_UNSUPPORTED";
    case SS_ERR_CUDA: return "SS_ERR_CUDA";
    case SS_ERR_TIMEOUT: return "SS_ERR_TIMEOUT";
    default: return "SS_UNKNOWN_STATUS";
  }
}

SS_API ss_status_t ss_selective_scan_fwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  // ---- validation: nothing is enqueued or written on error ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !y) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;
  if (!sizes_ok(batch, dim, dstate, seqlen, elt, &sz)) return SS_ERR_UNSUPPORTED;
  const int64_t x_bytes = sz.x_bytes, bc_bytes = sz.bc_bytes, a_elems = sz.a_elems,
                st_elems = sz.st_elems;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) ||
      !aligned(y, ea) || (z && !aligned(z, ea)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (delta_bias && !aligned(delta_bias, 4)) || (last_state && !aligned(last_state, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  // outputs must not overlap any input, nor each other
  const void* ins[] = {u, delta, B, C, z, A, D, delta_bias};
  const int64_t in_bytes[] = {x_bytes, x_bytes, bc_bytes, bc_bytes, z ? x_bytes : 0,
                              a_elems * 4, D ? dim * 4 : 0, delta_bias ? dim * 4 : 0};
  for (int i = 0; i < 8; ++i) {
    if (range_overlap(y, x_bytes, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    if (last_state && range_overlap(last_state, st_elems * 4, ins[i], in_bytes[i]))
      return SS_ERR_INVALID_ARGUMENT;
  }
  if (last_state && range_overlap(last_state, st_elems * 4, y, x_bytes))
    return SS_ERR_INVALID_ARGUMENT;

  // ---- launch plan ----
  const int sms = sm_count();
  if (sms <= 0) return SS_ERR_CUDA;
  const bool aligned16 = aligned(u, 16) && aligned(delta, 16) && aligned(B, 16) &&
                         aligned(C, 16) && aligned(y, 16) && (!z || aligned(z, 16));
  LaunchPlan plan{};
  if (!make_plan(batch, dim, dstate, seqlen, elt, aligned16, sms, &plan))
    return SS_ERR_UNSUPPORTED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ss::FwdParams p{};
  p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.bias = delta_bias;
  p.y = y; p.last_state = last_state;
  p.batch = batch; p.dim = dim; p.dstate = dstate; p.seqlen = seqlen;
  p.chunk_len = plan.chunk_len;
  p.nchunks = plan.nchunks;
  p.ns = plan.groups * plan.nt;
  p.softplus = delta_softplus ? 1 : 0;

  // ---- stream-ordered scratch: chunk aggregates and carries, partial y ----
  const int64_t scratch_bytes = plan.agg_bytes + plan.carry_bytes + plan.part_bytes;
  void* scratch = nullptr;
  (void)cudaGetLastError();
  if (scratch_bytes > 0) {
    if (cudaMallocAsync(&scratch, (size_t)scratch_bytes, st) != cudaSuccess) return SS_ERR_CUDA;
    char* base = static_cast<char*>(scratch);
    if (plan.agg_bytes) p.agg = reinterpret_cast<float2*>(base);
    if (plan.carry_bytes) p.carry = reinterpret_cast<float*>(base + plan.agg_bytes);
    if (plan.part_bytes)
      p.y_partial = reinterpret_cast<float*>(base + plan.agg_bytes + plan.carry_bytes);
  }

  const cudaError_t err = dtype == SS_F32 ? dispatch<float>(p, plan, st)
                                          : dispatch<__nv_bfloat16>(p, plan, st);
  if (scratch) {
    const cudaError_t ferr = cudaFreeAsync(scratch, st);
    if (err == cudaSuccess && ferr != cudaSuccess) return SS_ERR_CUDA;
  }
  return err == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

SS_API ss_status_t ss_selective_scan_plan(int64_t batch, int64_t dim, int64_t dstate,
                                          int64_t seqlen, ss_dtype_t dtype, int aligned16,
                                          int sm_count, ss_plan_t* out) {
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!out || batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0 || sm_count <= 0)
    return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;
  if (!sizes_ok(batch, dim, dstate, seqlen, elt, &sz)) return SS_ERR_UNSUPPORTED;
  LaunchPlan plan{};
  if (!make_plan(batch, dim, dstate, seqlen, elt, aligned16 != 0, sm_count, &plan))
    return SS_ERR_UNSUPPORTED;
  out->nchunks = plan.nchunks;
  out->chunk_len = plan.chunk_len;
  out->state_groups = plan.groups;
  out->ctas = plan.base_ctas * plan.nchunks;
  out->kernel_launches = plan.launches;
  out->scratch_bytes = plan.agg_bytes + plan.carry_bytes + plan.part_bytes;
  out->vector_path = plan.vec ? 1 : 0;
  return SS_OK;
}

SS_API ss_status_t ss_selective_scan_check(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SS_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_ss_device_error, sizeof(word)) != cudaSuccess)
    return SS_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_ss_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return SS_ERR_CUDA;
    return SS_ERR_TIMEOUT;
  }
  return SS_OK;
}

}  // extern "C"
