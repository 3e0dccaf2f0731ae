// C ABI of the selective-scan forward (declared in ss_selective_scan.h).
//
// Host side of one call: validate every argument (nothing is launched or
// written on error), pick the launch configuration from the sizes and the
// device, allocate stream-ordered scratch for chunk carries when the sequence
// is split, and enqueue the kernels on the caller's stream.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <utility>

#include "ss_bwd.cuh"
#include "ss_decode.cuh"
#include "ss_layout.cuh"
#include "ss_pc.cuh"
#include "ss_sched.cuh"
#include "ss_selective_scan.h"
#include "ss_ssd.cuh"

namespace {

constexpr int kThreads = 64;  // threads per CTA
constexpr int kRows = 2;      // channel rows per thread
constexpr int kMaxChunks = 1024;
// depth of the per-thread u/delta/z copy ring (16-byte vectors in flight): fp32
// workloads run at one or two warps per scheduler and need the deeper ring to
// cover HBM latency (measured: 6 beats 4 and 8 on the fp32 sequence sweep);
// bf16 vectors hold twice the steps, and 4 is best there
template <typename T>
constexpr int kStages = sizeof(T) == 4 ? 6 : 4;
// CTAs per SM the scheduled kernel's plan is sized for.  The fp32
// segment-stream instantiations (8 or 16 states, 58-67 KB of shared memory)
// fit three times in an SM; the plan still counts four: the CTAs past the
// resident ones start when tickets run out and leave at once, every wait is
// for a unit handed out earlier to a running CTA, and on the decoupled
// Mamba-130M layer that plan measured 0.088 ms against 0.100 ms when sized for
// three.
constexpr int kCtasPerSm = 4;
static_assert(3 * (ss::fwd_sched_dyn_smem<float, 16, 2, kThreads, kStages<float>>() + 2048) <=
                  227 * 1024,
              "three fp32 segment-stream CTAs per SM");

bool range_overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  if (!a || !b || a_bytes <= 0 || b_bytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A TMA descriptor of a bf16 tensor [d2][d1][d0] (d0 contiguous) read in boxes
// of 64 x 128 x 1 elements, 128-byte swizzled; elements past d1 read as zero.
bool tma_map_rows(CUtensorMap* map, const void* base, int64_t d0, int64_t d1, int64_t d2) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!encode) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  const cuuint64_t strides[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)(d0 * d1) * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
  int tgs;             // vector path: lanes sharing a row pair
  int groups;          // state groups
  bool vec;            // 16-byte vector path (scheduled kernel)
  int64_t rows_per_cta;
  int64_t dim_tiles;
  int64_t tiles;       // batch * dim_tiles
  int nchunks;
  int64_t chunk_len;
  int64_t grid;        // CTAs of each main launch
  int64_t slots;       // vector path: CTAs the schedule is sized for
  bool chained;        // scheduled kernel: chained (true) or decoupled units
  // scratch (bytes)
  int64_t sched_bytes_per_group;  // ticket + unit flags (zeroed per call)
  int64_t sched_bytes, unit_agg_bytes, unit_incl_bytes;     // vector path
  int64_t agg_bytes, carry_bytes;                           // scalar path
  int64_t part_bytes;                                       // dstate > 16
  int launches;
};

// Tuning and fault-injection knobs exist only in the test build of the
// library (compiled with SS_TEST_HOOKS, loaded by the tests that need them);
// the shipped library reads no environment variable.
#ifdef SS_TEST_HOOKS
int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : fallback;
}
#define SS_TUNING(name, fallback) env_int(name, fallback)
#else
#define SS_TUNING(name, fallback) (fallback)
#endif

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Speed of one warp of the scan kernel relative to a warp alone on its
// scheduler, against the warps sharing the scheduler: the SM's throughput
// grows by half from one to two warps per scheduler and little beyond
// (fitted to the kernel's measured times on GB300 for several chunk counts
// of the decoupled workloads).
double warp_speed(double w) {
  if (w <= 1.0) return 1.0;
  const double sm_rate = w <= 2.0 ? 1.0 + 0.5 * (w - 1.0)
                                  : (w <= 8.0 ? 1.5 + 0.025 * (w - 2.0) : 1.65);
  return sm_rate / w;
}

// Estimated duration, in step-times of a lone warp, of a decoupled launch with
// chunks of len steps: units run in rounds of at most `slots` CTAs; a unit of
// a split row makes two passes over its chunk (aggregate, then main), a whole
// row one; each unit also pays a fixed cost (look-back, pipeline fill) of
// kUnitOverheadSteps.
constexpr double kUnitOverheadSteps = 64.0;
double decoupled_makespan(int64_t tiles, int64_t seqlen, int64_t len, int64_t slots, int64_t nsm) {
  const int64_t n = (seqlen + len - 1) / len;
  const int64_t units = tiles * n;
  const double unit_steps = (n > 1 ? 2.0 : 1.0) * (double)len + kUnitOverheadSteps;
  const double warps_per_cta = kThreads / 32.0;
  auto round_time = [&](int64_t ctas) {
    const double w = (double)ctas / (double)nsm * warps_per_cta / 4.0;
    return unit_steps / warp_speed(w);
  };
  const int64_t full = units / slots, last = units % slots;
  return (double)full * round_time(slots) + (last > 0 ? round_time(last) : 0.0);
}

// Launch plan shared by ss_selective_scan_fwd and ss_selective_scan_plan.
//
// Vector path: one persistent kernel per state group with sms * ctas_per_sm
// CTAs taking (row tile, chunk) units.  With at least as many row tiles as
// CTAs, chunks are chained and cost nothing extra; they only give the
// dynamic balance (about eight units per CTA).  With fewer row tiles than
// CTAs the split over time is what provides the parallelism, at the cost of
// an aggregate pass in each decoupled unit; the chunk length is the one that
// minimises decoupled_makespan.
// Scalar path: aggregate, carry and main kernels over a fixed chunk grid.
// In the test build SS_NCHUNKS and SS_CTAS_PER_SM override the heuristics, so
// that the tests can force every scheduling mode and chunk shape.
bool make_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t elt,
               bool aligned16, int sms, LaunchPlan* plan) {
  plan->nt = dstate <= 4 ? 4 : (dstate <= 8 ? 8 : 16);
  plan->groups = (int)((dstate + plan->nt - 1) / plan->nt);
  plan->vec = aligned16 && seqlen % (16 / elt) == 0;
  // lanes sharing a row pair on the vector path: two for 8 or 16 states, one for 4
  plan->tgs = plan->nt >= 8 ? 2 : 1;
  plan->rows_per_cta = plan->vec ? 2 * kThreads / plan->tgs : kThreads * kRows;
  plan->dim_tiles = (dim + plan->rows_per_cta - 1) / plan->rows_per_cta;
  if (plan->dim_tiles > INT_MAX / std::max<int64_t>(batch, 1)) return false;
  plan->tiles = batch * plan->dim_tiles;
  const int64_t rows = batch * dim;
  const int64_t ns = (int64_t)plan->groups * plan->nt;
  const int env_chunks = SS_TUNING("SS_NCHUNKS", 0);
  plan->sched_bytes_per_group = plan->sched_bytes = plan->unit_agg_bytes = 0;
  plan->unit_incl_bytes = plan->agg_bytes = plan->carry_bytes = plan->part_bytes = 0;
  int64_t want;
  if (plan->vec) {
    const int64_t cap = std::max(1, SS_TUNING("SS_CTAS_PER_SM", kCtasPerSm));
    const int64_t nsm = std::max(sms, 1);
    // chained chunks need at least as many row tiles as CTAs: take the largest
    // residency (at most cap CTAs per SM) that allows it
    const int64_t chain_per_sm = std::min<int64_t>(cap, plan->tiles / nsm);
    int64_t slots = nsm * cap;
    if (env_chunks > 0) {
      want = env_chunks;
    } else if (chain_per_sm >= 2 && seqlen >= 512) {
      slots = nsm * chain_per_sm;
      want = std::min<int64_t>((8 * slots + plan->tiles - 1) / plan->tiles, seqlen / 256);
    } else {
      // decoupled (or one wave of whole rows): the shortest estimated makespan
      const int64_t max_n = std::max<int64_t>(1, std::min<int64_t>(seqlen / ss::kTileSteps, kMaxChunks));
      double best = 0.0;
      want = 1;
      for (int64_t n = 1; n <= max_n; ++n) {
        const int64_t len = round_up((seqlen + n - 1) / n, ss::kTileSteps);
        if ((seqlen + len - 1) / len != n) continue;  // same chunks as a smaller n
        const double t = decoupled_makespan(plan->tiles, seqlen, len, slots, nsm);
        if (n == 1 || t < best) {
          best = t;
          want = n;
        }
      }
    }
    plan->slots = slots;
    want = std::max<int64_t>(1, std::min<int64_t>({want, seqlen / ss::kTileSteps, kMaxChunks}));
    plan->chunk_len = round_up((seqlen + want - 1) / want, ss::kTileSteps);
    plan->nchunks = (int)((seqlen + plan->chunk_len - 1) / plan->chunk_len);
    plan->grid = std::min<int64_t>(plan->tiles * plan->nchunks, slots);
    plan->chained = plan->tiles >= plan->grid;
    if (plan->grid > INT_MAX) return false;
    plan->sched_bytes_per_group = round_up(128 + plan->nchunks * plan->tiles * 4, 256);
    plan->sched_bytes = plan->sched_bytes_per_group * plan->groups;
    const int64_t rec = (int64_t)plan->nchunks * plan->tiles * plan->rows_per_cta * plan->nt;
    plan->unit_agg_bytes = round_up(rec * 8, 256);
    plan->unit_incl_bytes = round_up(rec * 4, 256);
    plan->launches = plan->groups;
  } else {
    if (env_chunks > 0) {
      want = env_chunks;
    } else {
      const int64_t target = (int64_t)std::max(sms, 1) * 4;
      want = (target + plan->tiles - 1) / plan->tiles;
    }
    want = std::max<int64_t>(1, std::min<int64_t>({want, std::max<int64_t>(1, seqlen / ss::kTileSteps),
                                                   kMaxChunks}));
    plan->chunk_len = round_up((seqlen + want - 1) / want, ss::kTileSteps);
    plan->nchunks = (int)((seqlen + plan->chunk_len - 1) / plan->chunk_len);
    plan->grid = plan->tiles * plan->nchunks;
    if (plan->nchunks > 1) {
      plan->agg_bytes = (int64_t)(plan->nchunks - 1) * rows * ns * 8;
      plan->carry_bytes = (int64_t)plan->nchunks * rows * ns * 4;
    }
    plan->launches = plan->groups + (plan->nchunks > 1 ? 2 : 0);
  }
  if (plan->groups > 1) plan->part_bytes = round_up(rows * seqlen * 4, 256);
  return true;
}

int64_t scratch_bytes(const LaunchPlan& plan) {
  return plan.sched_bytes + plan.unit_agg_bytes + plan.unit_incl_bytes + plan.agg_bytes +
         plan.carry_bytes + plan.part_bytes;
}

template <typename T, int NT, int TGS, bool HAS_Z, bool MULTI>
cudaError_t enqueue_vec(ss::FwdParams p, const LaunchPlan& plan, cudaStream_t st) {
  auto kernel = ss::ss_fwd_sched<T, NT, TGS, kThreads, kStages<T>, HAS_Z, MULTI>;
  constexpr int dyn = ss::fwd_sched_dyn_smem<T, NT, TGS, kThreads, kStages<T>>();
  if constexpr (dyn > 0) {
    // once per instantiation (and device context of the first call)
    static const cudaError_t attr =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (attr != cudaSuccess) return attr;
  }
  char* sched = reinterpret_cast<char*>(p.ticket);
  for (int g = 0; g < plan.groups; ++g) {
    p.group = g;
    p.accum_in = g > 0;
    p.final_group = g == plan.groups - 1;
    p.ticket = reinterpret_cast<unsigned*>(sched + g * plan.sched_bytes_per_group);
    p.flags = p.ticket + 32;
    kernel<<<(unsigned)plan.grid, kThreads, dyn, st>>>(p);
  }
  return cudaGetLastError();
}

template <typename T, int NT, int TGS>
cudaError_t enqueue_vec_flags(const ss::FwdParams& p, const LaunchPlan& plan, cudaStream_t st) {
  const bool has_z = p.z != nullptr;
  if (plan.groups > 1)
    return has_z ? enqueue_vec<T, NT, TGS, true, true>(p, plan, st)
                 : enqueue_vec<T, NT, TGS, false, true>(p, plan, st);
  return has_z ? enqueue_vec<T, NT, TGS, true, false>(p, plan, st)
               : enqueue_vec<T, NT, TGS, false, false>(p, plan, st);
}

template <typename T, int NT>
cudaError_t enqueue_scalar(ss::FwdParams p, const LaunchPlan& plan, cudaStream_t st) {
  const dim3 block(kThreads);
  if (plan.nchunks > 1) {
    const dim3 grid_agg((unsigned)plan.tiles, (unsigned)(plan.nchunks - 1),
                        (unsigned)plan.groups);
    ss::ss_chunk_aggregate<T, NT, kRows, kThreads, false><<<grid_agg, block, 0, st>>>(p);
    const int64_t n = p.batch * p.dim * p.ns;
    ss::ss_chunk_carry<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p);
  }
  const dim3 grid((unsigned)plan.tiles, (unsigned)plan.nchunks);
  for (int g = 0; g < plan.groups; ++g) {
    p.group = g;
    p.accum_in = g > 0;
    p.final_group = g == plan.groups - 1;
    ss::ss_fwd_main<T, NT, kRows, kThreads, false><<<grid, block, 0, st>>>(p);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const ss::FwdParams& p, const LaunchPlan& plan, cudaStream_t st) {
  if (plan.vec) {
    switch (plan.nt) {
      case 4: return enqueue_vec_flags<T, 4, 1>(p, plan, st);
      case 8: return enqueue_vec_flags<T, 8, 2>(p, plan, st);
      default: return enqueue_vec_flags<T, 16, 2>(p, plan, st);
    }
  }
  switch (plan.nt) {
    case 4: return enqueue_scalar<T, 4>(p, plan, st);
    case 8: return enqueue_scalar<T, 8>(p, plan, st);
    default: return enqueue_scalar<T, 16>(p, plan, st);
  }
}

// The per-channel kernel for the given gate, vector-path and row-width choices.
// One CTA per SM (registers), so a launch is ceil(CTAs / SMs) waves whose
// length is set by the row work per CTA.  Rows of up to 32 lanes take CTAs of
// 7 warps instead of 8 when that costs no extra wave: less work per wave for
// the same count (measured on 8 x 5120 rows of 16 states: 5 waves either way,
// 0.441 against 0.457 ms; 6 or 5 warps per CTA were slower, 0.493 / 0.560).
template <typename T>
void pc_launch(const ss::PcParams& p, bool has_z, bool vec, int sms, cudaStream_t st) {
  const bool wide = p.seg_shift > 5;
  const int64_t threads = p.rows << p.seg_shift;
  const int64_t nsm = std::max(sms, 1);
  auto waves = [&](int64_t block) { return ((threads + block - 1) / block + nsm - 1) / nsm; };
  const int block = (!wide && waves(224) <= waves(256)) ? 224 : 256;
  const unsigned grid = (unsigned)((threads + block - 1) / block);
  auto go = [&](auto z, auto v, auto w) {
    ss::ss_fwd_pc<T, decltype(z)::value, decltype(v)::value, decltype(w)::value>
        <<<grid, block, 0, st>>>(p);
  };
  using F = std::false_type;
  using U = std::true_type;
  if (wide) {
    if (has_z) vec ? go(U{}, U{}, U{}) : go(U{}, F{}, U{});
    else vec ? go(F{}, U{}, U{}) : go(F{}, F{}, U{});
  } else {
    if (has_z) vec ? go(U{}, U{}, F{}) : go(U{}, F{}, F{});
    else vec ? go(F{}, U{}, F{}) : go(F{}, F{}, F{});
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
    case SS_ERR_SCRATCH_LIMIT: return "SS_ERR_SCRATCH_LIMIT";
    default: return "SS_UNKNOWN_STATUS";
  }
}

}  // extern "C"

namespace {

// The forward from an initial state h0 (null: zero); both forward entry
// points land here.
ss_status_t fwd_impl(const void* u, const void* delta, const float* A, const void* B,
                     const void* C, const float* D, const void* z, const float* delta_bias,
                     int delta_softplus, const float* h0, void* y, float* last_state,
                     int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                     ss_dtype_t dtype, void* stream);

constexpr int64_t kPadMinElems = 1 << 16;  // rows x steps below which ragged calls stay scalar
constexpr int64_t kHostPieces = 8;           // host-buffer calls: pieces (batch slices or segments)
constexpr int64_t kHostSegmentSteps = 4096;  // ... and steps per segment of a single sequence

// The forward of ragged rows through padded copies (see fwd_impl): u, delta,
// z, B and C copied into rows of seqlen rounded up to the vector, in
// stream-ordered scratch, the vector path run on them, and y copied back;
// last_state is the padded run's own (the padding leaves the state as it is).
ss_status_t fwd_padded(const void* u, const void* delta, const float* A, const void* B,
                       const void* C, const float* D, const void* z, const float* delta_bias,
                       int delta_softplus, const float* h0, void* y, float* last_state,
                       int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                       ss_dtype_t dtype, cudaStream_t st) {
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  const int64_t Lp = round_up(seqlen, 16 / elt);
  const int64_t rows = batch * dim, bc_rows = batch * dstate;
  const int64_t x_bytes = round_up(rows * Lp * elt, 256), bc_bytes = round_up(bc_rows * Lp * elt, 256);
  const int64_t total = (z ? 4 : 3) * x_bytes + 2 * bc_bytes;
  (void)cudaGetLastError();
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, (size_t)total, st) != cudaSuccess) return SS_ERR_CUDA;
  char* q = static_cast<char*>(scratch);
  char* up = q;               q += x_bytes;
  char* dp = q;               q += x_bytes;
  char* yp = q;               q += x_bytes;
  char* Bp = q;               q += bc_bytes;
  char* Cp = q;               q += bc_bytes;
  char* zp = z ? q : nullptr;
  const float neg_inf = -__builtin_huge_valf();
  const int64_t vecs = Lp / (16 / elt);
  auto grid_of = [&](int64_t nrows, int64_t nv) {
    return dim3((unsigned)std::min<int64_t>((nv + 255) / 256, 64),
                (unsigned)std::min<int64_t>(nrows, 65535));
  };
  auto pad = [&](const void* in, void* out, int64_t nrows, float fill, const float* neg_of) {
    const dim3 grid = grid_of(nrows, vecs);
    if (elt == 4)
      ss::ss_pad_rows<float><<<grid, 256, 0, st>>>(static_cast<const float*>(in),
                                                   static_cast<float*>(out), nrows, seqlen, Lp,
                                                   fill, neg_of, dim);
    else
      ss::ss_pad_rows<__nv_bfloat16><<<grid, 256, 0, st>>>(
          static_cast<const __nv_bfloat16*>(in), static_cast<__nv_bfloat16*>(out), nrows, seqlen,
          Lp, fill, neg_of, dim);
  };
  pad(u, up, rows, 0.f, nullptr);
  pad(delta, dp, rows, delta_softplus ? neg_inf : 0.f, delta_softplus ? nullptr : delta_bias);
  if (z) pad(z, zp, rows, 0.f, nullptr);
  pad(B, Bp, bc_rows, 0.f, nullptr);
  pad(C, Cp, bc_rows, 0.f, nullptr);
  ss_status_t status = cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  if (status == SS_OK)
    status = fwd_impl(up, dp, A, Bp, Cp, D, zp, delta_bias, delta_softplus, h0, yp, last_state,
                      batch, dim, dstate, Lp, dtype, st);
  if (status == SS_OK) {
    const dim3 grid = grid_of(rows, (seqlen + 16 / elt - 1) / (16 / elt));
    if (elt == 4)
      ss::ss_unpad_rows<float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(yp),
                                                     static_cast<float*>(y), rows, seqlen, Lp);
    else
      ss::ss_unpad_rows<__nv_bfloat16><<<grid, 256, 0, st>>>(
          reinterpret_cast<const __nv_bfloat16*>(yp), static_cast<__nv_bfloat16*>(y), rows,
          seqlen, Lp);
    if (cudaGetLastError() != cudaSuccess) status = SS_ERR_CUDA;
  }
  if (cudaFreeAsync(scratch, st) != cudaSuccess && status == SS_OK) status = SS_ERR_CUDA;
  return status;
}

ss_status_t fwd_impl(const void* u, const void* delta, const float* A, const void* B,
                     const void* C, const float* D, const void* z, const float* delta_bias,
                     int delta_softplus, const float* h0, void* y, float* last_state,
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
      (delta_bias && !aligned(delta_bias, 4)) || (last_state && !aligned(last_state, 4)) ||
      (h0 && !aligned(h0, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  // outputs must not overlap any input, nor each other; last_state may be h0
  // itself (the state updated in place)
  const void* ins[] = {u, delta, B, C, z, A, D, delta_bias, h0};
  const int64_t in_bytes[] = {x_bytes, x_bytes, bc_bytes, bc_bytes, z ? x_bytes : 0,
                              a_elems * 4, D ? dim * 4 : 0, delta_bias ? dim * 4 : 0,
                              h0 ? st_elems * 4 : 0};
  for (int i = 0; i < 9; ++i) {
    if (range_overlap(y, x_bytes, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    const bool in_place = i == 8 && last_state == h0;
    if (last_state && !in_place && range_overlap(last_state, st_elems * 4, ins[i], in_bytes[i]))
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
  // Ragged rows (seqlen not a multiple of the 16-byte vector, or unaligned
  // buffers): the vector path on padded copies is several times faster than
  // the scalar path, and exact when the padding leaves the state unchanged:
  // dt = 0 there (delta -inf under the softplus, else -bias, which is exact in
  // fp32), u = B = C = 0.  Small calls stay on the scalar path.
  if (!plan.vec && batch * dim * seqlen >= kPadMinElems &&
      (delta_softplus || dtype == SS_F32 || !delta_bias) && SS_TUNING("SS_NO_PAD", 0) == 0)
    return fwd_padded(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, last_state,
                      batch, dim, dstate, seqlen, dtype, st);

  ss::FwdParams p{};
  p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.bias = delta_bias;
  p.h0 = h0;
  p.y = y; p.last_state = last_state;
  p.batch = batch; p.dim = dim; p.dstate = dstate; p.seqlen = seqlen;
  p.chunk_len = plan.chunk_len;
  p.nchunks = plan.nchunks;
  p.ns = plan.groups * plan.nt;
  p.softplus = delta_softplus ? 1 : 0;

  // ---- stream-ordered scratch: schedule, unit records or chunk carries, partial y ----
  const int64_t total_scratch = scratch_bytes(plan);
  void* scratch = nullptr;
  (void)cudaGetLastError();
  if (total_scratch > 0) {
    if (cudaMallocAsync(&scratch, (size_t)total_scratch, st) != cudaSuccess) return SS_ERR_CUDA;
    char* base = static_cast<char*>(scratch);
    if (plan.sched_bytes) {
      if (cudaMemsetAsync(base, 0, (size_t)plan.sched_bytes, st) != cudaSuccess) {
        cudaFreeAsync(scratch, st);
        return SS_ERR_CUDA;
      }
      p.ticket = reinterpret_cast<unsigned*>(base);
#ifdef SS_TEST_HOOKS
      // test hook: the first SS_TEST_SKIP_UNITS units of every launch are
      // never handed out, so their successors' bounded waits run out
      const int skip = env_int("SS_TEST_SKIP_UNITS", 0);
      if (skip > 0) {
        for (int g = 0; g < plan.groups; ++g)
          ss::ss_set_ticket<<<1, 1, 0, st>>>(
              reinterpret_cast<unsigned*>(base + g * plan.sched_bytes_per_group), (unsigned)skip);
        if (cudaGetLastError() != cudaSuccess) {
          cudaFreeAsync(scratch, st);
          return SS_ERR_CUDA;
        }
      }
#endif
      base += plan.sched_bytes;
    }
    if (plan.unit_agg_bytes) {
      p.unit_agg = reinterpret_cast<float2*>(base);
      base += plan.unit_agg_bytes;
      p.unit_incl = reinterpret_cast<float*>(base);
      base += plan.unit_incl_bytes;
    }
    if (plan.agg_bytes) {
      p.agg = reinterpret_cast<float2*>(base);
      base += plan.agg_bytes;
      p.carry = reinterpret_cast<float*>(base);
      base += plan.carry_bytes;
    }
    if (plan.part_bytes) p.y_partial = reinterpret_cast<float*>(base);
  }
  p.tiles = plan.tiles;
  p.chained = plan.chained ? 1 : 0;
  p.y_pairs = (seqlen % (32 / elt) == 0 && aligned(y, 32)) ? 1 : 0;

  const cudaError_t err = dtype == SS_F32 ? dispatch<float>(p, plan, st)
                                          : dispatch<__nv_bfloat16>(p, plan, st);
  if (scratch) {
    const cudaError_t ferr = cudaFreeAsync(scratch, st);
    if (err == cudaSuccess && ferr != cudaSuccess) return SS_ERR_CUDA;
  }
  return err == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

extern "C" {

SS_API ss_status_t ss_selective_scan_fwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, y, last_state,
                  batch, dim, dstate, seqlen, dtype, stream);
}

SS_API ss_status_t ss_selective_scan_fwd_h0(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* h0, void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  return fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, last_state,
                  batch, dim, dstate, seqlen, dtype, stream);
}

SS_API ss_status_t ss_selective_scan_fwd_host(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* h0, void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  // ---- validation (host arrays): nothing is enqueued or written on error ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !y) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;
  if (!sizes_ok(batch, dim, dstate, seqlen, elt, &sz)) return SS_ERR_UNSUPPORTED;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) ||
      !aligned(y, ea) || (z && !aligned(z, ea)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (delta_bias && !aligned(delta_bias, 4)) || (last_state && !aligned(last_state, 4)) ||
      (h0 && !aligned(h0, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  const void* ins[] = {u, delta, B, C, z, A, D, delta_bias, h0};
  const int64_t in_bytes[] = {sz.x_bytes, sz.x_bytes, sz.bc_bytes, sz.bc_bytes,
                              z ? sz.x_bytes : 0, sz.a_elems * 4, D ? dim * 4 : 0,
                              delta_bias ? dim * 4 : 0, h0 ? sz.st_elems * 4 : 0};
  for (int i = 0; i < 9; ++i) {
    if (range_overlap(y, sz.x_bytes, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    const bool in_place = i == 8 && last_state == h0;
    if (last_state && !in_place && range_overlap(last_state, sz.st_elems * 4, ins[i], in_bytes[i]))
      return SS_ERR_INVALID_ARGUMENT;
  }
  if (last_state && range_overlap(last_state, sz.st_elems * 4, y, sz.x_bytes))
    return SS_ERR_INVALID_ARGUMENT;

  // ---- pieces, two in flight: slices of the batch (contiguous in host
  // memory, independent problems), or, for one sequence, segments of time
  // chained through the state (strided 2-D copies) ----
  const int64_t L = seqlen, N = dstate;
  const bool by_batch = batch > 1;
  int64_t npieces, nb, seg;
  if (by_batch) {
    npieces = std::min<int64_t>(batch, kHostPieces);
    nb = (batch + npieces - 1) / npieces;
    npieces = (batch + nb - 1) / nb;
    seg = L;
  } else {
    const int64_t n = std::max<int64_t>(1, std::min<int64_t>(kHostPieces, L / kHostSegmentSteps));
    seg = round_up((L + n - 1) / n, 64);
    npieces = (L + seg - 1) / seg;
    nb = 1;
  }
  const int64_t xs = round_up(nb * dim * seg * elt, 256), bcs = round_up(nb * N * seg * elt, 256);
  const int64_t ss_bytes = round_up(nb * dim * N * 4, 256);
  const int64_t slot_bytes = (z ? 4 : 3) * xs + 2 * bcs + ss_bytes;
  const int64_t par_bytes = round_up(sz.a_elems * 4, 256) + 2 * round_up(dim * 4, 256);
  const int64_t total = 2 * slot_bytes + par_bytes;

  cudaStream_t sc = static_cast<cudaStream_t>(stream), sh = nullptr, sd = nullptr;
  cudaEvent_t ev[7] = {};  // allocated, inputs in x2, scanned x2, outputs out x2
  void* base = nullptr;
  ss_status_t status = SS_OK;
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && status == SS_OK) status = SS_ERR_CUDA;
    return status == SS_OK;
  };
  (void)cudaGetLastError();
  ok(cudaStreamCreateWithFlags(&sh, cudaStreamNonBlocking));
  ok(cudaStreamCreateWithFlags(&sd, cudaStreamNonBlocking));
  for (auto& e : ev) ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  if (status == SS_OK && ok(cudaMallocAsync(&base, (size_t)total, sc))) {
    char* q = static_cast<char*>(base);
    char* slot[2][7];  // u, delta, y, B, C, z, state
    for (int s = 0; s < 2; ++s) {
      slot[s][0] = q; q += xs;
      slot[s][1] = q; q += xs;
      slot[s][2] = q; q += xs;
      slot[s][3] = q; q += bcs;
      slot[s][4] = q; q += bcs;
      slot[s][5] = z ? q : nullptr; if (z) q += xs;
      slot[s][6] = q; q += ss_bytes;
    }
    float* Ad = reinterpret_cast<float*>(q); q += round_up(sz.a_elems * 4, 256);
    float* Dd = D ? reinterpret_cast<float*>(q) : nullptr; q += round_up(dim * 4, 256);
    float* bd = delta_bias ? reinterpret_cast<float*>(q) : nullptr;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    ok(cudaMemcpyAsync(Ad, A, sz.a_elems * 4, h2d, sc));
    if (D) ok(cudaMemcpyAsync(Dd, D, dim * 4, h2d, sc));
    if (delta_bias) ok(cudaMemcpyAsync(bd, delta_bias, dim * 4, h2d, sc));
    float* chain = reinterpret_cast<float*>(slot[0][6]);  // time segments: one state, chained
    if (!by_batch) {
      if (h0) ok(cudaMemcpyAsync(chain, h0, sz.st_elems * 4, h2d, sc));
      else ok(cudaMemsetAsync(chain, 0, sz.st_elems * 4, sc));
    }
    ok(cudaEventRecord(ev[0], sc));
    ok(cudaStreamWaitEvent(sh, ev[0], 0));
    // rows of `rows` host rows of L steps from step t0, `len` steps each
    auto copy_in = [&](void* dst, const void* src, int64_t row0, int64_t rows, int64_t t0,
                       int64_t len) {
      const char* from = static_cast<const char*>(src) + (row0 * L + t0) * elt;
      if (len == L) return ok(cudaMemcpyAsync(dst, from, rows * L * elt, h2d, sh));
      return ok(cudaMemcpy2DAsync(dst, len * elt, from, L * elt, len * elt, rows, h2d, sh));
    };
    for (int64_t k = 0; k < npieces && status == SS_OK; ++k) {
      const int s = (int)(k & 1);
      const int64_t b0 = by_batch ? k * nb : 0, pb = by_batch ? std::min(nb, batch - b0) : 1;
      const int64_t t0 = by_batch ? 0 : k * seg, len = by_batch ? L : std::min(seg, L - t0);
      const int64_t rows = pb * dim, bc_rows = pb * N;
      float* state = by_batch ? reinterpret_cast<float*>(slot[s][6]) : chain;
      // inputs of piece k (its slot's previous piece is read by then)
      if (k >= 2) ok(cudaStreamWaitEvent(sh, ev[3 + s], 0));
      copy_in(slot[s][0], u, b0 * dim, rows, t0, len);
      copy_in(slot[s][1], delta, b0 * dim, rows, t0, len);
      copy_in(slot[s][3], B, b0 * N, bc_rows, t0, len);
      copy_in(slot[s][4], C, b0 * N, bc_rows, t0, len);
      if (z) copy_in(slot[s][5], z, b0 * dim, rows, t0, len);
      if (by_batch && h0) ok(cudaMemcpyAsync(state, h0 + b0 * dim * N, rows * N * 4, h2d, sh));
      ok(cudaEventRecord(ev[1 + s], sh));
      // the scan of piece k
      ok(cudaStreamWaitEvent(sc, ev[1 + s], 0));
      if (k >= 2) ok(cudaStreamWaitEvent(sc, ev[5 + s], 0));  // its outputs are copied out
      if (status != SS_OK) break;
      status = fwd_impl(slot[s][0], slot[s][1], Ad, slot[s][3], slot[s][4], Dd, slot[s][5], bd,
                        delta_softplus, (by_batch && !h0) ? nullptr : state, slot[s][2],
                        (by_batch && !last_state) ? nullptr : state, pb, dim, N, len, dtype, sc);
      ok(cudaEventRecord(ev[3 + s], sc));
      // outputs of piece k back into their place in the host arrays
      ok(cudaStreamWaitEvent(sd, ev[3 + s], 0));
      char* yto = static_cast<char*>(y) + (b0 * dim * L + t0) * elt;
      if (len == L)
        ok(cudaMemcpyAsync(yto, slot[s][2], rows * L * elt, d2h, sd));
      else
        ok(cudaMemcpy2DAsync(yto, L * elt, slot[s][2], len * elt, len * elt, rows, d2h, sd));
      if (by_batch && last_state)
        ok(cudaMemcpyAsync(last_state + b0 * dim * N, state, rows * N * 4, d2h, sd));
      ok(cudaEventRecord(ev[5 + s], sd));
    }
    if (status == SS_OK && !by_batch && last_state)
      ok(cudaMemcpyAsync(last_state, chain, sz.st_elems * 4, d2h, sc));
    cudaEventRecord(ev[0], sd);
    cudaStreamWaitEvent(sc, ev[0], 0);
    cudaEventRecord(ev[1], sh);
    cudaStreamWaitEvent(sc, ev[1], 0);
    cudaFreeAsync(base, sc);
  }
  if (cudaStreamSynchronize(sc) != cudaSuccess && status == SS_OK) status = SS_ERR_CUDA;
  if (sh) { cudaStreamSynchronize(sh); cudaStreamDestroy(sh); }
  if (sd) { cudaStreamSynchronize(sd); cudaStreamDestroy(sd); }
  for (auto& e : ev)
    if (e) cudaEventDestroy(e);
  return status;
}

SS_API ss_status_t ss_selective_state_update(
    float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* dt_bias, int dt_softplus, void* y,
    int64_t batch, int64_t dim, int64_t dstate, ss_dtype_t dtype, void* stream) {
  // ---- validation: nothing is enqueued or written on error ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!state || !x || !dt || !A || !B || !C || !y) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || dim <= 0 || dstate <= 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;  // one step: [b,d] rows, [b,N] B/C, [b,d,N] state
  if (!sizes_ok(batch, dim, dstate, 1, elt, &sz)) return SS_ERR_UNSUPPORTED;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(x, ea) || !aligned(dt, ea) || !aligned(B, ea) || !aligned(C, ea) ||
      !aligned(y, ea) || (z && !aligned(z, ea)) || !aligned(state, 4) || !aligned(A, 4) ||
      (D && !aligned(D, 4)) || (dt_bias && !aligned(dt_bias, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  const void* ins[] = {x, dt, B, C, z, A, D, dt_bias};
  const int64_t in_bytes[] = {sz.x_bytes, sz.x_bytes, sz.bc_bytes, sz.bc_bytes,
                              z ? sz.x_bytes : 0, sz.a_elems * 4, D ? dim * 4 : 0,
                              dt_bias ? dim * 4 : 0};
  for (int i = 0; i < 8; ++i) {
    if (range_overlap(y, sz.x_bytes, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    if (range_overlap(state, sz.st_elems * 4, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
  }
  if (range_overlap(state, sz.st_elems * 4, y, sz.x_bytes)) return SS_ERR_INVALID_ARGUMENT;

  ss::DecodeParams p{};
  p.state = state; p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.bias = dt_bias; p.y = y;
  p.batch = batch; p.dim = dim; p.dstate = dstate;
  p.softplus = dt_softplus ? 1 : 0;
  p.quads = (int)((dstate + 3) / 4);
  // lanes per row: enough that no lane holds more than kDecodeQuads quads
  p.seg_shift = 0;
  while ((ss::kDecodeQuads << p.seg_shift) < p.quads) ++p.seg_shift;
  const int64_t blocks_x = ((dim << p.seg_shift) + ss::kDecodeThreads - 1) / ss::kDecodeThreads;
  if (blocks_x > INT_MAX) return SS_ERR_UNSUPPORTED;
  // batch rows per CTA: as many as fit (up to kDecodeRows) while the CTAs
  // still cover every SM a few times
  const int64_t sms = std::max(1, sm_count());
  p.rows_per_cta = std::max<int64_t>(
      1, std::min<int64_t>(ss::kDecodeRows, (batch * blocks_x) / (4 * sms)));
  const int64_t groups = (batch + p.rows_per_cta - 1) / p.rows_per_cta;
  if (groups > 65535) return SS_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  const bool vec4 = dstate % 4 == 0 && aligned(state, 16) && aligned(A, 16);
  const dim3 grid((unsigned)blocks_x, (unsigned)groups);
  constexpr int kT = ss::kDecodeThreads;
  if (dtype == SS_F32) {
    if (vec4) ss::ss_state_update<float, true><<<grid, kT, 0, st>>>(p);
    else ss::ss_state_update<float, false><<<grid, kT, 0, st>>>(p);
  } else {
    if (vec4) ss::ss_state_update<__nv_bfloat16, true><<<grid, kT, 0, st>>>(p);
    else ss::ss_state_update<__nv_bfloat16, false><<<grid, kT, 0, st>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // extern "C"

namespace {

// The backward from an initial state h0 (null: zero), with its gradient dh0
// (null: not written); both backward entry points land here.
ss_status_t bwd_impl(const void* u, const void* delta, const float* A, const void* B,
                     const void* C, const float* D, const void* z, const float* delta_bias,
                     int delta_softplus, const float* h0, const void* dy,
                     const float* dlast_state, void* du, void* ddelta, float* dA, float* dB,
                     float* dC, float* dD, void* dz, float* dbias, float* dh0, int64_t batch,
                     int64_t dim, int64_t dstate, int64_t seqlen, ss_dtype_t dtype,
                     void* stream) {
  // ---- validation: nothing is enqueued or written on error ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC)
    return SS_ERR_INVALID_ARGUMENT;
  if (z && !dz) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;
  if (!sizes_ok(batch, dim, dstate, seqlen, elt, &sz)) return SS_ERR_UNSUPPORTED;
  const int groups = (int)((dstate + ss::kBwdLanes - 1) / ss::kBwdLanes);
  const int64_t npad = (int64_t)groups * ss::kBwdLanes;
  // rows per CTA: the main kernel runs in one wave of CTAs whose rows all take
  // the same time, so the SM with the most rows sets the makespan; one state
  // group takes 96-row CTAs when that lowers the most rows an SM holds (the
  // Mamba-2.8B layer's 40960 rows: 3 x 96 = 288 against 5 x 64 = 320, measured
  // 3.10 against 3.33 ms), else 64 (fewer rows than SMs x 64 fill more SMs
  // with the smaller CTAs: the Mamba-130M layer's 3072 rows, 1.62 against 1.94 ms)
  const int64_t nsm = std::max(1, sm_count());
  auto most_rows = [&](int64_t r) {
    const int64_t c = batch * ((dim + r - 1) / r);
    return (c + nsm - 1) / nsm * r;
  };
  const int64_t bwd_rows =
      (groups == 1 && most_rows(ss::kBwdRowsWide) < most_rows(ss::kBwdRows)) ? ss::kBwdRowsWide
                                                                              : ss::kBwdRows;
  const int64_t dtiles = (dim + bwd_rows - 1) / bwd_rows;
  const int64_t ctas = batch * dtiles;
  const int64_t nblk = (seqlen + ss::kBwdBlock - 1) / ss::kBwdBlock;
  int64_t ck_elems, bc_elems, row_elems = 0, tmp;
  if (!mul_ok(ctas * bwd_rows * ss::kBwdLanes, nblk, &ck_elems) ||
      !mul_ok(ctas * 2 * npad, seqlen, &bc_elems) || !mul_ok(ck_elems + bc_elems, 4, &tmp) ||
      (groups > 1 && !mul_ok(3 * sz.rows, seqlen, &row_elems)) || ctas > INT_MAX)
    return SS_ERR_UNSUPPORTED;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) ||
      !aligned(dy, ea) || !aligned(du, ea) || !aligned(ddelta, ea) || (z && !aligned(z, ea)) ||
      (dz && !aligned(dz, ea)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (delta_bias && !aligned(delta_bias, 4)) || (dlast_state && !aligned(dlast_state, 4)) ||
      !aligned(dA, 4) || !aligned(dB, 4) || !aligned(dC, 4) || (dD && !aligned(dD, 4)) ||
      (dbias && !aligned(dbias, 4)) || (h0 && !aligned(h0, 4)) || (dh0 && !aligned(dh0, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  // outputs must not overlap any input, nor each other
  const void* ins[] = {u, delta, A, B, C, D, z, delta_bias, dy, dlast_state, h0};
  const int64_t in_bytes[] = {sz.x_bytes, sz.x_bytes, sz.a_elems * 4, sz.bc_bytes, sz.bc_bytes,
                              D ? dim * 4 : 0, z ? sz.x_bytes : 0, delta_bias ? dim * 4 : 0,
                              sz.x_bytes, dlast_state ? sz.st_elems * 4 : 0,
                              h0 ? sz.st_elems * 4 : 0};
  const void* outs[] = {du, ddelta, dz, dA, dB, dC, dD, dbias, dh0};
  const int64_t out_bytes[] = {sz.x_bytes, sz.x_bytes, dz ? sz.x_bytes : 0, sz.a_elems * 4,
                               sz.bc_bytes / elt * 4, sz.bc_bytes / elt * 4, dD ? dim * 4 : 0,
                               dbias ? dim * 4 : 0, (h0 && dh0) ? sz.st_elems * 4 : 0};
  for (int o = 0; o < 9; ++o) {
    for (int i = 0; i < 11; ++i)
      if (range_overlap(outs[o], out_bytes[o], ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    for (int k = o + 1; k < 9; ++k)
      if (range_overlap(outs[o], out_bytes[o], outs[k], out_bytes[k])) return SS_ERR_INVALID_ARGUMENT;
  }

  // ---- scratch: checkpoints, per-CTA dB/dC sums, per-row dA/dD/dbias sums,
  //      and (several state groups) the row sums carried from group to group ----
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t a_elems = batch * dim * npad, dd_elems = batch * dim * 2;
  const int64_t scratch = round_up(ck_elems * 4, 256) + round_up(bc_elems * 4, 256) +
                          round_up(a_elems * 4, 256) + round_up(dd_elems * 4, 256) +
                          round_up(row_elems * 4, 256);
  (void)cudaGetLastError();
  void* base = nullptr;
  if (cudaMallocAsync(&base, (size_t)scratch, st) != cudaSuccess) return SS_ERR_CUDA;
  char* cur = static_cast<char*>(base);
  ss::BwdParams p{};
  p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.bias = delta_bias;
  p.softplus = delta_softplus ? 1 : 0;
  p.dy = dy; p.dlast = dlast_state; p.du = du; p.ddelta = ddelta; p.dz = dz;
  p.dA = dA; p.dB = dB; p.dC = dC; p.dD = D ? dD : nullptr; p.dbias = delta_bias ? dbias : nullptr;
  p.h0 = h0; p.dh0 = h0 ? dh0 : nullptr;
  p.ckpt = reinterpret_cast<float*>(cur);
  cur += round_up(ck_elems * 4, 256);
  p.part_bc = reinterpret_cast<float*>(cur);
  cur += round_up(bc_elems * 4, 256);
  p.part_a = reinterpret_cast<float*>(cur);
  cur += round_up(a_elems * 4, 256);
  p.part_dd = reinterpret_cast<float*>(cur);
  cur += round_up(dd_elems * 4, 256);
  p.part_row = groups > 1 ? reinterpret_cast<float*>(cur) : nullptr;
  p.npad = (int)npad;
  p.batch = batch; p.dim = dim; p.dstate = dstate; p.seqlen = seqlen;
  p.dtiles = dtiles; p.nblk = nblk;
  p.vec = seqlen % (16 / elt) == 0 && aligned(u, 16) && aligned(delta, 16) && aligned(dy, 16) &&
          (!z || aligned(z, 16));
  // the backward is latency-bound: the whole shared memory for resident CTAs
  static const bool carveout = [] {
    for (auto k : {(const void*)ss::ss_bwd_main<float, true, false>,
                   (const void*)ss::ss_bwd_main<float, false, false>,
                   (const void*)ss::ss_bwd_main<__nv_bfloat16, true, false>,
                   (const void*)ss::ss_bwd_main<__nv_bfloat16, false, false>,
                   (const void*)ss::ss_bwd_main<float, true, true>,
                   (const void*)ss::ss_bwd_main<float, false, true>,
                   (const void*)ss::ss_bwd_main<__nv_bfloat16, true, true>,
                   (const void*)ss::ss_bwd_main<__nv_bfloat16, false, true>})
      cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    for (auto k : {(const void*)ss::ss_bwd_main<float, true, false, ss::kBwdRowsWide>,
                   (const void*)ss::ss_bwd_main<float, false, false, ss::kBwdRowsWide>,
                   (const void*)ss::ss_bwd_main<__nv_bfloat16, true, false, ss::kBwdRowsWide>,
                   (const void*)ss::ss_bwd_main<__nv_bfloat16, false, false, ss::kBwdRowsWide>}) {
      cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sizeof(ss::BwdSmem<ss::kBwdRowsWide>));
    }
    return true;
  }();
  (void)carveout;
  (void)cudaGetLastError();
  const unsigned grid = (unsigned)ctas;
  constexpr int kR = ss::kBwdRows, kW = ss::kBwdRowsWide;
  constexpr unsigned kWideSmem = sizeof(ss::BwdSmem<ss::kBwdRowsWide>);
  for (int g = 0; g < groups; ++g) {
    p.group = g;
    p.final_group = g == groups - 1;
    if (groups == 1 && bwd_rows == kW) {
      if (dtype == SS_F32) {
        if (z) ss::ss_bwd_main<float, true, false, kW><<<grid, kW, kWideSmem, st>>>(p);
        else ss::ss_bwd_main<float, false, false, kW><<<grid, kW, kWideSmem, st>>>(p);
      } else {
        if (z) ss::ss_bwd_main<__nv_bfloat16, true, false, kW><<<grid, kW, kWideSmem, st>>>(p);
        else ss::ss_bwd_main<__nv_bfloat16, false, false, kW><<<grid, kW, kWideSmem, st>>>(p);
      }
    } else if (groups == 1) {
      if (dtype == SS_F32) {
        if (z) ss::ss_bwd_main<float, true, false><<<grid, kR, 0, st>>>(p);
        else ss::ss_bwd_main<float, false, false><<<grid, kR, 0, st>>>(p);
      } else {
        if (z) ss::ss_bwd_main<__nv_bfloat16, true, false><<<grid, kR, 0, st>>>(p);
        else ss::ss_bwd_main<__nv_bfloat16, false, false><<<grid, kR, 0, st>>>(p);
      }
    } else {
      if (dtype == SS_F32) {
        if (z) ss::ss_bwd_main<float, true, true><<<grid, kR, 0, st>>>(p);
        else ss::ss_bwd_main<float, false, true><<<grid, kR, 0, st>>>(p);
      } else {
        if (z) ss::ss_bwd_main<__nv_bfloat16, true, true><<<grid, kR, 0, st>>>(p);
        else ss::ss_bwd_main<__nv_bfloat16, false, true><<<grid, kR, 0, st>>>(p);
      }
    }
  }
  const int sms = std::max(1, sm_count());
  const int64_t bc_total = batch * dstate * seqlen, rows_total = dim * dstate;
  ss::ss_bwd_reduce_bc<<<(unsigned)std::min<int64_t>((bc_total + 255) / 256, 8 * sms), 256, 0,
                         st>>>(p);
  ss::ss_bwd_reduce_rows<<<(unsigned)std::min<int64_t>((rows_total + 255) / 256, 8 * sms), 256, 0,
                           st>>>(p);
  const cudaError_t err = cudaGetLastError();
  const cudaError_t ferr = cudaFreeAsync(base, st);
  return err == cudaSuccess && ferr == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// The general Mamba-2 path (any head dim, up to 256 states, fp32 or bf16):
// each head group runs as one selective scan over its heads' channels, on
// channel-major copies of its inputs (ss_layout.cuh), with A, D and the dt
// bias repeated per channel.  The scan's arithmetic is the Mamba-1 forward's
// (fp32 throughout; bf16 only where y is stored).  Scratch is allocated on the
// stream and freed after the last kernel that uses it.
ss_status_t mamba2_rows(const void* x, const void* dt, const float* A, const void* B,
                        const void* C, const float* D, const float* dt_bias, int dt_softplus,
                        const float* h0, void* y, float* final_state, int64_t batch,
                        int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                        int64_t dstate, ss_dtype_t dtype, cudaStream_t st) {
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  const int64_t L = seqlen, N = dstate, G = ngroups;
  const int64_t CH = nheads * headdim, Cg = CH / G;  // scan channels, per group
  if (batch > 65535 || L > (int64_t)INT_MAX * ss::kTile) return SS_ERR_UNSUPPORTED;  // grid z, y
  const int64_t rows_bytes = round_up(batch * CH * L * elt, 256);
  const int64_t bc_bytes = round_up(G * batch * N * L * elt, 256);
  const int64_t a_bytes = round_up(CH * N * 4, 256), v_bytes = round_up(CH * 4, 256);
  const int64_t st_bytes = G > 1 ? round_up(batch * CH * N * 4, 256) : 0;
  const int64_t total = 3 * rows_bytes + 2 * bc_bytes + a_bytes + 2 * v_bytes + 2 * st_bytes;
  (void)cudaGetLastError();
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, (size_t)total, st) != cudaSuccess) return SS_ERR_CUDA;
  char* p = static_cast<char*>(scratch);
  char* u = p;                   p += rows_bytes;
  char* delta = p;               p += rows_bytes;
  char* yr = p;                  p += rows_bytes;
  char* Bt = p;                  p += bc_bytes;
  char* Ct = p;                  p += bc_bytes;
  float* Ae = reinterpret_cast<float*>(p);  p += a_bytes;
  float* De = reinterpret_cast<float*>(p);  p += v_bytes;
  float* be = reinterpret_cast<float*>(p);  p += v_bytes;
  float* h0g = reinterpret_cast<float*>(p); p += st_bytes;
  float* lastg = reinterpret_cast<float*>(p);

  auto to_rows = [&](const void* in, void* out, int64_t Cin, int rep, int64_t groups) {
    const dim3 grid((unsigned)((Cin * rep + ss::kTile - 1) / ss::kTile),
                    (unsigned)((L + ss::kTile - 1) / ss::kTile), (unsigned)batch);
    if (elt == 4)
      ss::ss_to_rows<float><<<grid, 256, 0, st>>>(static_cast<const float*>(in),
                                                  static_cast<float*>(out), batch, L, Cin, rep,
                                                  groups);
    else
      ss::ss_to_rows<__nv_bfloat16><<<grid, 256, 0, st>>>(
          static_cast<const __nv_bfloat16*>(in), static_cast<__nv_bfloat16*>(out), batch, L, Cin,
          rep, groups);
  };
  to_rows(x, u, CH, 1, G);                  // x [b,L,H*P] -> [G][b][Cg][L]
  to_rows(dt, delta, nheads, (int)headdim, G);  // dt [b,L,H] -> every channel of its head
  to_rows(B, Bt, G * N, 1, G);              // B [b,L,G,N] -> [G][b][N][L]
  to_rows(C, Ct, G * N, 1, G);
  const int64_t pe = CH * N;
  ss::ss_expand_heads<<<(unsigned)std::min<int64_t>((pe + 255) / 256, 4096), 256, 0, st>>>(
      A, D, dt_bias, Ae, De, be, nheads, headdim, N);
  const int64_t se = batch * CH * N;
  const unsigned sgrid = (unsigned)std::min<int64_t>((se + 255) / 256, 8192);
  if (G > 1 && h0) ss::ss_group_rows<<<sgrid, 256, 0, st>>>(h0, h0g, batch, G, Cg, N, 1);
  ss_status_t status = cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  for (int64_t g = 0; g < G && status == SS_OK; ++g) {
    const int64_t ro = g * batch * Cg * L * elt, bo = g * batch * N * L * elt;
    const float* h0_g = G > 1 ? (h0 ? h0g + g * batch * Cg * N : nullptr) : h0;
    float* last_g = G > 1 ? (final_state ? lastg + g * batch * Cg * N : nullptr) : final_state;
    status = fwd_impl(u + ro, delta + ro, Ae + g * Cg * N, Bt + bo, Ct + bo,
                      D ? De + g * Cg : nullptr, nullptr, dt_bias ? be + g * Cg : nullptr,
                      dt_softplus, h0_g, yr + ro, last_g, batch, Cg, N, L, dtype, st);
  }
  if (status == SS_OK) {
    const dim3 grid((unsigned)((CH + ss::kTile - 1) / ss::kTile),
                    (unsigned)((L + ss::kTile - 1) / ss::kTile), (unsigned)batch);
    if (elt == 4)
      ss::ss_from_rows<float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(yr),
                                                    static_cast<float*>(y), batch, L, CH, G);
    else
      ss::ss_from_rows<__nv_bfloat16><<<grid, 256, 0, st>>>(
          reinterpret_cast<const __nv_bfloat16*>(yr), static_cast<__nv_bfloat16*>(y), batch, L,
          CH, G);
    if (G > 1 && final_state)
      ss::ss_group_rows<<<sgrid, 256, 0, st>>>(lastg, final_state, batch, G, Cg, N, 0);
    if (cudaGetLastError() != cudaSuccess) status = SS_ERR_CUDA;
  }
  if (cudaFreeAsync(scratch, st) != cudaSuccess && status == SS_OK) status = SS_ERR_CUDA;
  return status;
}

}  // namespace

extern "C" {

SS_API ss_status_t ss_selective_scan_bwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const void* dy, const float* dlast_state, void* du, void* ddelta, float* dA, float* dB,
    float* dC, float* dD, void* dz, float* dbias,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ss_dtype_t dtype, void* stream) {
  return bwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, dy, dlast_state,
                  du, ddelta, dA, dB, dC, dD, dz, dbias, nullptr, batch, dim, dstate, seqlen,
                  dtype, stream);
}

SS_API ss_status_t ss_selective_scan_bwd_h0(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, const float* h0,
    const void* dy, const float* dlast_state, void* du, void* ddelta, float* dA, float* dB,
    float* dC, float* dD, void* dz, float* dbias, float* dh0,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ss_dtype_t dtype, void* stream) {
  return bwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, dy, dlast_state, du,
                  ddelta, dA, dB, dC, dD, dz, dbias, dh0, batch, dim, dstate, seqlen, dtype,
                  stream);
}

SS_API ss_status_t ss_selective_scan_fwd_pc(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  return ss_selective_scan_fwd_pc_h0(u, delta, A, B, C, D, z, delta_bias, delta_softplus,
                                     nullptr, y, last_state, batch, dim, dstate, seqlen, dtype,
                                     stream);
}

SS_API ss_status_t ss_selective_scan_fwd_pc_h0(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* h0, void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  // ---- validation: nothing is enqueued or written on error ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !y) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;
  int64_t bc_bytes;
  if (!sizes_ok(batch, dim, dstate, seqlen, elt, &sz) || !mul_ok(sz.x_bytes, dstate, &bc_bytes))
    return SS_ERR_UNSUPPORTED;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) ||
      !aligned(y, ea) || (z && !aligned(z, ea)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (delta_bias && !aligned(delta_bias, 4)) || (last_state && !aligned(last_state, 4)) ||
      (h0 && !aligned(h0, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  const void* ins[] = {u, delta, B, C, z, A, D, delta_bias, h0};
  const int64_t in_bytes[] = {sz.x_bytes, sz.x_bytes, bc_bytes, bc_bytes, z ? sz.x_bytes : 0,
                              sz.a_elems * 4, D ? dim * 4 : 0, delta_bias ? dim * 4 : 0,
                              h0 ? sz.st_elems * 4 : 0};
  for (int i = 0; i < 9; ++i) {
    if (range_overlap(y, sz.x_bytes, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    // last_state may be h0 itself: each lane reads its states of h0 before it
    // writes them back
    if (last_state && !(i == 8 && last_state == h0) &&
        range_overlap(last_state, sz.st_elems * 4, ins[i], in_bytes[i]))
      return SS_ERR_INVALID_ARGUMENT;
  }
  if (last_state && range_overlap(last_state, sz.st_elems * 4, y, sz.x_bytes))
    return SS_ERR_INVALID_ARGUMENT;

  ss::PcParams p{};
  p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.bias = delta_bias;
  p.softplus = delta_softplus ? 1 : 0;
  p.y = y; p.last_state = last_state; p.h0 = h0;
  p.rows = batch * dim; p.dim = dim; p.dstate = dstate; p.seqlen = seqlen;
  const int quads = (int)((dstate + 3) / 4);
  p.seg_shift = 0;
  while ((1 << p.seg_shift) < quads) ++p.seg_shift;
  const int64_t blocks = ((p.rows << p.seg_shift) + 223) / 224;  // the smaller CTA size
  if (blocks > INT_MAX) return SS_ERR_UNSUPPORTED;
  const bool vec = seqlen % (32 / elt) == 0 && aligned(u, 32) && aligned(delta, 32) &&
                   aligned(B, 32) && aligned(C, 32) && aligned(y, 16) && (!z || aligned(z, 32));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  const int sms = sm_count();
  if (dtype == SS_F32) pc_launch<float>(p, z != nullptr, vec, sms, st);
  else pc_launch<__nv_bfloat16>(p, z != nullptr, vec, sms, st);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

SS_API ss_status_t ss_mamba2_fwd(
    const void* x, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const float* dt_bias, int dt_softplus, void* y, float* final_state,
    int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
    int64_t dstate, ss_dtype_t dtype, void* stream) {
  return ss_mamba2_fwd_h0(x, dt, A, B, C, D, dt_bias, dt_softplus, nullptr, y, final_state,
                          batch, seqlen, nheads, headdim, ngroups, dstate, dtype, stream);
}

SS_API ss_status_t ss_mamba2_fwd_h0(
    const void* x, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const float* dt_bias, int dt_softplus, const float* initial_state, void* y,
    float* final_state, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
    int64_t ngroups, int64_t dstate, ss_dtype_t dtype, void* stream) {
  // ---- validation: nothing is enqueued or written on error ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!x || !dt || !A || !B || !C || !y) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0)
    return SS_ERR_INVALID_ARGUMENT;
  if (nheads % ngroups != 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  int64_t tokens, x_elems, bc_elems, dt_elems, units, st_elems;
  if (!mul_ok(batch, seqlen, &tokens) || !mul_ok(tokens, nheads, &dt_elems) ||
      !mul_ok(dt_elems, headdim, &x_elems) || !mul_ok(tokens, ngroups, &bc_elems) ||
      !mul_ok(bc_elems, dstate, &bc_elems) || !mul_ok(batch, nheads, &units) ||
      !mul_ok(units, headdim * dstate, &st_elems) || x_elems > INT64_MAX / 4 ||
      bc_elems > INT64_MAX / 4 || st_elems > INT64_MAX / 4)
    return SS_ERR_UNSUPPORTED;
  if (units > INT_MAX) return SS_ERR_UNSUPPORTED;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(x, ea) || !aligned(B, ea) || !aligned(C, ea) || !aligned(y, ea) ||
      !aligned(dt, ea) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (dt_bias && !aligned(dt_bias, 4)) || (final_state && !aligned(final_state, 4)) ||
      (initial_state && !aligned(initial_state, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  const void* ins[] = {x, dt, B, C, A, D, dt_bias, initial_state};
  const int64_t in_bytes[] = {x_elems * elt, dt_elems * elt, bc_elems * elt, bc_elems * elt,
                              nheads * 4, D ? nheads * 4 : 0, dt_bias ? nheads * 4 : 0,
                              initial_state ? st_elems * 4 : 0};
  for (int i = 0; i < 8; ++i) {
    if (range_overlap(y, x_elems * elt, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    // final_state may be initial_state itself: each thread reads its part of
    // the given state before it writes the same elements back
    if (final_state && !(i == 7 && final_state == initial_state) &&
        range_overlap(final_state, st_elems * 4, ins[i], in_bytes[i]))
      return SS_ERR_INVALID_ARGUMENT;
  }
  if (final_state && range_overlap(final_state, st_elems * 4, y, x_elems * elt))
    return SS_ERR_INVALID_ARGUMENT;

  // the tensor-core kernel takes bf16, head dim 64 and 128 states with 16-byte
  // aligned x, B, C and y (TMA); every other call runs on the scan kernels
  const bool tc = dtype == SS_BF16 && headdim == ss::kSsdP && dstate == ss::kSsdN &&
                  aligned(x, 16) && aligned(B, 16) && aligned(C, 16) && aligned(y, 16) &&
                  SS_TUNING("SS_MAMBA2_ROWS", 0) == 0;
  if (!tc)
    return mamba2_rows(x, dt, A, B, C, D, dt_bias, dt_softplus, initial_state, y, final_state,
                       batch, seqlen, nheads, headdim, ngroups, dstate, dtype,
                       static_cast<cudaStream_t>(stream));

  if (seqlen > INT_MAX || batch > INT_MAX || nheads * headdim > INT_MAX ||
      ngroups * dstate > INT_MAX)
    return SS_ERR_UNSUPPORTED;  // TMA coordinates are 32-bit
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SS_ERR_CUDA;
  static std::once_flag smem_once[64];
  cudaError_t attr = cudaSuccess;
  std::call_once(smem_once[dev], [&] {
    attr = cudaFuncSetAttribute(ss::ss_ssd_fwd<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ss::kSsdSmemBytes);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(ss::ss_ssd_fwd<true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)ss::kSsdSmemBytes);
  });
  if (attr != cudaSuccess) return SS_ERR_CUDA;

  ss::SsdParams p{};
  // x as [batch, seqlen, nheads*headdim], B and C as [batch, seqlen, ngroups*dstate]
  if (!tma_map_rows(&p.tx, x, nheads * headdim, seqlen, batch) ||
      !tma_map_rows(&p.tb, B, ngroups * dstate, seqlen, batch) ||
      !tma_map_rows(&p.tc, C, ngroups * dstate, seqlen, batch))
    return SS_ERR_CUDA;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.dt = static_cast<const __nv_bfloat16*>(dt);
  p.A = A;
  p.B = static_cast<const __nv_bfloat16*>(B);
  p.C = static_cast<const __nv_bfloat16*>(C);
  p.D = D;
  p.bias = dt_bias;
  p.softplus = dt_softplus ? 1 : 0;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.h0 = initial_state;
  p.final_state = final_state;
  p.batch = batch; p.seqlen = seqlen; p.nheads = nheads; p.ngroups = ngroups;
  (void)cudaGetLastError();
  const auto kernel = initial_state ? ss::ss_ssd_fwd<true> : ss::ss_ssd_fwd<false>;
  kernel<<<(unsigned)units, ss::kSsdThreads, ss::kSsdSmemBytes,
           static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
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
  out->ctas = plan.grid;
  out->kernel_launches = plan.launches;
  out->scratch_bytes = scratch_bytes(plan);
  out->vector_path = plan.vec ? 1 : 0;
  return SS_OK;
}

SS_API ss_status_t ss_selective_scan_check(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SS_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, ss::g_ss_device_error, sizeof(word)) != cudaSuccess)
    return SS_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(ss::g_ss_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return SS_ERR_CUDA;
    return SS_ERR_TIMEOUT;
  }
  return SS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation entry point: the scheduled kernel with its scratch in a fixed
// buffer of the library's own device memory instead of stream-ordered
// allocations, for callers that cannot allocate during a call.
namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(16) << 20;  // 16 MiB per device
constexpr int kNoAllocMaxDevices = 64;

// The buffer itself.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
struct NoallocAddress {
  unsigned long long ctx_id = 0;  // the context the address belongs to (0: none yet)
  void* ptr = nullptr;
};
NoallocAddress g_noalloc_address[kNoAllocMaxDevices];

// Unique id of the current context (driver API, looked up through the
// runtime), or 0 if it cannot be had.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static const std::pair<GetCurrent, GetId> fns = [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      a = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      b = nullptr;
    return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!fns.first || !fns.second || fns.first(&ctx) != CUDA_SUCCESS || !ctx ||
      fns.second(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the buffer in the current context.  It is looked up with
// cudaGetSymbolAddress once per device context (the first call on a device
// does this set-up), and again whenever the context changed, e.g. after a
// cudaDeviceReset: the module is then loaded anew and its buffer can move.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  // 0 before the runtime has made the device's context current: then the
  // lookup below (which creates it) runs, and the next call records its id
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocAddress& a = g_noalloc_address[dev];
  if (ctx == 0 || a.ptr == nullptr || a.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    a.ptr = p;
    a.ctx_id = ctx;
  }
  *out = a.ptr;
  return cudaSuccess;
}

// Re-derive the chunked part of a vector-path plan for a forced chunk count.
void set_chunks(LaunchPlan* plan, int64_t seqlen, int64_t slots, int64_t want) {
  want = std::max<int64_t>(1, std::min<int64_t>(want, seqlen / ss::kTileSteps));
  plan->chunk_len = round_up((seqlen + want - 1) / want, ss::kTileSteps);
  plan->nchunks = (int)((seqlen + plan->chunk_len - 1) / plan->chunk_len);
  plan->grid = std::min<int64_t>(plan->tiles * plan->nchunks, slots);
  plan->chained = plan->tiles >= plan->grid;
  plan->sched_bytes_per_group = round_up(128 + plan->nchunks * plan->tiles * 4, 256);
  plan->sched_bytes = plan->sched_bytes_per_group * plan->groups;
  const int64_t rec = (int64_t)plan->nchunks * plan->tiles * plan->rows_per_cta * plan->nt;
  plan->unit_agg_bytes = round_up(rec * 8, 256);
  plan->unit_incl_bytes = round_up(rec * 4, 256);
}

// Plan of the no-allocation entry point: the regular vector-path plan with the
// largest chunk count, at most the regular one, whose carries fit the fixed
// buffer.  SS_ERR_SCRATCH_LIMIT if even one chunk does not fit.
ss_status_t noalloc_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int64_t elt,
                         int sms, LaunchPlan* plan) {
  if (!make_plan(batch, dim, dstate, seqlen, elt, true, sms, plan) || !plan->vec)
    return SS_ERR_UNSUPPORTED;
  for (int64_t n = plan->nchunks; scratch_bytes(*plan) > kNoAllocScratchBytes && n > 1;) {
    set_chunks(plan, seqlen, plan->slots, --n);
    n = std::min<int64_t>(n, plan->nchunks);
  }
  if (plan->nchunks == 1) plan->unit_agg_bytes = plan->unit_incl_bytes = 0;  // no carries
  return scratch_bytes(*plan) > kNoAllocScratchBytes ? SS_ERR_SCRATCH_LIMIT : SS_OK;
}

}  // namespace

#ifdef SS_TEST_HOOKS
// ---- test build only: inspection of the no-allocation entry point ----------------
extern "C" {
// The plan ss_selective_scan_fwd_noalloc would run (host only).
SS_API ss_status_t ss_test_noalloc_plan(int64_t batch, int64_t dim, int64_t dstate,
                                        int64_t seqlen, ss_dtype_t dtype, int sm_count,
                                        ss_plan_t* out) {
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  LaunchPlan plan{};
  const ss_status_t st =
      noalloc_plan(batch, dim, dstate, seqlen, dtype == SS_F32 ? 4 : 2, sm_count, &plan);
  if (st != SS_OK) return st;
  out->nchunks = plan.nchunks;
  out->chunk_len = plan.chunk_len;
  out->state_groups = plan.groups;
  out->ctas = plan.grid;
  out->kernel_launches = plan.launches;
  out->scratch_bytes = scratch_bytes(plan);
  out->vector_path = 1;
  return SS_OK;
}
// The buffer address the entry point would use now, and a fresh lookup.
SS_API int ss_test_noalloc_addresses(void** used, void** fresh) {
  if (noalloc_scratch(used) != cudaSuccess) return 1;
  return cudaGetSymbolAddress(fresh, g_noalloc_scratch) == cudaSuccess ? 0 : 2;
}
// Runtime calls of the library's own CUDA runtime, for a test process that
// resets the device without torch.
SS_API int ss_test_device_reset() { return (int)cudaDeviceReset(); }
SS_API int ss_test_malloc(void** p, size_t bytes) { return (int)cudaMalloc(p, bytes); }
SS_API int ss_test_free(void* p) { return (int)cudaFree(p); }
SS_API int ss_test_memcpy(void* dst, const void* src, size_t bytes) {
  return (int)cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
}
}  // extern "C"
#endif

extern "C" SS_API ss_status_t ss_selective_scan_fwd_noalloc(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream) {
  // ---- validation, as ss_selective_scan_fwd ----
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !y) return SS_ERR_INVALID_ARGUMENT;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return SS_ERR_INVALID_ARGUMENT;
  if (dstate > 256) return SS_ERR_UNSUPPORTED;
  const int64_t elt = dtype == SS_F32 ? 4 : 2;
  Sizes sz;
  if (!sizes_ok(batch, dim, dstate, seqlen, elt, &sz)) return SS_ERR_UNSUPPORTED;
  const uintptr_t ea = (uintptr_t)elt;
  if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) ||
      !aligned(y, ea) || (z && !aligned(z, ea)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
      (delta_bias && !aligned(delta_bias, 4)) || (last_state && !aligned(last_state, 4)))
    return SS_ERR_INVALID_ARGUMENT;
  const void* ins[] = {u, delta, B, C, z, A, D, delta_bias};
  const int64_t in_bytes[] = {sz.x_bytes, sz.x_bytes, sz.bc_bytes, sz.bc_bytes,
                              z ? sz.x_bytes : 0, sz.a_elems * 4, D ? dim * 4 : 0,
                              delta_bias ? dim * 4 : 0};
  for (int i = 0; i < 8; ++i) {
    if (range_overlap(y, sz.x_bytes, ins[i], in_bytes[i])) return SS_ERR_INVALID_ARGUMENT;
    if (last_state && range_overlap(last_state, sz.st_elems * 4, ins[i], in_bytes[i]))
      return SS_ERR_INVALID_ARGUMENT;
  }
  if (last_state && range_overlap(last_state, sz.st_elems * 4, y, sz.x_bytes))
    return SS_ERR_INVALID_ARGUMENT;

  // ---- plan: the vector path only, its carries fitted into the fixed buffer ----
  const bool aligned16 = aligned(u, 16) && aligned(delta, 16) && aligned(B, 16) &&
                         aligned(C, 16) && aligned(y, 16) && (!z || aligned(z, 16));
  if (!aligned16 || seqlen % (16 / elt) != 0) return SS_ERR_UNSUPPORTED;
  const int sms = sm_count();
  if (sms <= 0) return SS_ERR_CUDA;
  LaunchPlan plan{};
  const ss_status_t planned = noalloc_plan(batch, dim, dstate, seqlen, elt, sms, &plan);
  if (planned != SS_OK) return planned;

  void* base_ptr = nullptr;
  if (noalloc_scratch(&base_ptr) != cudaSuccess) return SS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ss::FwdParams p{};
  p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.bias = delta_bias;
  p.y = y; p.last_state = last_state;
  p.batch = batch; p.dim = dim; p.dstate = dstate; p.seqlen = seqlen;
  p.chunk_len = plan.chunk_len;
  p.nchunks = plan.nchunks;
  p.ns = plan.groups * plan.nt;
  p.softplus = delta_softplus ? 1 : 0;
  p.tiles = plan.tiles;
  p.chained = plan.chained ? 1 : 0;
  p.y_pairs = (seqlen % (32 / elt) == 0 && aligned(y, 32)) ? 1 : 0;
  char* base = static_cast<char*>(base_ptr);
  (void)cudaGetLastError();
  // the tickets and unit flags of the previous call must not be seen
  if (cudaMemsetAsync(base, 0, (size_t)plan.sched_bytes, st) != cudaSuccess) return SS_ERR_CUDA;
  p.ticket = reinterpret_cast<unsigned*>(base);
  base += plan.sched_bytes;
  if (plan.unit_agg_bytes) {
    p.unit_agg = reinterpret_cast<float2*>(base);
    base += plan.unit_agg_bytes;
    p.unit_incl = reinterpret_cast<float*>(base);
    base += plan.unit_incl_bytes;
  }
  if (plan.part_bytes) p.y_partial = reinterpret_cast<float*>(base);
  const cudaError_t err = dtype == SS_F32 ? dispatch<float>(p, plan, st)
                                          : dispatch<__nv_bfloat16>(p, plan, st);
  return err == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
