/*
 * CPU oracle for the Mamba selective-scan forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes is the plain sequential definition of the scan, in
 * double precision, one (batch, channel) row at a time:
 *
 *   for t in 0..L-1:
 *     dt   = delta[b,d,t] + delta_bias[d];  if softplus: dt = log(1 + e^dt)
 *     for n: h[n] = exp(dt * A[d,n]) * h[n] + dt * B[b,n,t] * u[b,d,t]
 *     y    = sum_n C[b,n,t] * h[n] + D[d] * u[b,d,t]
 *     if z: y = y * z / (1 + e^-z)                       (silu gate)
 *     out[b,d,t] = y
 *   last_state[b,d,n] = h[n]
 *
 * Passages it follows:
 *   - "ТЕХНИЧЕСКОЕ ЗАДАНИЕ: Реализовать selective scan (Mamba)", Этап 1,
 *     step 3 (the maths: A_bar = exp(delta*A), B_bar = delta*B,
 *     delta = softplus(Delta)) and step 4 (the prototype's loop: state update,
 *     read-out C*state summed over the state axis, D skip, silu(z) gate
 *     applied after the skip).
 *   - "Mamba CUDA 实现解析" (mamba-code-explained), section "Mamba SSM简化",
 *     eq (4)-(6): channels independent, A a length-N vector, diagonal
 *     discretised transition; eq (7): the scalar recurrence
 *     v_k = a_k v_{k-1} + b_k u_k per state element.
 *   - "从顺序到并行用PyTorch实现Blelloch算法加速Mamba状态空间模型", section 4.1:
 *     deltaA = exp(delta * A), deltaB = delta * B broadcast over channels,
 *     y = hs . C + D * x.
 *
 * Readings where the pages are silent or garbled (each one is listed with
 * its reason in the design notes of the repository):
 *   - the state is [batch, dim, dstate]; B_bar = dt * B (Euler form) times u
 *     once; delta_bias is added inside the softplus; with softplus off,
 *     dt = delta + bias;
 *   - the initial state is zero unless h0 is given;
 *   - softplus is evaluated as max(x,0) + log1p(exp(-|x|)), which equals
 *     log(1 + e^x) for every x without overflow;
 *   - no clamp is applied to A.
 *
 * Inputs are read in the ABI layouts (u/delta/z [b,d,L], B/C [b,N,L],
 * A [d,N], D and bias [d]); dtype 0 means float32 values, dtype 1 means
 * bfloat16 bit patterns, widened exactly to double.  Outputs are double.
 * Rows are split over nthreads POSIX threads; each row is independent.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

typedef struct {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* bias;
  int softplus;
  const double* h0;
  double* y;
  double* last_state;
  int64_t batch, dim, dstate, seqlen;
  int dtype;
  int64_t row_begin, row_end;
  int status;
} oracle_job;

/* Widen element i of an fp32 or bf16 array to double. */
static double load_elem(const void* p, int64_t i, int dtype) {
  if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* softplus(x) = log(1 + e^x), written so that it neither overflows for large
 * x nor loses the small result for very negative x. */
static double softplus(double x) {
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

static void run_rows(oracle_job* j) {
  const int64_t N = j->dstate, L = j->seqlen, dim = j->dim;
  double* h = (double*)malloc(sizeof(double) * (size_t)N);
  if (!h) {
    j->status = 2;
    return;
  }
  for (int64_t row = j->row_begin; row < j->row_end; ++row) {
    const int64_t b = row / dim, d = row % dim;
    for (int64_t n = 0; n < N; ++n) h[n] = j->h0 ? j->h0[row * N + n] : 0.0;
    const double bias = j->bias ? (double)j->bias[d] : 0.0;
    const double Dd = j->D ? (double)j->D[d] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      const int64_t x_idx = row * L + t;
      const double u = load_elem(j->u, x_idx, j->dtype);
      double dt = load_elem(j->delta, x_idx, j->dtype) + bias;
      if (j->softplus) dt = softplus(dt);
      double y = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double a_bar = exp(dt * (double)j->A[d * N + n]);
        const double b_bar = dt * load_elem(j->B, (b * N + n) * L + t, j->dtype);
        h[n] = a_bar * h[n] + b_bar * u;
        y += load_elem(j->C, (b * N + n) * L + t, j->dtype) * h[n];
      }
      y += Dd * u;
      if (j->z) y *= silu(load_elem(j->z, x_idx, j->dtype));
      j->y[x_idx] = y;
    }
    if (j->last_state)
      for (int64_t n = 0; n < N; ++n) j->last_state[row * N + n] = h[n];
  }
  free(h);
}

static void* thread_main(void* arg) {
  run_rows((oracle_job*)arg);
  return NULL;
}

/* Returns 0 on success, 1 on a bad argument, 2 on an allocation or thread
 * failure.  h0 and last_state are [b,d,N] doubles and may be NULL; D, z and
 * delta_bias may be NULL (zero skip, no gate, zero bias). */
int ss_oracle_fwd(const void* u, const void* delta, const float* A, const void* B,
                  const void* C, const float* D, const void* z, const float* delta_bias,
                  int delta_softplus, const double* h0, double* y, double* last_state,
                  int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int dtype,
                  int nthreads) {
  if (!u || !delta || !A || !B || !C || !y) return 1;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return 1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return 1;
  const int64_t rows = batch * dim;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > rows) nthreads = (int)rows;

  oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* created = (char*)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !created) {
    free(jobs);
    free(tids);
    free(created);
    return 2;
  }
  int status = 0;
  for (int i = 0; i < nthreads; ++i) {
    oracle_job* j = &jobs[i];
    j->u = u; j->delta = delta; j->A = A; j->B = B; j->C = C; j->D = D; j->z = z;
    j->bias = delta_bias; j->softplus = delta_softplus; j->h0 = h0;
    j->y = y; j->last_state = last_state;
    j->batch = batch; j->dim = dim; j->dstate = dstate; j->seqlen = seqlen;
    j->dtype = dtype;
    j->row_begin = rows * i / nthreads;
    j->row_end = rows * (i + 1) / nthreads;
    if (nthreads == 1) {
      run_rows(j);
    } else if (pthread_create(&tids[i], NULL, thread_main, j) == 0) {
      created[i] = 1;
    } else {
      run_rows(j); /* run inline if a thread cannot be created */
    }
  }
  for (int i = 0; i < nthreads; ++i)
    if (created[i]) pthread_join(tids[i], NULL);
  for (int i = 0; i < nthreads; ++i)
    if (jobs[i].status) status = jobs[i].status;
  free(jobs);
  free(tids);
  free(created);
  return status;
}

/* The associative operator of "Mamba CUDA 实现解析", section
 * "Mamba SSM并行计算", eq (10):
 *   (a1, v1) (+) (a2, c2) = (a2 * a1, a2 * v1 + c2)
 * applied elementwise over count pairs: out may alias either input. */
void ss_oracle_combine(const double* a1, const double* v1, const double* a2,
                       const double* c2, double* a_out, double* v_out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) {
    const double a = a2[i] * a1[i];
    const double v = a2[i] * v1[i] + c2[i];
    a_out[i] = a;
    v_out[i] = v;
  }
}
