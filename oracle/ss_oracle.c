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
 * Inputs are read in the ABI layouts (u/delta/z [b,d,L], B/C [b,N,L] or, for
 * ss_oracle_fwd_pc, [b,d,N,L], A [d,N], D and bias [d]); dtype 0 means float32 values, dtype 1 means
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
  int bc_per_channel; /* B, C are [b,d,N,L] (one row per channel) instead of [b,N,L] */
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
    const int64_t bc = j->bc_per_channel ? row : b;  /* B/C row of this channel */
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
        const double b_bar = dt * load_elem(j->B, (bc * N + n) * L + t, j->dtype);
        h[n] = a_bar * h[n] + b_bar * u;
        y += load_elem(j->C, (bc * N + n) * L + t, j->dtype) * h[n];
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
 * delta_bias may be NULL (zero skip, no gate, zero bias).  bc_per_channel:
 * B and C are [b,d,N,L], one row per channel (the task spec's kernel sketch
 * layout), instead of [b,N,L] shared by the channels of a batch row. */
static int oracle_fwd_impl(const void* u, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* delta_bias, int delta_softplus, const double* h0,
                           double* y, double* last_state, int64_t batch, int64_t dim,
                           int64_t dstate, int64_t seqlen, int dtype, int nthreads,
                           int bc_per_channel) {
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
    j->bc_per_channel = bc_per_channel;
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

int ss_oracle_fwd(const void* u, const void* delta, const float* A, const void* B,
                  const void* C, const float* D, const void* z, const float* delta_bias,
                  int delta_softplus, const double* h0, double* y, double* last_state,
                  int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int dtype,
                  int nthreads) {
  return oracle_fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, last_state,
                         batch, dim, dstate, seqlen, dtype, nthreads, 0);
}

/* The forward with B and C given per channel, [b,d,N,L]. */
int ss_oracle_fwd_pc(const void* u, const void* delta, const float* A, const void* B,
                     const void* C, const float* D, const void* z, const float* delta_bias,
                     int delta_softplus, const double* h0, double* y, double* last_state,
                     int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int dtype,
                     int nthreads) {
  return oracle_fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, last_state,
                         batch, dim, dstate, seqlen, dtype, nthreads, 1);
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

/* ---------------------------------------------------------------------------
 * Backward pass: the exact derivative of ss_oracle_fwd, in reverse mode.
 *
 * The pages ask for a backward checked with gradcheck ("ТЕХНИЧЕСКОЕ ЗАДАНИЕ:
 * Реализовать selective scan (Mamba)", Этап 3 step 4 and section 5, the
 * acceptance criteria; the Blelloch article, section 5.3, a custom backward
 * for autograd) but print no formulas for it.  What follows is the chain rule
 * applied to the forward definition above, for a loss whose gradient with
 * respect to y is dy (and, optionally, to last_state is dlast):
 *   gate:     dy'_t = dy_t * silu(z_t),  dz_t = dy_t * y'_t * silu'(z_t)
 *             silu'(z) = s (1 + z (1 - s)), s = 1 / (1 + e^-z)
 *   skip:     dD += dy'_t u_t,  du_t += dy'_t D
 *   read-out: dC[n,t] += dy'_t h_t[n];  g_t[n] = C[n,t] dy'_t + a_{t+1}[n] g_{t+1}[n]
 *             (g_t = dL/dh_t; g after the last step is dlast)
 *   update h_t = a_t h_{t-1} + dt_t B[n,t] u_t with a_t = exp(dt_t A[n]):
 *             d(dt_t) += g_t[n] (A[n] a_t h_{t-1}[n] + B[n,t] u_t)
 *             dA[n]   += g_t[n] dt_t a_t h_{t-1}[n]
 *             dB[n,t] += g_t[n] dt_t u_t,   du_t += g_t[n] dt_t B[n,t]
 *   step:     dx_t = d(dt_t) * (softplus ? sigmoid(x_t) : 1), x_t = delta_t + bias;
 *             ddelta_t = dx_t, dbias += dx_t
 *   initial:  dh0[n] = a_0[n] g_0[n]
 * The forward states are recomputed and kept for the whole row.  Gradients of
 * inputs shared between rows (dA, dB, dC, dD, dbias) are summed per thread and
 * the per-thread sums added in thread order, so the result is deterministic.
 * All outputs are double.  Optional outputs (dD, dz, dbias, dh0) may be NULL.
 * ------------------------------------------------------------------------- */
typedef struct {
  const oracle_job* fwd;        /* inputs, sizes, dtype */
  const void* dy;
  const double* dlast;
  double *du, *ddelta, *dz, *dh0;
  double *dA, *dB, *dC, *dD, *dbias;  /* this thread's partial sums (zeroed) */
  int status;
} oracle_bwd_job;

static void bwd_rows(oracle_bwd_job* j) {
  const oracle_job* f = j->fwd;
  const int64_t N = f->dstate, L = f->seqlen, dim = f->dim;
  double* h = (double*)malloc(sizeof(double) * (size_t)(N * L));
  double* a = (double*)malloc(sizeof(double) * (size_t)(N * L));
  double* ypre = (double*)malloc(sizeof(double) * (size_t)L);
  double* dtv = (double*)malloc(sizeof(double) * (size_t)L);
  double* xv = (double*)malloc(sizeof(double) * (size_t)L);
  double* g = (double*)malloc(sizeof(double) * (size_t)N);
  if (!h || !a || !ypre || !dtv || !xv || !g) {
    j->status = 2;
    free(h); free(a); free(ypre); free(dtv); free(xv); free(g);
    return;
  }
  for (int64_t row = f->row_begin; row < f->row_end; ++row) {
    const int64_t d = row % dim, b = row / dim;
    const double bias = f->bias ? (double)f->bias[d] : 0.0;
    const double Dd = f->D ? (double)f->D[d] : 0.0;
    /* forward, keeping every state */
    for (int64_t t = 0; t < L; ++t) {
      const int64_t xi = row * L + t;
      const double u = load_elem(f->u, xi, f->dtype);
      const double x = load_elem(f->delta, xi, f->dtype) + bias;
      const double dt = f->softplus ? softplus(x) : x;
      xv[t] = x;
      dtv[t] = dt;
      double yp = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double prev = t > 0 ? h[(t - 1) * N + n] : (f->h0 ? f->h0[row * N + n] : 0.0);
        const double an = exp(dt * (double)f->A[d * N + n]);
        const double hn = an * prev + dt * load_elem(f->B, (b * N + n) * L + t, f->dtype) * u;
        a[t * N + n] = an;
        h[t * N + n] = hn;
        yp += load_elem(f->C, (b * N + n) * L + t, f->dtype) * hn;
      }
      ypre[t] = yp + Dd * u;
    }
    /* reverse */
    for (int64_t n = 0; n < N; ++n) g[n] = j->dlast ? j->dlast[row * N + n] : 0.0;
    double dD = 0.0, dbias = 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
      const int64_t xi = row * L + t;
      const double u = load_elem(f->u, xi, f->dtype);
      const double dy = load_elem(j->dy, xi, f->dtype);
      double dyp = dy;
      if (f->z) {
        const double zt = load_elem(f->z, xi, f->dtype);
        const double s = 1.0 / (1.0 + exp(-zt));
        dyp = dy * zt * s;
        if (j->dz) j->dz[xi] = dy * ypre[t] * s * (1.0 + zt * (1.0 - s));
      }
      dD += dyp * u;
      double du = dyp * Dd, ddt = 0.0;
      const double dt = dtv[t];
      for (int64_t n = 0; n < N; ++n) {
        const double Bn = load_elem(f->B, (b * N + n) * L + t, f->dtype);
        const double Cn = load_elem(f->C, (b * N + n) * L + t, f->dtype);
        const double gn = Cn * dyp + g[n];              /* g[n] holds a_{t+1} g_{t+1} */
        const double prev = t > 0 ? h[(t - 1) * N + n] : (f->h0 ? f->h0[row * N + n] : 0.0);
        const double an = a[t * N + n];
        const double An = (double)f->A[d * N + n];
        j->dC[(b * N + n) * L + t] += dyp * h[t * N + n];
        j->dB[(b * N + n) * L + t] += gn * dt * u;
        j->dA[d * N + n] += gn * dt * an * prev;
        ddt += gn * (An * an * prev + Bn * u);
        du += gn * dt * Bn;
        g[n] = an * gn;
      }
      const double dx = f->softplus ? ddt / (1.0 + exp(-xv[t])) : ddt;
      j->ddelta[xi] = dx;
      j->du[xi] = du;
      dbias += dx;
    }
    if (j->dD) j->dD[d] += dD;
    if (j->dbias) j->dbias[d] += dbias;
    if (j->dh0)
      for (int64_t n = 0; n < N; ++n) j->dh0[row * N + n] = g[n];
  }
  free(h); free(a); free(ypre); free(dtv); free(xv); free(g);
}

static void* bwd_thread_main(void* arg) {
  bwd_rows((oracle_bwd_job*)arg);
  return NULL;
}

/* Returns 0 on success, 1 on a bad argument, 2 on an allocation or thread
 * failure.  Inputs as for ss_oracle_fwd plus dy (dtype, [b,d,L]) and dlast
 * (double [b,d,N] or NULL).  Outputs (double): du, ddelta [b,d,L]; dA [d,N];
 * dB, dC [b,N,L]; dD, dbias [d] (may be NULL); dz [b,d,L] (NULL when z is
 * NULL); dh0 [b,d,N] (may be NULL). */
int ss_oracle_bwd(const void* u, const void* delta, const float* A, const void* B,
                  const void* C, const float* D, const void* z, const float* delta_bias,
                  int delta_softplus, const double* h0, const void* dy, const double* dlast,
                  double* du, double* ddelta, double* dA, double* dB, double* dC, double* dD,
                  double* dz, double* dbias, double* dh0, int64_t batch, int64_t dim,
                  int64_t dstate, int64_t seqlen, int dtype, int nthreads) {
  if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC) return 1;
  if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen <= 0) return 1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return 1;
  const int64_t rows = batch * dim;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > rows) nthreads = (int)rows;
  const size_t nA = (size_t)(dim * dstate), nBC = (size_t)(batch * dstate * seqlen);
  const size_t per = nA + 2 * nBC + 2 * (size_t)dim;

  oracle_job* fj = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
  oracle_bwd_job* bj = (oracle_bwd_job*)calloc((size_t)nthreads, sizeof(oracle_bwd_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* created = (char*)calloc((size_t)nthreads, 1);
  double* partial = (double*)calloc((size_t)nthreads * per, sizeof(double));
  int status = 0;
  if (!fj || !bj || !tids || !created || !partial) {
    status = 2;
    goto done;
  }
  for (int i = 0; i < nthreads; ++i) {
    oracle_job* f = &fj[i];
    f->u = u; f->delta = delta; f->A = A; f->B = B; f->C = C; f->D = D; f->z = z;
    f->bias = delta_bias; f->softplus = delta_softplus; f->h0 = h0;
    f->batch = batch; f->dim = dim; f->dstate = dstate; f->seqlen = seqlen; f->dtype = dtype;
    f->row_begin = rows * i / nthreads;
    f->row_end = rows * (i + 1) / nthreads;
    oracle_bwd_job* j = &bj[i];
    double* base = partial + (size_t)i * per;
    j->fwd = f; j->dy = dy; j->dlast = dlast;
    j->du = du; j->ddelta = ddelta; j->dz = z ? dz : NULL; j->dh0 = dh0;
    j->dA = base; j->dB = base + nA; j->dC = base + nA + nBC;
    j->dD = D ? base + nA + 2 * nBC : NULL;
    j->dbias = delta_bias ? base + nA + 2 * nBC + dim : NULL;
    if (nthreads == 1) {
      bwd_rows(j);
    } else if (pthread_create(&tids[i], NULL, bwd_thread_main, j) == 0) {
      created[i] = 1;
    } else {
      bwd_rows(j);
    }
  }
  for (int i = 0; i < nthreads; ++i)
    if (created[i]) pthread_join(tids[i], NULL);
  for (int i = 0; i < nthreads; ++i)
    if (bj[i].status) status = bj[i].status;
  if (status == 0) {
    /* per-thread sums, added in thread order */
    memset(dA, 0, sizeof(double) * nA);
    memset(dB, 0, sizeof(double) * nBC);
    memset(dC, 0, sizeof(double) * nBC);
    if (dD) memset(dD, 0, sizeof(double) * (size_t)dim);
    if (dbias) memset(dbias, 0, sizeof(double) * (size_t)dim);
    for (int i = 0; i < nthreads; ++i) {
      const double* base = partial + (size_t)i * per;
      for (size_t k = 0; k < nA; ++k) dA[k] += base[k];
      for (size_t k = 0; k < nBC; ++k) dB[k] += base[nA + k];
      for (size_t k = 0; k < nBC; ++k) dC[k] += base[nA + nBC + k];
      if (dD)
        for (int64_t k = 0; k < dim; ++k) dD[k] += D ? base[nA + 2 * nBC + k] : 0.0;
      if (dbias)
        for (int64_t k = 0; k < dim; ++k)
          dbias[k] += delta_bias ? base[nA + 2 * nBC + dim + k] : 0.0;
    }
  }
done:
  free(fj); free(bj); free(tids); free(created); free(partial);
  return status;
}

/* ---------------------------------------------------------------------------
 * Mamba-2 forward (one scalar decay per head), the recurrence that the Mamba-2
 * cuTile news page ("Прорыв в оптимизации SSM-моделей", section
 * "Технические детали оптимизации") writes for the state of a head:
 *
 *   h_t = exp(A * dt_t) * h_{t-1} + dt_t * B_t * x_t
 *
 * with h the head's state [P, N] (P = head dim, N = dstate), x_t [P] the
 * head's slice of token t, B_t and C_t [N] the token's rows for the head's
 * group, and the read-out with the skip connection that the page's
 * compute_out kernel fuses:
 *
 *   y_t[p] = sum_n C_t[n] * h_t[p,n] + D * x_t[p]
 *
 * dt_t = softplus(dt[b,t,h] + dt_bias[h]) when dt_softplus is set, else
 * dt + bias.  The state starts at zero (or at h0, ss_oracle_ssd_h0).  Layouts: x, y [b,L,H,P]; dt [b,L,H];
 * B, C [b,L,G,N] (head h reads group h / (H/G)); A, D, dt_bias [H];
 * final_state [b,H,P,N].  Units (b, h) are independent and are split over
 * the threads.
 */
typedef struct {
  const void* x;
  const void* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const float* bias;
  int softplus;
  const double* h0;
  double* y;
  double* final_state;
  int64_t batch, seqlen, nheads, headdim, ngroups, dstate;
  int dtype;
  int64_t unit_begin, unit_end;
  int status;
} oracle_ssd_job;

static void ssd_units(oracle_ssd_job* j) {
  const int64_t L = j->seqlen, H = j->nheads, P = j->headdim, G = j->ngroups, N = j->dstate;
  double* h = (double*)malloc(sizeof(double) * (size_t)(P * N));
  if (!h) {
    j->status = 2;
    return;
  }
  for (int64_t unit = j->unit_begin; unit < j->unit_end; ++unit) {
    const int64_t b = unit / H, hd = unit % H;
    const int64_t g = hd / (H / G);  /* the head's group */
    for (int64_t i = 0; i < P * N; ++i) h[i] = j->h0 ? j->h0[unit * P * N + i] : 0.0;
    const double A = (double)j->A[hd];
    const double bias = j->bias ? (double)j->bias[hd] : 0.0;
    const double Dh = j->D ? (double)j->D[hd] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
      double dt = load_elem(j->dt, (b * L + t) * H + hd, j->dtype) + bias;
      if (j->softplus) dt = softplus(dt);
      const double decay = exp(A * dt);
      const int64_t xrow = ((b * L + t) * H + hd) * P;   /* x_t, y_t of this head */
      const int64_t bcrow = ((b * L + t) * G + g) * N;   /* B_t, C_t of its group */
      for (int64_t p = 0; p < P; ++p) {
        const double xp = load_elem(j->x, xrow + p, j->dtype);
        double y = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          h[p * N + n] = decay * h[p * N + n] + dt * load_elem(j->B, bcrow + n, j->dtype) * xp;
          y += load_elem(j->C, bcrow + n, j->dtype) * h[p * N + n];
        }
        j->y[xrow + p] = y + Dh * xp;
      }
    }
    if (j->final_state)
      for (int64_t i = 0; i < P * N; ++i) j->final_state[unit * P * N + i] = h[i];
  }
  free(h);
}

static void* ssd_thread_main(void* arg) {
  ssd_units((oracle_ssd_job*)arg);
  return NULL;
}

/* Returns 0 on success, 1 on a bad argument (a null required pointer, a size
 * <= 0, nheads not a multiple of ngroups, an unknown dtype), 2 on an
 * allocation failure.  y is [b,L,H,P] doubles; final_state [b,H,P,N] doubles
 * or NULL; D and dt_bias may be NULL (no skip, zero bias). */
int ss_oracle_ssd_h0(const void* x, const void* dt, const float* A, const void* B,
                     const void* C, const float* D, const float* dt_bias, int dt_softplus,
                     const double* h0, double* y, double* final_state, int64_t batch,
                     int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                     int64_t dstate, int dtype, int nthreads);

int ss_oracle_ssd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                  const float* D, const float* dt_bias, int dt_softplus, double* y,
                  double* final_state, int64_t batch, int64_t seqlen, int64_t nheads,
                  int64_t headdim, int64_t ngroups, int64_t dstate, int dtype, int nthreads) {
  return ss_oracle_ssd_h0(x, dt, A, B, C, D, dt_bias, dt_softplus, NULL, y, final_state, batch,
                          seqlen, nheads, headdim, ngroups, dstate, dtype, nthreads);
}

/* The same from a given state h0 [b,H,P,N] (doubles; NULL: zero): the state
 * before the first step, as for a sequence that continues an earlier one. */
int ss_oracle_ssd_h0(const void* x, const void* dt, const float* A, const void* B,
                     const void* C, const float* D, const float* dt_bias, int dt_softplus,
                     const double* h0, double* y, double* final_state, int64_t batch,
                     int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                     int64_t dstate, int dtype, int nthreads) {
  if (!x || !dt || !A || !B || !C || !y) return 1;
  if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0)
    return 1;
  if (nheads % ngroups != 0) return 1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return 1;
  const int64_t units = batch * nheads;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > units) nthreads = (int)units;
  oracle_ssd_job* jobs = (oracle_ssd_job*)calloc((size_t)nthreads, sizeof(oracle_ssd_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* created = (char*)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !created) {
    free(jobs);
    free(tids);
    free(created);
    return 2;
  }
  for (int i = 0; i < nthreads; ++i) {
    oracle_ssd_job* j = &jobs[i];
    j->x = x; j->dt = dt; j->A = A; j->B = B; j->C = C; j->D = D; j->bias = dt_bias;
    j->softplus = dt_softplus; j->h0 = h0; j->y = y; j->final_state = final_state;
    j->batch = batch; j->seqlen = seqlen; j->nheads = nheads; j->headdim = headdim;
    j->ngroups = ngroups; j->dstate = dstate; j->dtype = dtype;
    j->unit_begin = units * i / nthreads;
    j->unit_end = units * (i + 1) / nthreads;
    if (nthreads == 1) {
      ssd_units(j);
    } else if (pthread_create(&tids[i], NULL, ssd_thread_main, j) == 0) {
      created[i] = 1;
    } else {
      ssd_units(j);
    }
  }
  int status = 0;
  for (int i = 0; i < nthreads; ++i)
    if (created[i]) pthread_join(tids[i], NULL);
  for (int i = 0; i < nthreads; ++i)
    if (jobs[i].status) status = jobs[i].status;
  free(jobs);
  free(tids);
  free(created);
  return status;
}
