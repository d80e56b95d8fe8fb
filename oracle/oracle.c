/*
 * Plain fp64 CPU oracle for the Mamba2 selective state-space recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or runs
 * this file; only the test suite, the package's smoke check and the bench's CPU
 * baseline do.  It shares no code with the CUDA library.
 *
 * What it computes (the plain definition, token by token, per head h with group
 * g(h) = h / (H/G)):
 *
 *   delta_t  = softplus(dt_t + dt_bias[h])              raw dt plus bias through
 *                                                       softplus (exact-replay RFC,
 *                                                       vLLM issue 55524, section 3)
 *   S_t      = exp(delta_t * A[h]) * S_{t-1}
 *              + delta_t * x_t (outer) B_t              state [P x N]
 *   y_t      = S_t C_t + D[h] * x_t                     output [P]
 *
 * which is the recurrence S_h = gamma S + sum gamma v k^T of the ReplaySSM
 * reproduction notes ("Core equations") with v = delta * x, k = B, q = C and
 * alpha = exp(delta * A).  All arithmetic is IEEE fp64 in program order; the
 * file must be compiled without -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* softplus(z) = log(1 + exp(z)), evaluated without overflow. */
static double softplus64(double z) {
  if (z > 0.0) return z + log1p(exp(-z));
  return log1p(exp(z));
}

typedef struct {
  int nseq, H, G, P, N;
  const int64_t* cu;     /* [nseq+1] token offsets into the packed arrays */
  const double* x;       /* [T, H, P] */
  const double* dt;      /* [T, H] raw */
  const double* A;       /* [H] */
  const double* B;       /* [T, G, N] */
  const double* C;       /* [T, G, N] */
  const double* D;       /* [H] */
  const double* dt_bias; /* [H] */
  double* state;         /* [nseq, H, P, N] in: initial state, out: final state */
  double* y;             /* [T, H, P] */
  int64_t next;          /* work counter over (seq, head) */
  pthread_mutex_t lock;
} job_t;

static void run_one(job_t* j, int s, int h) {
  const int H = j->H, G = j->G, P = j->P, N = j->N;
  const int g = h / (H / G);
  double* S = j->state + ((int64_t)s * H + h) * (int64_t)P * N;
  for (int64_t t = j->cu[s]; t < j->cu[s + 1]; ++t) {
    const double delta = softplus64(j->dt[t * H + h] + j->dt_bias[h]);
    const double decay = exp(delta * j->A[h]);
    const double* xt = j->x + (t * H + h) * P;
    const double* Bt = j->B + (t * G + g) * N;
    const double* Ct = j->C + (t * G + g) * N;
    double* yt = j->y + (t * H + h) * P;
    for (int d = 0; d < P; ++d) {
      double* Sd = S + (int64_t)d * N;
      const double v = delta * xt[d];
      double acc = 0.0;
      for (int n = 0; n < N; ++n) {
        Sd[n] = decay * Sd[n] + v * Bt[n];
        acc += Sd[n] * Ct[n];
      }
      yt[d] = acc + j->D[h] * xt[d];
    }
  }
}

static void* worker(void* arg) {
  job_t* j = (job_t*)arg;
  const int64_t total = (int64_t)j->nseq * j->H;
  for (;;) {
    pthread_mutex_lock(&j->lock);
    int64_t k = j->next++;
    pthread_mutex_unlock(&j->lock);
    if (k >= total) break;
    run_one(j, (int)(k / j->H), (int)(k % j->H));
  }
  return NULL;
}

/*
 * Runs the recurrence over nseq packed sequences (sequence s owns tokens
 * [cu[s], cu[s+1])).  state holds each sequence's initial state on entry and
 * its final state on return.  Work over (sequence, head) pairs is spread over
 * nthreads POSIX threads; each pair is computed by one thread in token order,
 * so the result does not depend on nthreads.  Returns 0 on success.
 */
int oracle_ssm_recurrence(int nseq, int H, int G, int P, int N, const int64_t* cu, const double* x,
                          const double* dt, const double* A, const double* B, const double* C,
                          const double* D, const double* dt_bias, double* state, double* y,
                          int nthreads) {
  if (nseq < 0 || H <= 0 || G <= 0 || P <= 0 || N <= 0 || H % G != 0) return 1;
  job_t j;
  memset(&j, 0, sizeof(j));
  j.nseq = nseq; j.H = H; j.G = G; j.P = P; j.N = N;
  j.cu = cu; j.x = x; j.dt = dt; j.A = A; j.B = B; j.C = C; j.D = D; j.dt_bias = dt_bias;
  j.state = state; j.y = y; j.next = 0;
  pthread_mutex_init(&j.lock, NULL);
  if (nthreads <= 1) {
    worker(&j);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return 2;
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
      if (pthread_create(&th[i], NULL, worker, &j) == 0) ++started;
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    if (started == 0) worker(&j);
    free(th);
  }
  pthread_mutex_destroy(&j.lock);
  return 0;
}

/* Exposed for the pins: fp64 softplus exactly as the recurrence uses it. */
double oracle_softplus(double z) { return softplus64(z); }
