/*
 * gdn_oracle.c — fp64 CPU oracle for the Gated DeltaNet recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under gated_deltanet_linear_recurrence_gb300/) never calls it
 * and shares no code with it.
 *
 * What it computes.  The page "Optimizing on-device inference for Apple
 * Silicon" (section "Qwen creates three distinct workload shapes") describes
 * the Gated DeltaNet layer in words: a fixed-size matrix state per head, a
 * learned gate that keeps a fraction of the old state, and a delta update that
 * writes the current token, each token depending on the state the previous
 * token left.  The section "Keep the recurrent state on-chip" fixes the state
 * and its gate to fp32 in the engine.  The equation this file evaluates is the
 * gated delta rule that the description names, per value head h:
 *
 *     alpha_t = exp(g_t)
 *     S_t     = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t     = S_t (scale * q_t)                       (read after the update)
 *
 * S is d_v x d_k (row i = value dimension, column j = key dimension), stored
 * [seq][h_v][d_v][d_k].  Value head h reads key/query head h / (h_v / h_k).
 *
 * The oracle is the definition written out, token after token, in fp64.
 * Because (I - beta k k^T) multiplies S from the right, row i of S_t depends
 * only on row i of S_{t-1}; the product S (I - beta k k^T) is expanded for
 * each row as S_i - beta (S_i . k) k^T, which is the matrix product itself
 * (no reassociation across tokens, no blocking).  Rows are therefore
 * independent tasks and run on a pool of POSIX threads.
 *
 * Inputs are read in the storage type the GPU sees (bf16, fp32 or fp64) and
 * widened exactly to fp64 before any arithmetic.
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   - the readout is taken after the update (o_t = S_t q_t);
 *   - q is multiplied by `scale` (1 in every workload);
 *   - value heads 2j and 2j+1 (generally G*j ... G*j+G-1) share key head j;
 *   - one gate g and one write strength beta per (token, value head);
 *   - an empty sequence leaves its state unchanged and writes no output;
 *   - a NULL initial state means zeros;
 *   - with qk_l2norm set, q and k of every (token, key head) are first divided
 *     by sqrt(sum of their squares + 1e-6): the page (section "Reduce
 *     intermediate and state traffic") fuses the recurrent update with "its
 *     normalization" without giving its form, and L2 normalisation of q and k
 *     per head is the plainest reading; eps = 1e-6 is the usual choice.
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC -pthread (see oracle/build.py).
 * ORACLE_MUTANT selects a deliberately wrong variant; only the pin-strength
 * tests build it, to show that the pins catch each such mistake.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

#define QK_NORM_EPS 1e-6

enum {
  ORC_OK = 0,
  ORC_ERR_ARG = 1,
  ORC_ERR_CU_SEQLENS = 2,
  ORC_ERR_NOMEM = 3,
  ORC_ERR_THREAD = 4
};

/* Exact widening of one stored element to fp64. */
static double widen(const void* base, int dtype, int64_t idx) {
  if (dtype == ORC_F64) return ((const double*)base)[idx];
  if (dtype == ORC_F32) return (double)((const float*)base)[idx];
  /* bf16: the upper 16 bits of an IEEE binary32 */
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const void* state_in; /* may be NULL */
  int qkv_dtype;
  int f_dtype; /* dtype of g, beta, state_in */
  const int32_t* cu;
  int32_t num_seqs;
  int64_t total_tokens;
  int32_t h_k, h_v, d_k, d_v;
  double scale;
  int qk_l2norm; /* divide q and k by their L2 norm (+ eps) first */
  /* task list: (seq, head, row) triples; NULL means every row of every head */
  const int64_t* tasks;
  int64_t num_tasks;
  /* full-layout outputs (tasks == NULL) */
  double* o_full;     /* [T][h_v][d_v] */
  double* state_full; /* [N][h_v][d_v][d_k] */
  /* per-task outputs (tasks != NULL) */
  double* o_task;     /* concatenated: task j holds L(seq_j) values */
  double* state_task; /* [num_tasks][d_k] */
  const int64_t* o_task_off;
  /* work distribution */
  int64_t next; /* guarded by mu */
  pthread_mutex_t mu;
} job_t;

/* One value-row task: evaluate row i of head h of sequence n over all of the
 * sequence's tokens.  `krow` and `qrow` are scratch of d_k doubles each, `srow`
 * holds the state row.  Outputs go to o_dst[(t - t0) * o_stride] and to the
 * d_k values of the final state row at s_dst (element j at s_dst[j * s_stride]).
 *
 * The ORACLE_MUTANT branches each plant one plausible mistake; the default
 * build (ORACLE_MUTANT == 0) compiles none of them. */
static void run_row(const job_t* J, int32_t n, int32_t h, int32_t i, double* srow,
                    double* krow, double* qrow, double* o_dst, int64_t o_stride,
                    double* s_dst, int64_t s_stride) {
  const int32_t G = J->h_v / J->h_k;
#if ORACLE_MUTANT == 7 /* wrong head map: h mod h_k */
  const int32_t hk = h % J->h_k;
#else
  const int32_t hk = h / G;
#endif
  const int32_t dk = J->d_k, dv = J->d_v;
  const int64_t t0 = J->cu[n], t1 = J->cu[n + 1];
  const int64_t s_base = ((int64_t)n * J->h_v + h) * (int64_t)dv * dk;
#if ORACLE_MUTANT == 10 /* state read as [d_k][d_v] (transposed) */
  const int64_t s_row = i, s_col = dv;
#else
  const int64_t s_row = (int64_t)i * dk, s_col = 1;
#endif
#if ORACLE_MUTANT == 11 /* scale ignored */
  const double scale = 1.0;
#else
  const double scale = J->scale;
#endif
  (void)G;

  for (int32_t j = 0; j < dk; ++j)
    srow[j] = J->state_in ? widen(J->state_in, J->f_dtype, s_base + s_row + j * s_col) : 0.0;

  for (int64_t t = t0; t < t1; ++t) {
    const int64_t qk_off = (t * J->h_k + hk) * (int64_t)dk;
    const int64_t gv_off = t * J->h_v + h;
    for (int32_t j = 0; j < dk; ++j) {
      krow[j] = widen(J->k, J->qkv_dtype, qk_off + j);
      qrow[j] = widen(J->q, J->qkv_dtype, qk_off + j);
    }
#if ORACLE_MUTANT == 13
    if (J->qk_l2norm)
      for (int32_t j = 0; j < dk; ++j) qrow[j] *= scale;
#endif
    if (J->qk_l2norm) { /* k <- k / sqrt(|k|^2 + eps), the same for q */
      double kss = 0.0, qss = 0.0;
      for (int32_t j = 0; j < dk; ++j) {
        kss += krow[j] * krow[j];
        qss += qrow[j] * qrow[j];
      }
      const double kn = 1.0 / sqrt(kss + QK_NORM_EPS), qn = 1.0 / sqrt(qss + QK_NORM_EPS);
      for (int32_t j = 0; j < dk; ++j) {
        krow[j] *= kn;
#if ORACLE_MUTANT != 12 /* q left unnormalised */
        qrow[j] *= qn;
#endif
      }
#if ORACLE_MUTANT == 12
      (void)qn;
#endif
    }
#if ORACLE_MUTANT == 13 /* scale applied before the normalisation (cancels) */
    if (!J->qk_l2norm)
#endif
    for (int32_t j = 0; j < dk; ++j) qrow[j] *= scale;
    const double g = widen(J->g, J->f_dtype, gv_off);
    const double b = widen(J->beta, J->f_dtype, gv_off);
    const double vi = widen(J->v, J->qkv_dtype, (t * J->h_v + h) * (int64_t)dv + i);
#if ORACLE_MUTANT == 1 /* gate used as a factor, not exponentiated */
    const double alpha = g;
#elif ORACLE_MUTANT == 8 /* gate ignored */
    const double alpha = 1.0;
#else
    const double alpha = exp(g);
#endif

#if ORACLE_MUTANT == 6
    double o_before = 0.0;
    for (int32_t j = 0; j < dk; ++j) o_before += srow[j] * qrow[j];
#endif
#if ORACLE_MUTANT == 1 || ORACLE_MUTANT == 8
    (void)g;
#endif

    /* (S_{t-1} k_t)_i : row i of S times k */
    double sk = 0.0;
    for (int32_t j = 0; j < dk; ++j) sk += srow[j] * krow[j];

    /* S_t,i = alpha (S_{t-1,i} - beta (S_{t-1,i}.k) k^T) + beta v_i k^T */
    for (int32_t j = 0; j < dk; ++j) {
#if ORACLE_MUTANT == 2 /* dropped delta correction */
      srow[j] = alpha * srow[j] + b * vi * krow[j];
#elif ORACLE_MUTANT == 3 /* wrong sign of the correction */
      srow[j] = alpha * (srow[j] + b * sk * krow[j]) + b * vi * krow[j];
#elif ORACLE_MUTANT == 4 /* write not scaled by beta */
      srow[j] = alpha * (srow[j] - b * sk * krow[j]) + vi * krow[j];
#elif ORACLE_MUTANT == 9 /* gate applied to the write as well */
      srow[j] = alpha * (srow[j] - b * sk * krow[j] + b * vi * krow[j]);
#else
      srow[j] = alpha * (srow[j] - b * sk * krow[j]) + b * vi * krow[j];
#endif
    }

    /* o_t,i = S_t,i . q  (after the update) */
    double o = 0.0;
#if ORACLE_MUTANT == 5 /* readout with k instead of q */
    for (int32_t j = 0; j < dk; ++j) o += srow[j] * krow[j];
#elif ORACLE_MUTANT == 6 /* readout before the update */
    o = o_before;
#else
    for (int32_t j = 0; j < dk; ++j) o += srow[j] * qrow[j];
#endif
    o_dst[(t - t0) * o_stride] = o;
  }
  for (int32_t j = 0; j < dk; ++j) s_dst[j * s_stride] = srow[j];
}

static void decode_task(const job_t* J, int64_t idx, int32_t* n, int32_t* h, int32_t* i) {
  if (J->tasks) {
    *n = (int32_t)J->tasks[3 * idx + 0];
    *h = (int32_t)J->tasks[3 * idx + 1];
    *i = (int32_t)J->tasks[3 * idx + 2];
  } else {
    const int64_t per_seq = (int64_t)J->h_v * J->d_v;
    *n = (int32_t)(idx / per_seq);
    *h = (int32_t)((idx % per_seq) / J->d_v);
    *i = (int32_t)(idx % J->d_v);
  }
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  double* buf = (double*)malloc(sizeof(double) * 3 * (size_t)J->d_k);
  if (!buf) return (void*)1;
  double *srow = buf, *krow = buf + J->d_k, *qrow = buf + 2 * J->d_k;
  const int64_t total =
      J->tasks ? J->num_tasks : (int64_t)J->num_seqs * J->h_v * J->d_v;
  const int64_t grab = 8;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t start = J->next;
    J->next += grab;
    pthread_mutex_unlock(&J->mu);
    if (start >= total) break;
    int64_t stop = start + grab < total ? start + grab : total;
    for (int64_t idx = start; idx < stop; ++idx) {
      int32_t n, h, i;
      decode_task(J, idx, &n, &h, &i);
      if (J->tasks) {
        run_row(J, n, h, i, srow, krow, qrow, J->o_task + J->o_task_off[idx], 1,
                J->state_task + idx * J->d_k, 1);
      } else {
        const int64_t t0 = J->cu[n];
        const int64_t s_base = ((int64_t)n * J->h_v + h) * (int64_t)J->d_v * J->d_k;
#if ORACLE_MUTANT == 10
        double* s_dst = J->state_full + s_base + i;
        const int64_t s_stride = J->d_v;
#else
        double* s_dst = J->state_full + s_base + (int64_t)i * J->d_k;
        const int64_t s_stride = 1;
#endif
        run_row(J, n, h, i, srow, krow, qrow,
                J->o_full + (t0 * J->h_v + h) * (int64_t)J->d_v + i,
                (int64_t)J->h_v * J->d_v, s_dst, s_stride);
      }
    }
  }
  free(buf);
  return NULL;
}

static int check_common(const job_t* J) {
  if (!J->q || !J->k || !J->v || !J->g || !J->beta || !J->cu) return ORC_ERR_ARG;
  if (J->num_seqs < 0 || J->total_tokens < 0) return ORC_ERR_ARG;
  if (J->h_k <= 0 || J->h_v <= 0 || J->d_k <= 0 || J->d_v <= 0) return ORC_ERR_ARG;
  if (J->d_k > 4096) return ORC_ERR_ARG;
  if (J->h_v % J->h_k != 0) return ORC_ERR_ARG;
  if (J->qkv_dtype < ORC_F64 || J->qkv_dtype > ORC_BF16) return ORC_ERR_ARG;
  if (J->f_dtype != ORC_F64 && J->f_dtype != ORC_F32) return ORC_ERR_ARG;
  if (J->cu[0] != 0) return ORC_ERR_CU_SEQLENS;
  for (int32_t n = 0; n < J->num_seqs; ++n)
    if (J->cu[n + 1] < J->cu[n]) return ORC_ERR_CU_SEQLENS;
  if ((int64_t)J->cu[J->num_seqs] != J->total_tokens) return ORC_ERR_CU_SEQLENS;
  return ORC_OK;
}

static int run_pool(job_t* J, int32_t threads) {
  if (threads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    threads = c > 0 ? (int32_t)c : 1;
  }
  if (threads > 1024) threads = 1024;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
  if (!th) return ORC_ERR_NOMEM;
  J->next = 0;
  pthread_mutex_init(&J->mu, NULL);
  int started = 0, rc = ORC_OK;
  for (int32_t w = 0; w < threads; ++w) {
    if (pthread_create(&th[w], NULL, worker, J) != 0) {
      rc = ORC_ERR_THREAD;
      break;
    }
    ++started;
  }
  for (int w = 0; w < started; ++w) {
    void* ret = NULL;
    pthread_join(th[w], &ret);
    if (ret) rc = ORC_ERR_NOMEM;
  }
  pthread_mutex_destroy(&J->mu);
  free(th);
  return rc;
}

/* Number of threads a call with threads <= 0 uses. */
int gdn_oracle_default_threads(void) {
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

/*
 * Full evaluation.  o_out: [T][h_v][d_v] fp64 (rows of empty sequences are not
 * touched); state_out: [N][h_v][d_v][d_k] fp64.  Returns 0 or an ORC_ERR code.
 */
int gdn_oracle_prefill(int qkv_dtype, int f_dtype, const void* q, const void* k,
                       const void* v, const void* g, const void* beta,
                       const void* state_in, const int32_t* cu_seqlens,
                       int32_t num_seqs, int64_t total_tokens, int32_t h_k,
                       int32_t h_v, int32_t d_k, int32_t d_v, double scale, int qk_l2norm,
                       double* o_out, double* state_out, int32_t threads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.state_in = state_in;
  J.qkv_dtype = qkv_dtype; J.f_dtype = f_dtype; J.cu = cu_seqlens;
  J.num_seqs = num_seqs; J.total_tokens = total_tokens;
  J.h_k = h_k; J.h_v = h_v; J.d_k = d_k; J.d_v = d_v; J.scale = scale;
  J.qk_l2norm = qk_l2norm;
  J.o_full = o_out; J.state_full = state_out;
  int rc = check_common(&J);
  if (rc) return rc;
  if (!o_out || !state_out) return ORC_ERR_ARG;
  return run_pool(&J, threads);
}

/*
 * Sampled evaluation of selected value rows: tasks holds num_tasks triples
 * (seq, value head, row).  Task j writes the L(seq_j) outputs o[t, h, row]
 * for the sequence's tokens in order to o_out + o_off[j], and its final state
 * row (d_k values) to state_out + j * d_k.
 */
int gdn_oracle_rows(int qkv_dtype, int f_dtype, const void* q, const void* k,
                    const void* v, const void* g, const void* beta,
                    const void* state_in, const int32_t* cu_seqlens,
                    int32_t num_seqs, int64_t total_tokens, int32_t h_k, int32_t h_v,
                    int32_t d_k, int32_t d_v, double scale, int qk_l2norm,
                    const int64_t* tasks,
                    int64_t num_tasks, const int64_t* o_off, double* o_out,
                    double* state_out, int32_t threads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.state_in = state_in;
  J.qkv_dtype = qkv_dtype; J.f_dtype = f_dtype; J.cu = cu_seqlens;
  J.num_seqs = num_seqs; J.total_tokens = total_tokens;
  J.h_k = h_k; J.h_v = h_v; J.d_k = d_k; J.d_v = d_v; J.scale = scale;
  J.qk_l2norm = qk_l2norm;
  J.tasks = tasks; J.num_tasks = num_tasks; J.o_task = o_out;
  J.state_task = state_out; J.o_task_off = o_off;
  int rc = check_common(&J);
  if (rc) return rc;
  if (!tasks || !o_off || !o_out || !state_out || num_tasks < 0) return ORC_ERR_ARG;
  for (int64_t j = 0; j < num_tasks; ++j) {
    if (tasks[3 * j] < 0 || tasks[3 * j] >= num_seqs) return ORC_ERR_ARG;
    if (tasks[3 * j + 1] < 0 || tasks[3 * j + 1] >= h_v) return ORC_ERR_ARG;
    if (tasks[3 * j + 2] < 0 || tasks[3 * j + 2] >= d_v) return ORC_ERR_ARG;
  }
  return run_pool(&J, threads);
}
