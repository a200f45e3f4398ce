/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA)
 * recurrence.  TEST INFRASTRUCTURE ONLY: the GPU library never links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (the gated delta rule with per-channel decay, as stated for
 * KDA in "Kimi K3 on vLLM: Up to 370 Tokens/sec", section "Kimi Delta
 * Attention: a hybrid recurrent + full-attention stack", and in "Kimi K3 +
 * vLLM: Inside the Day-0 Production Integration", section "Kimi Delta
 * Attention: When Prefix Caching Meets Recurrent State": a fixed-size
 * matrix-valued recurrent state per sequence and head):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * with S in R^{dk x dv}.  It is evaluated token by token in the equivalent
 * order
 *     S'  = Diag(exp g_t) S_{t-1}        (row i scaled by exp g_{t,i})
 *     u   = beta_t (v_t - S'^T k_t)
 *     S_t = S' + k_t u^T
 *     o_t = S_t^T q_t
 * which is the same matrix: with S' = Diag(exp g_t) S_{t-1},
 * (I - b k k^T) S' + b k v^T = S' - k (b S'^T k)^T + k (b v)^T = S' + k u^T.
 *
 * Snapshots (the per-prefix state checkpoints of the hybrid prefix cache,
 * "Separating Physical Blocks, Scheduler Alignment, and Prefix Matching"):
 * snapshot j of a sequence is the state after (j+1)*snap_interval tokens of
 * that sequence's segment, stored densely in sequence-major order.
 *
 * Columns of S evolve independently (every operation above acts on each
 * column j of S with the same row-side vectors), so the work is split into
 * independent (sequence, head, column block) units over plain pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_COL_BLOCK 16

typedef struct {
  const double *q, *k, *v, *g, *beta; /* [T][H][dk], v: [T][H][dv], beta: [T][H] */
  const int64_t *cu;                  /* [B+1] token offsets */
  int32_t B, H, dk, dv;
  const double *init;                 /* [B][H][dk][dv] or NULL (zero state) */
  int32_t snap_interval;              /* 0: no snapshots */
  const int64_t *snap_off;            /* [B] first snapshot index per sequence */
  double *out;                        /* [T][H][dv] or NULL */
  double *final_states;               /* [B][H][dk][dv] or NULL */
  double *snaps;                      /* [n_snaps][H][dk][dv] or NULL */
  int no_delta;                       /* test hook: u = v (ungated linear attention) */
  const int32_t *unit_mask;           /* [B*H] nonzero = compute, or NULL = all */
  int32_t col_lo, col_hi;             /* column range to compute */
  int64_t n_units;
  int64_t next;                       /* shared work counter */
} oracle_job;

static void run_unit(const oracle_job *J, int64_t unit) {
  const int32_t ncb = (J->col_hi - J->col_lo + ORACLE_COL_BLOCK - 1) / ORACLE_COL_BLOCK;
  const int64_t bh = unit / ncb;
  const int32_t cb = (int32_t)(unit % ncb);
  const int32_t b = (int32_t)(bh / J->H), h = (int32_t)(bh % J->H);
  if (J->unit_mask && !J->unit_mask[bh]) return;
  const int32_t dk = J->dk, dv = J->dv, H = J->H;
  const int32_t j0 = J->col_lo + cb * ORACLE_COL_BLOCK;
  const int32_t j1 = (j0 + ORACLE_COL_BLOCK < J->col_hi) ? j0 + ORACLE_COL_BLOCK : J->col_hi;
  const int32_t nc = j1 - j0;

  double S[128 * ORACLE_COL_BLOCK];
  double x[ORACLE_COL_BLOCK], u[ORACLE_COL_BLOCK];
  for (int32_t i = 0; i < dk; ++i)
    for (int32_t c = 0; c < nc; ++c)
      S[i * ORACLE_COL_BLOCK + c] =
          J->init ? J->init[(((int64_t)b * H + h) * dk + i) * dv + j0 + c] : 0.0;

  const int64_t t0 = J->cu[b], t1 = J->cu[b + 1];
  for (int64_t t = t0; t < t1; ++t) {
    const double *qt = J->q + (t * H + h) * dk;
    const double *kt = J->k + (t * H + h) * dk;
    const double *gt = J->g + (t * H + h) * dk;
    const double *vt = J->v + (t * H + h) * dv;
    const double bt = J->beta[t * H + h];
    /* S' = Diag(exp g) S */
    for (int32_t i = 0; i < dk; ++i) {
      const double a = exp(gt[i]);
      for (int32_t c = 0; c < nc; ++c) S[i * ORACLE_COL_BLOCK + c] *= a;
    }
    /* x = S'^T k */
    for (int32_t c = 0; c < nc; ++c) x[c] = 0.0;
    for (int32_t i = 0; i < dk; ++i)
      for (int32_t c = 0; c < nc; ++c) x[c] += S[i * ORACLE_COL_BLOCK + c] * kt[i];
    /* u = beta (v - x) ; the no_delta hook drops the correction: u = v */
    for (int32_t c = 0; c < nc; ++c) u[c] = J->no_delta ? vt[j0 + c] : bt * (vt[j0 + c] - x[c]);
    /* S = S' + k u^T */
    for (int32_t i = 0; i < dk; ++i)
      for (int32_t c = 0; c < nc; ++c) S[i * ORACLE_COL_BLOCK + c] += kt[i] * u[c];
    /* o = S^T q */
    if (J->out) {
      for (int32_t c = 0; c < nc; ++c) {
        double acc = 0.0;
        for (int32_t i = 0; i < dk; ++i) acc += S[i * ORACLE_COL_BLOCK + c] * qt[i];
        J->out[(t * H + h) * dv + j0 + c] = acc;
      }
    }
    /* snapshot after every snap_interval tokens of this segment */
    const int64_t done = t - t0 + 1;
    if (J->snaps && J->snap_interval > 0 && done % J->snap_interval == 0) {
      const int64_t s = J->snap_off[b] + done / J->snap_interval - 1;
      double *dst = J->snaps + (s * H + h) * (int64_t)dk * dv;
      for (int32_t i = 0; i < dk; ++i)
        for (int32_t c = 0; c < nc; ++c) dst[(int64_t)i * dv + j0 + c] = S[i * ORACLE_COL_BLOCK + c];
    }
  }
  if (J->final_states) {
    double *dst = J->final_states + ((int64_t)b * H + h) * (int64_t)dk * dv;
    for (int32_t i = 0; i < dk; ++i)
      for (int32_t c = 0; c < nc; ++c) dst[(int64_t)i * dv + j0 + c] = S[i * ORACLE_COL_BLOCK + c];
  }
}

static void *worker(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  for (;;) {
    const int64_t unit = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (unit >= J->n_units) break;
    run_unit(J, unit);
  }
  return NULL;
}

/*
 * Runs the recurrence for every (sequence, head) whose unit_mask entry is
 * nonzero (all when unit_mask is NULL), for state columns [col_lo, col_hi).
 * Returns 0, or -1 on a bad argument.  Outputs for masked-out units or
 * columns are left untouched.
 */
int kda_oracle_run(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const int64_t *cu_seqlens, int32_t B, int32_t H,
                   int32_t dk, int32_t dv, const double *init_states, int32_t snap_interval,
                   const int64_t *snap_off, double *out, double *final_states, double *snaps,
                   int32_t no_delta, const int32_t *unit_mask, int32_t col_lo, int32_t col_hi,
                   int32_t nthreads) {
  if (B < 0 || H <= 0 || dk <= 0 || dk > 128 || dv <= 0 || col_lo < 0 || col_hi > dv ||
      col_lo >= col_hi || snap_interval < 0)
    return -1;
  if (snaps && (snap_interval == 0 || !snap_off)) return -1;
  for (int32_t b = 0; b < B; ++b)
    if (cu_seqlens[b + 1] < cu_seqlens[b]) return -1;
  oracle_job J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
  J.cu = cu_seqlens; J.B = B; J.H = H; J.dk = dk; J.dv = dv;
  J.init = init_states; J.snap_interval = snap_interval; J.snap_off = snap_off;
  J.out = out; J.final_states = final_states; J.snaps = snaps;
  J.no_delta = no_delta; J.unit_mask = unit_mask; J.col_lo = col_lo; J.col_hi = col_hi;
  const int32_t ncb = (col_hi - col_lo + ORACLE_COL_BLOCK - 1) / ORACLE_COL_BLOCK;
  J.n_units = (int64_t)B * H * ncb;
  J.next = 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads == 1 || J.n_units <= 1) {
    worker(&J);
    return 0;
  }
  pthread_t th[256];
  int32_t started = 0;
  for (int32_t i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) worker(&J);
  for (int32_t i = 0; i < started; ++i) pthread_join(th[i], NULL);
  return 0;
}
