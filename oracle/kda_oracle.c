/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the Kimi Delta Attention (KDA)
 * forward recurrence, token by token.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load this file.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it computes (per sequence s, head h; t runs over the sequence):
 *
 *   gate     g_t   = g_min * sigmoid(theta_t)            (vector over dk)
 *            -- "Architecture Deep Dive: Kimi K3's MoE, Linear Attention, and
 *               Long-Context Engineering", sec. 3.2, eq. 1 (gamma_t =
 *               gamma_min * Sigmoid(theta_t), gamma_min = -5); the same gate
 *               in "Kimi K3 Deep Dive", section "The Design" and its code
 *               snippet (log_decay = g_min * sigmoid(e)).
 *   decay    S    <- Diag(exp(g_t)) S                     (row i of S scaled)
 *   delta    S    <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T
 *   read     o_t   = S^T q_t
 *
 * i.e. S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T,
 * o_t = S_t^T q_t: the gated delta rule with channel-wise forgetting that the
 * explainer chapter "Kimi K3" (section "Across the sequence") describes as a
 * fixed-size state that each token reads, selectively forgets and writes.
 *
 * The state starts from init_state (or zero) at every sequence start.
 *
 * Layouts (row-major, all fp64):
 *   fixed length (cu_seqlens == NULL): q,k,theta [B,T,H,dk]; v,out [B,T,H,dv];
 *       beta [B,T,H]; init/final state [B,H,dk,dv].
 *   packed varlen (cu_seqlens != NULL): B = number of sequences, T = total
 *       tokens, tensors are [1,T,H,.], sequence s spans tokens
 *       [cu_seqlens[s], cu_seqlens[s+1]); states are [B,H,dk,dv].
 *
 * Flags:
 *   theta_is_g  -- nonzero: the "theta" array already holds the log-decay g
 *                  (the gate is bypassed, g_min unused).  Lets tests set g = 0.
 *   erase       -- nonzero: the delta rule above.  Zero: the erase term is
 *                  dropped, S <- Diag(exp(g)) S + beta k v^T (gated linear
 *                  attention with a per-token write weight).
 *   mutation    -- 0 in every normal use.  Nonzero values plant one known
 *                  mistake so the tests can show that the pins catch it.
 *   nthreads    -- worker threads over (sequence, head) pairs (<=0 means 1).
 *
 * Returns 0, or -1 on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
  MUT_NONE = 0,
  MUT_NO_DECAY = 1,        /* the Diag(exp(g)) step is skipped               */
  MUT_DECAY_AFTER = 2,     /* decay applied after the delta update           */
  MUT_ERASE_SIGN = 3,      /* erase term added instead of subtracted         */
  MUT_READ_BEFORE = 4,     /* o_t read from S_{t-1} instead of S_t           */
  MUT_READ_TRANSPOSED = 5, /* o_t = S q_t instead of S^T q_t (dk == dv)      */
  MUT_ERASE_NO_BETA = 6,   /* erase term missing its beta factor             */
  MUT_GATE_SIGN = 7,       /* g = g_min * sigmoid(-theta)                    */
  MUT_DECAY_CHANNEL = 8,   /* decay of channel i taken from channel dk-1-i   */
  MUT_NO_RESET = 9,        /* varlen: state carried over between sequences   */
  MUT_BETA_SHIFT = 10,     /* beta of the previous token used                */
  MUT_WRITE_KEY = 11       /* write uses q_t instead of k_t                   */
};

typedef struct {
  const double *q, *k, *v, *theta, *beta, *init_state;
  double *out, *final_state;
  const int32_t *cu_seqlens;
  double g_min;
  int B, H, T, dk, dv;
  int theta_is_g, erase, mutation;
  int64_t n_pairs;
  int64_t next;              /* next (sequence, head) pair to take          */
  pthread_mutex_t lock;
} job_t;

static double gate_one(double theta, double g_min, int mutation) {
  double x = (mutation == MUT_GATE_SIGN) ? -theta : theta;
  return g_min * (1.0 / (1.0 + exp(-x)));
}

/* One (sequence, head) pair.  S, u, a are scratch of dk*dv, dv, dk doubles. */
static void run_pair(const job_t* J, int64_t pair, double* S, double* u, double* dec) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  const int s = (int)(pair / H), h = (int)(pair % H);
  int64_t t0, t1;
  if (J->cu_seqlens) {
    t0 = J->cu_seqlens[s];
    t1 = J->cu_seqlens[s + 1];
  } else {
    t0 = (int64_t)s * J->T;
    t1 = t0 + J->T;
  }
  /* state at sequence start */
  if (J->mutation == MUT_NO_RESET && J->cu_seqlens && s > 0) {
    /* keep whatever the previous sequence of this head left (only meaningful
       when one thread runs the pairs in order; used by a single-thread test) */
  } else if (J->init_state) {
    memcpy(S, J->init_state + ((int64_t)s * H + h) * dk * dv, sizeof(double) * dk * dv);
  } else {
    memset(S, 0, sizeof(double) * dk * dv);
  }

  for (int64_t t = t0; t < t1; ++t) {
    const int64_t row = t * H + h; /* token-head row in the flattened [.,H,.] layout */
    const double* qt = J->q + row * dk;
    const double* kt = J->k + row * dk;
    const double* vt = J->v + row * dv;
    const double* th = J->theta + row * dk;
    double bt = J->beta[row];
    if (J->mutation == MUT_BETA_SHIFT && t > t0) bt = J->beta[row - H];
    double* ot = J->out + row * dv;
    const double* wkey = (J->mutation == MUT_WRITE_KEY) ? qt : kt;

    for (int i = 0; i < dk; ++i) {
      int src = (J->mutation == MUT_DECAY_CHANNEL) ? (dk - 1 - i) : i;
      double g = J->theta_is_g ? th[src] : gate_one(th[src], J->g_min, J->mutation);
      dec[i] = exp(g);
    }

    if (J->mutation == MUT_READ_BEFORE) {
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * qt[i];
        ot[j] = acc;
      }
    }

    /* decay: S <- Diag(exp(g_t)) S */
    if (J->mutation != MUT_NO_DECAY && J->mutation != MUT_DECAY_AFTER) {
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= dec[i];
    }

    if (J->erase) {
      /* u = k_t^T S (a row over dv) */
      for (int j = 0; j < dv; ++j) u[j] = 0.0;
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) u[j] += kt[i] * S[(int64_t)i * dv + j];
      double be = (J->mutation == MUT_ERASE_NO_BETA) ? 1.0 : bt;
      double sgn = (J->mutation == MUT_ERASE_SIGN) ? 1.0 : -1.0;
      /* S <- S - beta k (k^T S) + beta k v^T */
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
          S[(int64_t)i * dv + j] += sgn * be * kt[i] * u[j] + bt * wkey[i] * vt[j];
    } else {
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] += bt * wkey[i] * vt[j];
    }

    if (J->mutation == MUT_DECAY_AFTER) {
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= dec[i];
    }

    if (J->mutation == MUT_READ_BEFORE) continue;

    /* o_t = S^T q_t */
    if (J->mutation == MUT_READ_TRANSPOSED) {
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(int64_t)j * dv + i] * qt[i];
        ot[j] = acc;
      }
    } else {
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * qt[i];
        ot[j] = acc;
      }
    }
  }
  if (J->final_state)
    memcpy(J->final_state + ((int64_t)s * H + h) * dk * dv, S, sizeof(double) * dk * dv);
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  double* S = (double*)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double* u = (double*)malloc(sizeof(double) * (size_t)J->dv);
  double* dec = (double*)malloc(sizeof(double) * (size_t)J->dk);
  if (!S || !u || !dec) {
    free(S); free(u); free(dec);
    return (void*)1;
  }
  /* MUT_NO_RESET needs the pairs of one head in sequence order with the state
     carried: run them h-major so each head's sequences come one after another */
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int64_t p = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (p >= J->n_pairs) break;
    int64_t pair = p;
    if (J->mutation == MUT_NO_RESET) {
      int64_t h = p / J->B, s = p % J->B;
      pair = s * J->H + h;
    }
    run_pair(J, pair, S, u, dec);
  }
  free(S); free(u); free(dec);
  return NULL;
}

int kda_oracle_fwd_f64(const double* q, const double* k, const double* v, const double* theta,
                       const double* beta, double g_min, const double* init_state, double* out,
                       double* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                       int dk, int dv, int theta_is_g, int erase, int mutation, int nthreads) {
  if (!q || !k || !v || !theta || !beta || !out) return -1;
  if (B <= 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
  if (mutation == MUT_READ_TRANSPOSED && dk != dv) return -1;
  if (cu_seqlens) {
    if (cu_seqlens[0] != 0 || cu_seqlens[B] != T) return -1;
    for (int s = 0; s < B; ++s)
      if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
  }
  job_t J;
  J.q = q; J.k = k; J.v = v; J.theta = theta; J.beta = beta; J.init_state = init_state;
  J.out = out; J.final_state = final_state; J.cu_seqlens = cu_seqlens; J.g_min = g_min;
  J.B = B; J.H = H; J.T = T; J.dk = dk; J.dv = dv;
  J.theta_is_g = theta_is_g; J.erase = erase; J.mutation = mutation;
  J.n_pairs = (int64_t)B * H;
  J.next = 0;
  pthread_mutex_init(&J.lock, NULL);
  if (mutation == MUT_NO_RESET) nthreads = 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > J.n_pairs) nthreads = (int)J.n_pairs;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  int rc = 0;
  if (!th) return -1;
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) {
    /* no thread could be started: run inline */
    if (worker(&J) != NULL) rc = -1;
  }
  for (int i = 0; i < started; ++i) {
    void* r = NULL;
    pthread_join(th[i], &r);
    if (r != NULL) rc = -1;
  }
  free(th);
  pthread_mutex_destroy(&J.lock);
  return rc;
}

/* Elementwise gate g = g_min * sigmoid(theta) in fp64 (used by the pins). */
void kda_oracle_gate_f64(const double* theta, double g_min, int64_t n, double* g) {
  for (int64_t i = 0; i < n; ++i) g[i] = gate_one(theta[i], g_min, MUT_NONE);
}
