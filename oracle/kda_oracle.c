/*
 * KDA oracle: a plain, slow, fp64 CPU implementation of the Kimi Delta
 * Attention (KDA) gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check in
 * __graft_entry__.py and the CPU-baseline leg of bench.py load this library.
 * The CUDA library shares no code, header, table or helper with it.
 *
 * Cited page: "Kimi K3：从 3T 稀疏预训练到百万 Token Agent 的端到端扩展"
 * (liuzhao09.github.io/papers/kimi-k3), called [K3-notes] below.
 *
 *  - [K3-notes §2.2, KDA state recurrence]:
 *        S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *        o~_t = S_t^T q_t,
 *    S_t in R^{dk x dv} per head, alpha_t in (0,1)^{dk} per channel, beta_t a
 *    scalar.  alpha_t = exp(g_t) with g the log-decay ([K3-notes §2.2, decay
 *    lower-bound equation (Eq. 5)]).
 *  - [K3-notes §2.2, chunkwise form]: per chunk of C tokens, cumulative decay
 *    gamma^{i->j} = prod_{r=i..j} alpha^r, Gamma row r = gamma^{1->r},
 *    pseudo-value V~ = U - W S, A = Tril[(Q o Gamma)(K / Gamma)^T] with the
 *    diagonal included, O = (Gamma o Q) S + A V~.  The page does not print U, W
 *    or the state carry; the plainest reading consistent with the recurrence is
 *        L  = StrictTril[diag(beta) (Gamma o K)(K / Gamma)^T],  T = (I + L)^{-1},
 *        U  = T diag(beta) V,   W = T diag(beta) (Gamma o K),
 *        S' = Diag(gamma_C) S + (K o gamma_C / Gamma)^T V~.
 *  - [K3-notes §2.5, context-parallel affine pair]: a segment maps its entry
 *    state to S_out = S~_local + M_local S_in.
 *  - [K3-notes §2.5, Fig. 12, prefix-cache resume]: the state after a prefix
 *    is what a request sharing that prefix resumes from; the recurrence can
 *    record it every `every` tokens (oracle_kda_recurrent_ckpt).
 *  - Gradients (oracle_kda_backward): the page says the chunk form serves
 *    training but prints no backward, so the oracle takes the plainest one,
 *    reverse-mode differentiation of the token recurrence above for the loss
 *    L = sum_t <dO_t, o~_t> + <dS_T, S_T>, written out in kda_token_bwd.
 *  - [K3-notes §2.2, Eq. 5 and the KDA output equation], the layer's gates
 *    around the recurrence (oracle_kda_layer, oracle_kda_layer_decode_step):
 *        g_t = g_min Sigmoid(exp(A_h) z_t)          (per channel; z the decay logits)
 *        y_t = Sigmoid(gate_t) o RMSNorm(o~_t)      (per token and head, over dv)
 *    with RMSNorm(x) = x / sqrt(mean_j x_j^2 + eps) o w.  The page gives no eps
 *    or weight; the plainest reading is the usual RMSNorm with a learned
 *    per-channel weight w [dv] (shared by the heads) and a small eps, both
 *    passed in.  y_t is what W_o then projects; W_o and W_g x_t are plain
 *    projections outside the recurrence (gate_t = W_g x_t is an input here).
 *
 * Layouts (all row-major, token-major like the CUDA library's inputs):
 *   q, k, g : [T_total][H][dk] float32  (the exact values the GPU receives)
 *   v       : [T_total][H][dv] float32
 *   beta    : [T_total][H]     float32
 *   states  : [N][H][dk][dv]   double   (dv contiguous)
 *   o       : [T_total][H][dv] double
 * Sequence n owns tokens [cu[n], cu[n+1]).  A "chain" is one (n, h) pair,
 * numbered n*H + h.  Chains run on host threads; each chain is a plain loop.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

/* Planted mistakes for the pin-strength tests.  0 is the oracle itself; the
 * others are deliberate errors that the tests must catch. */
enum {
  MUT_NONE = 0,
  MUT_NO_DECAY = 1,          /* alpha treated as 1                               */
  MUT_SIGN_ERASE = 2,        /* u = beta (v + x) instead of beta (v - x)          */
  MUT_UNDECAYED_PREDICT = 3, /* prediction from S_{t-1} before the decay          */
  MUT_READ_TRANSPOSED = 4,   /* o = S q instead of S^T q (needs dk == dv)         */
  MUT_READ_BEFORE_WRITE = 5, /* o read from the decayed state before the write    */
  MUT_BETA_ONLY_ON_WRITE = 6,/* erase term without beta: u = beta v - x           */
  MUT_DECAY_BY_COLUMN = 7,   /* Diag(alpha) applied to dv index (needs dk == dv)  */
  MUT_BETA_SQUARED = 8,      /* u = beta^2 (v - x)                                */
  /* layer gates (oracle_kda_layer only) */
  MUT_GATE_NEG_LOGIT = 9,    /* g = g_min Sigmoid(-exp(A) z)                      */
  MUT_GATE_NO_EXP = 10,      /* g = g_min Sigmoid(A z)                            */
  MUT_GATE_HEAD0 = 11,       /* every head uses A_0                               */
  MUT_NORM_SUM = 12,         /* RMS over the sum of squares, not the mean         */
  MUT_NORM_EPS_OUTSIDE = 13, /* 1 / (sqrt(mean x^2) + eps)                        */
  MUT_OGATE_NEG = 14,        /* Sigmoid(-gate)                                    */
  MUT_NORM_W_REVERSED = 15,  /* weight indexed dv-1-j                             */
  /* backward (oracle_kda_backward only) */
  MUT_BWD_DS_UNDECAYED = 16, /* dS_{t-1} = dP instead of Diag(alpha) dP            */
  MUT_BWD_DK_NO_PREDICT = 17,/* dk misses the prediction term P dx                 */
  MUT_BWD_DG_FROM_DS = 18,   /* dg from dS instead of dP = dS + k dx^T             */
  MUT_COUNT = 19
};

typedef struct {
  int N, H, dk, dv;
  const int64_t *cu;
  const float *q, *k, *v, *g, *beta;
  const double *s0;  /* nullable: zero initial state */
  double *o;         /* nullable */
  double *s_final;   /* nullable */
  const int32_t *chains;
  int nchains;
  int mutation;
  int chunk;         /* chunk form only */
  int subtile_ref;   /* chunk form only */
  int ckpt_every;    /* > 0: record the state every ckpt_every tokens */
  const int64_t *cu_ckpt;
  double *ckpt;
  /* layer gates (nullable z / ogate): see the header */
  const float *z;      /* [T][H][dk] decay logits; g is then ignored */
  const float *A_log;  /* [H] */
  double g_min;
  const float *ogate;  /* [T][H][dv] output gate logits */
  const float *norm_w; /* [dv], NULL: ones */
  double norm_eps;
  int next;          /* work counter */
  int status;
} job_t;

/* ---------------------------------------------------------------- recurrence */

/* One token of [K3-notes §2.2, KDA state recurrence] applied to S (dk x dv):
 *   S <- Diag(alpha) S                       (decay first, as the equation reads)
 *   x  = S^T k                               (what the decayed state predicts for k)
 *   u  = beta (v - x)                        ((I - beta k k^T) erases along k ...)
 *   S <- S + k u^T                           (... and beta k v^T writes)
 *   o  = S^T q
 * The middle three lines expand (I - beta k k^T) Diag(alpha) S + beta k v^T.
 * work: dk + dv doubles of scratch. */
static void kda_token(int dk, int dv, double *S, const float *q, const float *k,
                      const float *v, const double *g, double beta, double *o,
                      double *work, int mutation) {
  double *x = work;       /* dv */
  double *u = work + dv;  /* dv */
  (void)u;
  if (mutation == MUT_UNDECAYED_PREDICT) {
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * (double)k[i];
      x[j] = acc;
    }
  }
  if (mutation != MUT_NO_DECAY) {
    for (int i = 0; i < dk; ++i) {
      for (int j = 0; j < dv; ++j) {
        double a = exp(g[mutation == MUT_DECAY_BY_COLUMN ? j : i]);
        S[(size_t)i * dv + j] *= a;
      }
    }
  }
  if (mutation != MUT_UNDECAYED_PREDICT) {
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * (double)k[i];
      x[j] = acc;
    }
  }
  if (mutation == MUT_READ_BEFORE_WRITE) {
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * (double)q[i];
      o[j] = acc;
    }
  }
  for (int j = 0; j < dv; ++j) {
    double uj;
    switch (mutation) {
      case MUT_SIGN_ERASE: uj = beta * ((double)v[j] + x[j]); break;
      case MUT_BETA_ONLY_ON_WRITE: uj = beta * (double)v[j] - x[j]; break;
      case MUT_BETA_SQUARED: uj = beta * beta * ((double)v[j] - x[j]); break;
      default: uj = beta * ((double)v[j] - x[j]); break;
    }
    for (int i = 0; i < dk; ++i) S[(size_t)i * dv + j] += (double)k[i] * uj;
  }
  if (mutation == MUT_READ_BEFORE_WRITE) return;
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    if (mutation == MUT_READ_TRANSPOSED) {
      for (int i = 0; i < dk; ++i) acc += S[(size_t)j * dv + i] * (double)q[i];
    } else {
      for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * (double)q[i];
    }
    o[j] = acc;
  }
}

/* [K3-notes §2.2, Eq. 5]: the log-decay of one token's dk channels from its
 * decay logits, g_i = g_min Sigmoid(exp(A_h) z_i), Sigmoid(x) = 1 / (1 + e^-x). */
static void decay_from_logits(int dk, const float *z, double A_log, double g_min, double *g,
                              int mutation) {
  const double scale = mutation == MUT_GATE_NO_EXP ? A_log : exp(A_log);
  const double sgn = mutation == MUT_GATE_NEG_LOGIT ? -1.0 : 1.0;
  for (int i = 0; i < dk; ++i) g[i] = g_min / (1.0 + exp(-sgn * scale * (double)z[i]));
}

/* [K3-notes §2.2, KDA output]: o <- Sigmoid(gate) o RMSNorm(o) over the dv
 * channels of one token and head, RMSNorm(x)_j = x_j w_j / sqrt(mean x^2 + eps). */
static void output_norm_gate(int dv, double *o, const float *gate, const float *w, double eps,
                             int mutation) {
  double ms = 0.0;
  for (int j = 0; j < dv; ++j) ms += o[j] * o[j];
  if (mutation != MUT_NORM_SUM) ms /= (double)dv;
  const double r = mutation == MUT_NORM_EPS_OUTSIDE ? 1.0 / (sqrt(ms) + eps) : 1.0 / sqrt(ms + eps);
  const double sgn = mutation == MUT_OGATE_NEG ? -1.0 : 1.0;
  for (int j = 0; j < dv; ++j) {
    const double wj = w ? (double)w[mutation == MUT_NORM_W_REVERSED ? dv - 1 - j : j] : 1.0;
    o[j] = o[j] * r * wj / (1.0 + exp(-sgn * (double)gate[j]));
  }
}

static int next_chain(job_t *J) { return __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED); }

/* ------------------------------------------------------------------ backward */

/* Reverse of one kda_token step.  Sp = S_{t-1} and St = S_t (dk x dv), dS on
 * entry = dL/dS_t from the later tokens; on return dS = dL/dS_{t-1}.  With
 *   P = Diag(alpha) Sp,  x = P^T k,  u = beta (v - x),  S_t = P + k u^T,  o = S_t^T q:
 *   dS += q do^T                  (o = S_t^T q)
 *   dq  = S_t do
 *   du  = dS^T k,   dk = dS u     (S_t = P + k u^T)
 *   dbeta = du . (v - x),  dv = beta du,  dx = -beta du
 *   dk += P dx,  dP = dS + k dx^T (x = P^T k)
 *   dalpha_i = sum_j dP_ij Sp_ij,  dg = alpha o dalpha,  dS_{t-1} = Diag(alpha) dP.
 * work: 3 dv + dk doubles. */
static void kda_token_bwd(int dk, int dv, const double *Sp, const double *St, double *dS, const float *q,
                          const float *k, const float *v, const double *g, double beta, const float *dO,
                          double *dq, double *dkv, double *dvv, double *dg, double *dbeta, double *work,
                          int mutation) {
  double *x = work, *u = work + dv, *du = work + 2 * dv, *alpha = work + 3 * dv;
  for (int i = 0; i < dk; ++i) alpha[i] = exp(g[i]);
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < dk; ++i) acc += alpha[i] * Sp[(size_t)i * dv + j] * (double)k[i];
    x[j] = acc;
    u[j] = beta * ((double)v[j] - acc);
  }
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) dS[(size_t)i * dv + j] += (double)q[i] * (double)dO[j];
  for (int i = 0; i < dk; ++i) {
    double acc = 0.0;
    for (int j = 0; j < dv; ++j) acc += St[(size_t)i * dv + j] * (double)dO[j];
    dq[i] = acc;
  }
  double db = 0.0;
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < dk; ++i) acc += dS[(size_t)i * dv + j] * (double)k[i];
    du[j] = acc;
    db += acc * ((double)v[j] - x[j]);
    dvv[j] = beta * acc;
  }
  *dbeta = db;
  for (int i = 0; i < dk; ++i) {
    double acc = 0.0;
    for (int j = 0; j < dv; ++j) {
      acc += dS[(size_t)i * dv + j] * u[j];
      if (mutation != MUT_BWD_DK_NO_PREDICT) acc += alpha[i] * Sp[(size_t)i * dv + j] * (-beta * du[j]);
    }
    dkv[i] = acc;
  }
  for (int i = 0; i < dk; ++i) {
    double da = 0.0;
    for (int j = 0; j < dv; ++j) {
      const double dP = dS[(size_t)i * dv + j] + (double)k[i] * (-beta * du[j]);
      da += (mutation == MUT_BWD_DG_FROM_DS ? dS[(size_t)i * dv + j] : dP) * Sp[(size_t)i * dv + j];
      dS[(size_t)i * dv + j] = mutation == MUT_BWD_DS_UNDECAYED ? dP : alpha[i] * dP;
    }
    dg[i] = alpha[i] * da;
  }
}

/* Work item of the backward: one chain, its states recomputed a block of
 * kBwdBlock tokens at a time from states kept at block starts. */
enum { kBwdBlock = 64 };

typedef struct {
  job_t base;
  const float *dO;      /* [T][H][dv] */
  const float *dST;     /* [N][H][dk][dv] or NULL */
  double *dq, *dk, *dv, *dg, *dbeta, *ds0;
} bwd_job_t;

static void *backward_worker(void *arg) {
  bwd_job_t *B = (bwd_job_t *)arg;
  job_t *J = &B->base;
  const int dk = J->dk, dv = J->dv, H = J->H;
  const size_t SS = (size_t)dk * dv;
  int64_t maxlen = 0;
  for (int n = 0; n < J->N; ++n)
    if (J->cu[n + 1] - J->cu[n] > maxlen) maxlen = J->cu[n + 1] - J->cu[n];
  const int64_t nblk = (maxlen + kBwdBlock - 1) / kBwdBlock;
  double *starts = (double *)malloc(sizeof(double) * SS * (size_t)(nblk > 0 ? nblk : 1));
  double *states = (double *)malloc(sizeof(double) * SS * (kBwdBlock + 1));
  double *dS = (double *)malloc(sizeof(double) * SS);
  double *work = (double *)malloc(sizeof(double) * (size_t)(3 * dv + dk));
  double *grow = (double *)malloc(sizeof(double) * (size_t)dk);
  double *obuf = (double *)malloc(sizeof(double) * (size_t)dv);
  if (!starts || !states || !dS || !work || !grow || !obuf) {
    J->status = ORACLE_ENOMEM;
    free(starts); free(states); free(dS); free(work); free(grow); free(obuf);
    return NULL;
  }
  for (;;) {
    int w = next_chain(J);
    if (w >= J->nchains) break;
    const int n = w / H, h = w % H;
    const int64_t t0 = J->cu[n], t1 = J->cu[n + 1];
    const size_t sidx = ((size_t)n * H + h) * SS;
    /* forward: keep the state at every block start */
    double *S = states;
    if (J->s0) memcpy(S, J->s0 + sidx, sizeof(double) * SS);
    else memset(S, 0, sizeof(double) * SS);
    for (int64_t t = t0; t < t1; ++t) {
      if ((t - t0) % kBwdBlock == 0) memcpy(starts + (size_t)((t - t0) / kBwdBlock) * SS, S, sizeof(double) * SS);
      const size_t th = (size_t)t * H + h;
      for (int i = 0; i < dk; ++i) grow[i] = (double)J->g[th * dk + i];
      kda_token(dk, dv, S, J->q + th * dk, J->k + th * dk, J->v + th * dv, grow, (double)J->beta[th], obuf,
                work, MUT_NONE);
    }
    /* backward, block by block from the end */
    if (B->dST) for (size_t e = 0; e < SS; ++e) dS[e] = (double)B->dST[sidx + e];
    else memset(dS, 0, sizeof(double) * SS);
    for (int64_t b = (t1 - t0 + kBwdBlock - 1) / kBwdBlock - 1; b >= 0; --b) {
      const int64_t bs = t0 + b * kBwdBlock, be = (bs + kBwdBlock < t1) ? bs + kBwdBlock : t1;
      memcpy(states, starts + (size_t)b * SS, sizeof(double) * SS);
      for (int64_t t = bs; t < be; ++t) {  /* states[t - bs] = S_{t-1}; states[t - bs + 1] = S_t */
        double *Sn = states + (size_t)(t - bs + 1) * SS;
        memcpy(Sn, states + (size_t)(t - bs) * SS, sizeof(double) * SS);
        const size_t th = (size_t)t * H + h;
        for (int i = 0; i < dk; ++i) grow[i] = (double)J->g[th * dk + i];
        kda_token(dk, dv, Sn, J->q + th * dk, J->k + th * dk, J->v + th * dv, grow, (double)J->beta[th], obuf,
                  work, MUT_NONE);
      }
      for (int64_t t = be - 1; t >= bs; --t) {
        const size_t th = (size_t)t * H + h;
        for (int i = 0; i < dk; ++i) grow[i] = (double)J->g[th * dk + i];
        kda_token_bwd(dk, dv, states + (size_t)(t - bs) * SS, states + (size_t)(t - bs + 1) * SS, dS,
                      J->q + th * dk, J->k + th * dk, J->v + th * dv, grow, (double)J->beta[th], B->dO + th * dv,
                      B->dq + th * dk, B->dk + th * dk, B->dv + th * dv, B->dg + th * dk, B->dbeta + th, work,
                      J->mutation);
      }
    }
    if (B->ds0) memcpy(B->ds0 + sidx, dS, sizeof(double) * SS);
  }
  free(starts); free(states); free(dS); free(work); free(grow); free(obuf);
  return NULL;
}

static void *recurrent_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int dk = J->dk, dv = J->dv, H = J->H;
  double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *work = (double *)malloc(sizeof(double) * (size_t)(2 * dv));
  double *obuf = (double *)malloc(sizeof(double) * (size_t)dv);
  double *grow = (double *)malloc(sizeof(double) * (size_t)dk);
  if (!S || !work || !obuf || !grow) {
    J->status = ORACLE_ENOMEM;
    free(S); free(work); free(obuf); free(grow);
    return NULL;
  }
  for (;;) {
    int w = next_chain(J);
    if (w >= J->nchains) break;
    int c = J->chains ? J->chains[w] : w;
    int n = c / H, h = c % H;
    size_t sidx = ((size_t)n * H + h) * (size_t)dk * dv;
    if (J->s0) memcpy(S, J->s0 + sidx, sizeof(double) * (size_t)dk * dv);
    else memset(S, 0, sizeof(double) * (size_t)dk * dv);
    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
      size_t th = (size_t)t * H + h;
      if (J->z) {
        decay_from_logits(dk, J->z + th * dk, (double)J->A_log[J->mutation == MUT_GATE_HEAD0 ? 0 : h],
                          J->g_min, grow, J->mutation);
      } else {
        for (int i = 0; i < dk; ++i) grow[i] = (double)J->g[th * dk + i];
      }
      kda_token(dk, dv, S, J->q + th * dk, J->k + th * dk, J->v + th * dv, grow,
                (double)J->beta[th], obuf, work, J->mutation);
      if (J->ogate) output_norm_gate(dv, obuf, J->ogate + th * dv, J->norm_w, J->norm_eps, J->mutation);
      if (J->o) memcpy(J->o + th * dv, obuf, sizeof(double) * (size_t)dv);
      const int64_t done = t - J->cu[n] + 1;
      if (J->ckpt && done % J->ckpt_every == 0) {
        const int64_t slot = J->cu_ckpt[n] + done / J->ckpt_every - 1;
        memcpy(J->ckpt + ((size_t)slot * H + h) * (size_t)dk * dv, S, sizeof(double) * (size_t)dk * dv);
      }
    }
    if (J->s_final) memcpy(J->s_final + sidx, S, sizeof(double) * (size_t)dk * dv);
  }
  free(S); free(work); free(obuf); free(grow);
  return NULL;
}

static int run_threads(job_t *J, int nthreads, void *(*fn)(void *)) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > J->nchains) nthreads = J->nchains > 0 ? J->nchains : 1;
  J->next = 0;
  J->status = ORACLE_OK;
  if (nthreads == 1) {
    fn(J);
    return J->status;
  }
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!tid) return ORACLE_ENOMEM;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, fn, J) != 0) break;
    ++started;
  }
  if (started == 0) fn(J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  free(tid);
  return J->status;
}

static int check_common(int N, int H, int dk, int dv, const int64_t *cu) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu) return ORACLE_EINVAL;
  for (int n = 0; n < N; ++n)
    if (cu[n + 1] < cu[n]) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Token-by-token recurrence over every chain listed in `chains` (all N*H
 * chains when chains == NULL).  Rows of o that belong to other chains are
 * left untouched. */
int oracle_kda_recurrent(int N, int H, int dk, int dv, const int64_t *cu, const float *q,
                         const float *k, const float *v, const float *g, const float *beta,
                         const double *s0, double *o, double *s_final, const int32_t *chains,
                         int nchains, int nthreads, int mutation) {
  int st = check_common(N, H, dk, dv, cu);
  if (st) return st;
  if ((mutation == MUT_READ_TRANSPOSED || mutation == MUT_DECAY_BY_COLUMN) && dk != dv)
    return ORACLE_EINVAL;
  if (mutation < 0 || mutation >= MUT_GATE_NEG_LOGIT) return ORACLE_EINVAL;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.N = N; J.H = H; J.dk = dk; J.dv = dv; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
  J.s0 = s0; J.o = o; J.s_final = s_final;
  J.chains = chains; J.nchains = chains ? nchains : N * H;
  J.mutation = mutation;
  return run_threads(&J, nthreads, recurrent_worker);
}

/* oracle_kda_recurrent over all chains that also records each sequence's
 * state after every `every` tokens: after its first j*every tokens (j >= 1)
 * into slot cu_ckpt[n] + j - 1 of ckpt [slots][H][dk][dv]; cu_ckpt[n+1] -
 * cu_ckpt[n] must be floor(len_n / every). */
int oracle_kda_recurrent_ckpt(int N, int H, int dk, int dv, const int64_t *cu, const float *q,
                              const float *k, const float *v, const float *g, const float *beta,
                              const double *s0, double *o, double *s_final, int every,
                              const int64_t *cu_ckpt, double *ckpt, int nthreads) {
  int st = check_common(N, H, dk, dv, cu);
  if (st) return st;
  if (every <= 0 || !cu_ckpt || !ckpt) return ORACLE_EINVAL;
  for (int n = 0; n < N; ++n)
    if (cu_ckpt[n + 1] - cu_ckpt[n] != (cu[n + 1] - cu[n]) / every) return ORACLE_EINVAL;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.N = N; J.H = H; J.dk = dk; J.dv = dv; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
  J.s0 = s0; J.o = o; J.s_final = s_final;
  J.nchains = N * H;
  J.ckpt_every = every; J.cu_ckpt = cu_ckpt; J.ckpt = ckpt;
  return run_threads(&J, nthreads, recurrent_worker);
}

/* The KDA layer around the recurrence ([K3-notes §2.2]): the log-decay comes
 * from the decay logits z (Eq. 5) and, when ogate is given, each output row
 * goes through the per-head RMSNorm and the sigmoid output gate.  All chains;
 * arguments otherwise as oracle_kda_recurrent. */
int oracle_kda_layer(int N, int H, int dk, int dv, const int64_t *cu, const float *q, const float *k,
                     const float *v, const float *z, const float *A_log, double g_min, const float *beta,
                     const float *ogate, const float *norm_w, double norm_eps, const double *s0,
                     double *o, double *s_final, int nthreads, int mutation) {
  int st = check_common(N, H, dk, dv, cu);
  if (st) return st;
  if (!z || !A_log || (ogate && !(norm_eps >= 0.0))) return ORACLE_EINVAL;
  if (mutation != MUT_NONE && mutation < MUT_GATE_NEG_LOGIT) return ORACLE_EINVAL;
  if (mutation < 0 || mutation >= MUT_COUNT) return ORACLE_EINVAL;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.N = N; J.H = H; J.dk = dk; J.dv = dv; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = NULL; J.beta = beta;
  J.z = z; J.A_log = A_log; J.g_min = g_min;
  J.ogate = ogate; J.norm_w = norm_w; J.norm_eps = norm_eps;
  J.s0 = s0; J.o = o; J.s_final = s_final;
  J.nchains = N * H;
  J.mutation = mutation;
  return run_threads(&J, nthreads, recurrent_worker);
}

/* One decode step of the layer (oracle_kda_layer with every sequence one
 * token long); state [N][H][dk][dv] updated in place. */
int oracle_kda_layer_decode_step(int N, int H, int dk, int dv, const float *q, const float *k,
                                 const float *v, const float *z, const float *A_log, double g_min,
                                 const float *beta, const float *ogate, const float *norm_w,
                                 double norm_eps, double *state, double *o, int nthreads) {
  if (N <= 0) return ORACLE_EINVAL;
  int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N + 1));
  if (!cu) return ORACLE_ENOMEM;
  for (int n = 0; n <= N; ++n) cu[n] = n;
  int st = oracle_kda_layer(N, H, dk, dv, cu, q, k, v, z, A_log, g_min, beta, ogate, norm_w, norm_eps,
                            state, o, state, nthreads, MUT_NONE);
  free(cu);
  return st;
}

/* Gradients of L = sum_t <dO_t, o~_t> + <dST, S_T> (dST NULL: 0) with respect
 * to q, k, v, g (log-decay), beta and the initial state, by reverse-mode
 * differentiation of the token recurrence.  Layouts as the forward; ds0 is
 * [N][H][dk][dv] (nullable).  All chains. */
int oracle_kda_backward(int N, int H, int dk, int dv, const int64_t *cu, const float *q, const float *k,
                        const float *v, const float *g, const float *beta, const double *s0, const float *dO,
                        const float *dST, double *dq, double *dk_out, double *dv_out, double *dg, double *dbeta,
                        double *ds0, int nthreads, int mutation) {
  int st = check_common(N, H, dk, dv, cu);
  if (st) return st;
  if (!dO || !dq || !dk_out || !dv_out || !dg || !dbeta) return ORACLE_EINVAL;
  if (mutation != MUT_NONE && (mutation < MUT_BWD_DS_UNDECAYED || mutation >= MUT_COUNT)) return ORACLE_EINVAL;
  bwd_job_t B;
  memset(&B, 0, sizeof(B));
  job_t *J = &B.base;
  J->N = N; J->H = H; J->dk = dk; J->dv = dv; J->cu = cu;
  J->q = q; J->k = k; J->v = v; J->g = g; J->beta = beta; J->s0 = s0;
  J->nchains = N * H;
  J->mutation = mutation;
  B.dO = dO; B.dST = dST;
  B.dq = dq; B.dk = dk_out; B.dv = dv_out; B.dg = dg; B.dbeta = dbeta; B.ds0 = ds0;
  return run_threads(J, nthreads, backward_worker);
}

/* One decode step for N independent sequences: each (n, h) consumes one token
 * (row n of q/k/v/g/beta) and updates state[n][h] in place.  This is the same
 * recurrence with every sequence one token long. */
int oracle_kda_decode_step(int N, int H, int dk, int dv, const float *q, const float *k,
                           const float *v, const float *g, const float *beta, double *state,
                           double *o, const int32_t *chains, int nchains, int nthreads) {
  if (N <= 0) return ORACLE_EINVAL;
  int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N + 1));
  if (!cu) return ORACLE_ENOMEM;
  for (int n = 0; n <= N; ++n) cu[n] = n;
  int st = oracle_kda_recurrent(N, H, dk, dv, cu, q, k, v, g, beta, state, o, state, chains,
                                nchains, nthreads, MUT_NONE);
  free(cu);
  return st;
}

/* ------------------------------------------------------------- chunk form */

/* The chunkwise form of [K3-notes §2.2] written out in fp64 with the U, W and
 * carry formulas stated in the file header.  It is not blocked or fused beyond
 * what those formulas state.  subtile_ref selects how the Gram products
 * (Q o Gamma)(K / Gamma)^T are factored: 0 uses the chunk start as the decay
 * reference for every pair (the page's literal form); 1 uses, for each key
 * column s, the cumulative decay at the start of s's 16-token tile, which is
 * the tile-range argument of [K3-notes §2.2, Fig. 3].  Both are the same
 * number in exact arithmetic; in fp64 both stay in range for C <= 64 and
 * g >= -5. */
static void *chunk_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int dk = J->dk, dv = J->dv, H = J->H, C = J->chunk;
  size_t need = (size_t)dk * dv          /* S */
                + (size_t)C * dk * 2     /* G, Gamma */
                + (size_t)C * C * 3      /* A, L, T */
                + (size_t)C * dv * 3     /* U, Vt, O */
                + (size_t)C * dk         /* W */
                + (size_t)dk * dv;       /* S next */
  double *buf = (double *)malloc(sizeof(double) * need);
  if (!buf) { J->status = ORACLE_ENOMEM; return NULL; }
  for (;;) {
    int w = next_chain(J);
    if (w >= J->nchains) break;
    int c = J->chains ? J->chains[w] : w;
    int n = c / H, h = c % H;
    double *S = buf;
    double *G = S + (size_t)dk * dv;
    double *Gam = G + (size_t)C * dk;
    double *A = Gam + (size_t)C * dk;
    double *L = A + (size_t)C * C;
    double *T = L + (size_t)C * C;
    double *U = T + (size_t)C * C;
    double *Vt = U + (size_t)C * dv;
    double *O = Vt + (size_t)C * dv;
    double *W = O + (size_t)C * dv;
    double *Sn = W + (size_t)C * dk;
    size_t sidx = ((size_t)n * H + h) * (size_t)dk * dv;
    if (J->s0) memcpy(S, J->s0 + sidx, sizeof(double) * (size_t)dk * dv);
    else memset(S, 0, sizeof(double) * (size_t)dk * dv);
    for (int64_t t0 = J->cu[n]; t0 < J->cu[n + 1]; t0 += C) {
      int len = (int)((J->cu[n + 1] - t0) < C ? (J->cu[n + 1] - t0) : C);
#define IDX(t, d) (((size_t)(t0 + (t)) * H + h) * (size_t)(d))
      /* cumulative log-decay within the chunk, G[r] = sum_{t<=r} g_t */
      for (int i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (int r = 0; r < len; ++r) {
          acc += (double)J->g[IDX(r, dk) + i];
          G[(size_t)r * dk + i] = acc;
          Gam[(size_t)r * dk + i] = exp(acc);
        }
      }
      /* A (diagonal included) and L (strict) */
      for (int r = 0; r < len; ++r) {
        for (int s = 0; s < len; ++s) {
          double a = 0.0, l = 0.0;
          if (s <= r) {
            int s0 = J->subtile_ref ? (s / 16) * 16 : 0;
            for (int i = 0; i < dk; ++i) {
              double ref = s0 > 0 ? G[(size_t)(s0 - 1) * dk + i] : 0.0;
              double qb = (double)J->q[IDX(r, dk) + i] * exp(G[(size_t)r * dk + i] - ref);
              double gk = (double)J->k[IDX(r, dk) + i] * exp(G[(size_t)r * dk + i] - ref);
              double kb = (double)J->k[IDX(s, dk) + i] * exp(ref - G[(size_t)s * dk + i]);
              a += qb * kb;
              l += gk * kb;
            }
          }
          A[(size_t)r * C + s] = a;
          L[(size_t)r * C + s] = (s < r) ? (double)J->beta[IDX(r, 1)] * l : 0.0;
        }
      }
      /* T = (I + L)^{-1}, forward substitution row by row */
      for (int r = 0; r < len; ++r) {
        for (int s = 0; s < len; ++s) {
          double acc = (r == s) ? 1.0 : 0.0;
          for (int m = 0; m < r; ++m) acc -= L[(size_t)r * C + m] * T[(size_t)m * C + s];
          T[(size_t)r * C + s] = acc;
        }
      }
      /* U = T diag(beta) V ; W = T diag(beta) (Gamma o K) */
      for (int r = 0; r < len; ++r) {
        for (int j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (int s = 0; s < len; ++s)
            acc += T[(size_t)r * C + s] * (double)J->beta[IDX(s, 1)] * (double)J->v[IDX(s, dv) + j];
          U[(size_t)r * dv + j] = acc;
        }
        for (int i = 0; i < dk; ++i) {
          double acc = 0.0;
          for (int s = 0; s < len; ++s)
            acc += T[(size_t)r * C + s] * (double)J->beta[IDX(s, 1)] * Gam[(size_t)s * dk + i] *
                   (double)J->k[IDX(s, dk) + i];
          W[(size_t)r * dk + i] = acc;
        }
      }
      /* V~ = U - W S */
      for (int r = 0; r < len; ++r)
        for (int j = 0; j < dv; ++j) {
          double acc = U[(size_t)r * dv + j];
          for (int i = 0; i < dk; ++i) acc -= W[(size_t)r * dk + i] * S[(size_t)i * dv + j];
          Vt[(size_t)r * dv + j] = acc;
        }
      /* O = (Gamma o Q) S + A V~ */
      for (int r = 0; r < len; ++r)
        for (int j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (int i = 0; i < dk; ++i)
            acc += Gam[(size_t)r * dk + i] * (double)J->q[IDX(r, dk) + i] * S[(size_t)i * dv + j];
          for (int s = 0; s <= r; ++s) acc += A[(size_t)r * C + s] * Vt[(size_t)s * dv + j];
          O[(size_t)r * dv + j] = acc;
        }
      /* S' = Diag(gamma_C) S + (K o gamma_C / Gamma)^T V~ */
      for (int i = 0; i < dk; ++i) {
        double GC = G[(size_t)(len - 1) * dk + i];
        for (int j = 0; j < dv; ++j) {
          double acc = exp(GC) * S[(size_t)i * dv + j];
          for (int r = 0; r < len; ++r)
            acc += (double)J->k[IDX(r, dk) + i] * exp(GC - G[(size_t)r * dk + i]) *
                   Vt[(size_t)r * dv + j];
          Sn[(size_t)i * dv + j] = acc;
        }
      }
      memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
      if (J->o)
        for (int r = 0; r < len; ++r)
          memcpy(J->o + IDX(r, dv), O + (size_t)r * dv, sizeof(double) * (size_t)dv);
#undef IDX
    }
    if (J->s_final) memcpy(J->s_final + sidx, S, sizeof(double) * (size_t)dk * dv);
  }
  free(buf);
  return NULL;
}

int oracle_kda_chunked(int N, int H, int dk, int dv, const int64_t *cu, const float *q,
                       const float *k, const float *v, const float *g, const float *beta,
                       const double *s0, double *o, double *s_final, const int32_t *chains,
                       int nchains, int nthreads, int chunk, int subtile_ref) {
  int st = check_common(N, H, dk, dv, cu);
  if (st) return st;
  if (chunk <= 0 || chunk > 256) return ORACLE_EINVAL;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.N = N; J.H = H; J.dk = dk; J.dv = dv; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
  J.s0 = s0; J.o = o; J.s_final = s_final;
  J.chains = chains; J.nchains = chains ? nchains : N * H;
  J.chunk = chunk; J.subtile_ref = subtile_ref;
  return run_threads(&J, nthreads, chunk_worker);
}

/* ------------------------------------------------------------ affine pair */

/* [K3-notes §2.5, context-parallel affine pair] for tokens [t0, t1) of head h:
 * the segment maps any entry state S_in to S_out = S~ + M S_in.  M (dk x dk)
 * is the ordered product of the per-token transitions
 * (I - beta_t k_t k_t^T) Diag(alpha_t); S~ (dk x dv) is the segment's state when
 * it starts from zero.  Both follow from the recurrence by carrying M as extra
 * state columns that receive no write. */
int oracle_kda_affine_pair(int H, int dk, int dv, int h, int64_t t0, int64_t t1, const float *k,
                           const float *v, const float *g, const float *beta, double *M,
                           double *St) {
  if (H <= 0 || dk <= 0 || dv <= 0 || h < 0 || h >= H || t1 < t0) return ORACLE_EINVAL;
  double *x = (double *)malloc(sizeof(double) * (size_t)(dk + dv));
  if (!x) return ORACLE_ENOMEM;
  for (int i = 0; i < dk; ++i)
    for (int m = 0; m < dk; ++m) M[(size_t)i * dk + m] = (i == m) ? 1.0 : 0.0;
  memset(St, 0, sizeof(double) * (size_t)dk * dv);
  for (int64_t t = t0; t < t1; ++t) {
    size_t th = (size_t)t * H + h;
    const float *kt = k + th * dk, *vt = v + th * dv, *gt = g + th * dk;
    double b = (double)beta[th];
    for (int i = 0; i < dk; ++i) {
      double a = exp((double)gt[i]);
      for (int m = 0; m < dk; ++m) M[(size_t)i * dk + m] *= a;
      for (int j = 0; j < dv; ++j) St[(size_t)i * dv + j] *= a;
    }
    /* M <- M - beta k (k^T M);   S~ <- S~ + k beta (v - S~^T k)^T */
    for (int m = 0; m < dk; ++m) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += (double)kt[i] * M[(size_t)i * dk + m];
      x[m] = acc;
    }
    for (int i = 0; i < dk; ++i)
      for (int m = 0; m < dk; ++m) M[(size_t)i * dk + m] -= b * (double)kt[i] * x[m];
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += (double)kt[i] * St[(size_t)i * dv + j];
      x[j] = b * ((double)vt[j] - acc);
    }
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) St[(size_t)i * dv + j] += (double)kt[i] * x[j];
  }
  free(x);
  return ORACLE_OK;
}

int oracle_mutation_count(void) { return MUT_COUNT; }
