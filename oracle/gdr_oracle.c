/*
 * gdr_oracle.c -- plain fp64 CPU oracle for the gated delta rule (GDR).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this library.  The CUDA product
 * path never links, loads or calls it, and it shares no code with the CUDA
 * path.
 *
 * What it computes (FlashQLA PR #34, "SM120/121: Add support for fused
 * backward kernel", Summary and "Current status": the operator is the chunked
 * gated delta rule with fixed-length and variable-length inputs, initial and
 * final states, and autograd).  The pages never write the recurrence out; the
 * operator is fixed as
 *
 *     S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale * S_t q_t                     (scale = 1/sqrt(DK) by default)
 *
 * with S in R^{DV x DK}.  This file evaluates that recurrence token by token
 * (no chunking at all) and its reverse-time gradient, derived by hand from
 * the same recurrence:
 *
 *     G := dL/dS_t, starting at dS_T (or 0); for t = L-1 .. 0, with p = S_{t-1} k_t:
 *       G     += scale * do_t q_t^T
 *       dq_t   = scale * S_t^T do_t
 *       u      = G k_t
 *       dv_t   = beta_t u
 *       dbeta_t= u^T (v_t - alpha_t p)
 *       dg_t   = alpha_t * (<G, S_{t-1}> - beta_t u^T p)
 *       dk_t   = beta_t (G^T (v_t - alpha_t p) - alpha_t S_{t-1}^T u)
 *       G      = alpha_t (G - beta_t u k_t^T)
 *     dS0 = G
 *
 * Data layout (all fp64, contiguous, packed token-major):
 *   q, k, dq, dk : [T_total][Hk][DK]
 *   v, o, dO, dv : [T_total][Hv][DV]
 *   g, beta, dg, dbeta : [T_total][Hv]
 *   S0, S_T, dS_T, dS0 : [num_seqs][Hv][DV][DK]   (S itself, "VK" orientation)
 *   S_chunks : [n_chunks_total][Hv][DV][DK], the state at the start of every
 *              64-token chunk; chunk c of sequence n has global index
 *              chunk_offset[n] + c with chunk_offset[n] = sum_{n'<n} ceil(L_n'/64).
 *   cu_seqlens : int64 [num_seqs+1] token offsets (fixed length B x T is
 *                cu_seqlens = 0, T, 2T, ...).
 * v-head j reads q/k head j / (Hv/Hk) (contiguous groups); g and beta are
 * per v-head; dq and dk sum over the v-heads of a group.
 *
 * Threads: one work unit = (sequence, q/k head); its v-heads run one after the
 * other in a fixed order so that dq/dk sums are deterministic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_CHUNK 64

typedef struct {
  int num_seqs;
  const int64_t* cu;
  int Hk, Hv, DK, DV;
  double scale;
  const double *q, *k, *v, *g, *beta, *S0;
  double *o, *S_T, *S_chunks;
  const double *dO, *dS_T;
  double *dq, *dk, *dv, *dg, *dbeta, *dS0;
  int backward;
  int64_t* chunk_offset; /* [num_seqs + 1] */
  int n_units;
  int next_unit;
  int failed;
  pthread_mutex_t lock;
} oracle_job;

/* One token step of the forward recurrence: S <- alpha S (I - b k k^T) + b v k^T.
 * p (length DV) receives S_{t-1} k on return. */
static void step_forward(double* S, int DV, int DK, double alpha, double b,
                         const double* kt, const double* vt, double* p) {
  for (int a = 0; a < DV; ++a) {
    double acc = 0.0;
    const double* row = S + (size_t)a * DK;
    for (int c = 0; c < DK; ++c) acc += row[c] * kt[c];
    p[a] = acc;
  }
  for (int a = 0; a < DV; ++a) {
    double* row = S + (size_t)a * DK;
    const double coef = b * vt[a] - alpha * b * p[a];
    for (int c = 0; c < DK; ++c) row[c] = alpha * row[c] + coef * kt[c];
  }
}

static void run_forward_head(oracle_job* J, int n, int i, int j, double* S, double* p) {
  const int DK = J->DK, DV = J->DV, Hk = J->Hk, Hv = J->Hv;
  const int64_t t0 = J->cu[n], t1 = J->cu[n + 1];
  const size_t SS = (size_t)DV * DK;
  if (J->S0)
    memcpy(S, J->S0 + ((size_t)n * Hv + j) * SS, SS * sizeof(double));
  else
    memset(S, 0, SS * sizeof(double));
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t local = t - t0;
    if (J->S_chunks && local % ORACLE_CHUNK == 0) {
      const int64_t cidx = J->chunk_offset[n] + local / ORACLE_CHUNK;
      memcpy(J->S_chunks + ((size_t)cidx * Hv + j) * SS, S, SS * sizeof(double));
    }
    const double alpha = exp(J->g[(size_t)t * Hv + j]);
    const double b = J->beta[(size_t)t * Hv + j];
    const double* kt = J->k + ((size_t)t * Hk + i) * DK;
    const double* qt = J->q + ((size_t)t * Hk + i) * DK;
    const double* vt = J->v + ((size_t)t * Hv + j) * DV;
    step_forward(S, DV, DK, alpha, b, kt, vt, p);
    if (J->o) {
      double* ot = J->o + ((size_t)t * Hv + j) * DV;
      for (int a = 0; a < DV; ++a) {
        double acc = 0.0;
        const double* row = S + (size_t)a * DK;
        for (int c = 0; c < DK; ++c) acc += row[c] * qt[c];
        ot[a] = J->scale * acc;
      }
    }
  }
  if (J->S_T) memcpy(J->S_T + ((size_t)n * Hv + j) * SS, S, SS * sizeof(double));
}

/* Reverse-time gradient of one (sequence, v-head).  States are checkpointed
 * every 64 tokens and recomputed forward inside each 64-token segment. */
static int run_backward_head(oracle_job* J, int n, int i, int j) {
  const int DK = J->DK, DV = J->DV, Hk = J->Hk, Hv = J->Hv;
  const int64_t t0 = J->cu[n], t1 = J->cu[n + 1];
  const int64_t L = t1 - t0;
  const size_t SS = (size_t)DV * DK;
  const int64_t nseg = (L + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
  double* ckpt = (double*)malloc((size_t)(nseg > 0 ? nseg : 1) * SS * sizeof(double));
  double* states = (double*)malloc((size_t)(ORACLE_CHUNK + 1) * SS * sizeof(double));
  double* G = (double*)malloc(SS * sizeof(double));
  double* p = (double*)malloc((size_t)DV * sizeof(double));
  double* u = (double*)malloc((size_t)DV * sizeof(double));
  double* w = (double*)malloc((size_t)DV * sizeof(double));
  if (!ckpt || !states || !G || !p || !u || !w) {
    free(ckpt); free(states); free(G); free(p); free(u); free(w);
    return -1;
  }
  /* forward pass keeping the state before every segment */
  double* S = states; /* scratch */
  if (J->S0)
    memcpy(S, J->S0 + ((size_t)n * Hv + j) * SS, SS * sizeof(double));
  else
    memset(S, 0, SS * sizeof(double));
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t local = t - t0;
    if (local % ORACLE_CHUNK == 0)
      memcpy(ckpt + (size_t)(local / ORACLE_CHUNK) * SS, S, SS * sizeof(double));
    const double alpha = exp(J->g[(size_t)t * Hv + j]);
    const double b = J->beta[(size_t)t * Hv + j];
    step_forward(S, DV, DK, alpha, b, J->k + ((size_t)t * Hk + i) * DK,
                 J->v + ((size_t)t * Hv + j) * DV, p);
  }
  if (J->dS_T)
    memcpy(G, J->dS_T + ((size_t)n * Hv + j) * SS, SS * sizeof(double));
  else
    memset(G, 0, SS * sizeof(double));

  for (int64_t seg = nseg - 1; seg >= 0; --seg) {
    const int64_t s0 = t0 + seg * ORACLE_CHUNK;
    const int64_t s1 = (s0 + ORACLE_CHUNK < t1) ? s0 + ORACLE_CHUNK : t1;
    /* states[m] = S before token s0+m, states[m+1] = S after it */
    memcpy(states, ckpt + (size_t)seg * SS, SS * sizeof(double));
    for (int64_t t = s0; t < s1; ++t) {
      double* nxt = states + (size_t)(t - s0 + 1) * SS;
      memcpy(nxt, states + (size_t)(t - s0) * SS, SS * sizeof(double));
      const double alpha = exp(J->g[(size_t)t * Hv + j]);
      const double b = J->beta[(size_t)t * Hv + j];
      step_forward(nxt, DV, DK, alpha, b, J->k + ((size_t)t * Hk + i) * DK,
                   J->v + ((size_t)t * Hv + j) * DV, p);
    }
    for (int64_t t = s1 - 1; t >= s0; --t) {
      const double* Sprev = states + (size_t)(t - s0) * SS;
      const double* Scur = states + (size_t)(t - s0 + 1) * SS;
      const double alpha = exp(J->g[(size_t)t * Hv + j]);
      const double b = J->beta[(size_t)t * Hv + j];
      const double* kt = J->k + ((size_t)t * Hk + i) * DK;
      const double* qt = J->q + ((size_t)t * Hk + i) * DK;
      const double* vt = J->v + ((size_t)t * Hv + j) * DV;
      const double* dot = J->dO ? J->dO + ((size_t)t * Hv + j) * DV : NULL;
      double* dqt = J->dq + ((size_t)t * Hk + i) * DK;
      double* dkt = J->dk + ((size_t)t * Hk + i) * DK;
      /* o_t = scale * S_t q_t  ->  dL/dS_t += scale * do_t q_t^T, dq_t += scale * S_t^T do_t */
      if (dot) {
        for (int a = 0; a < DV; ++a) {
          double* Grow = G + (size_t)a * DK;
          const double sa = J->scale * dot[a];
          for (int c = 0; c < DK; ++c) Grow[c] += sa * qt[c];
        }
        for (int c = 0; c < DK; ++c) {
          double acc = 0.0;
          for (int a = 0; a < DV; ++a) acc += Scur[(size_t)a * DK + c] * dot[a];
          dqt[c] += J->scale * acc;
        }
      }
      /* u = G k_t, p = S_{t-1} k_t, w = v_t - alpha p */
      for (int a = 0; a < DV; ++a) {
        double au = 0.0, ap = 0.0;
        const double* Grow = G + (size_t)a * DK;
        const double* Prow = Sprev + (size_t)a * DK;
        for (int c = 0; c < DK; ++c) {
          au += Grow[c] * kt[c];
          ap += Prow[c] * kt[c];
        }
        u[a] = au;
        p[a] = ap;
        w[a] = vt[a] - alpha * ap;
      }
      double* dvt = J->dv + ((size_t)t * Hv + j) * DV;
      double dbeta = 0.0, up = 0.0, GS = 0.0;
      for (int a = 0; a < DV; ++a) {
        dvt[a] = b * u[a];
        dbeta += u[a] * w[a];
        up += u[a] * p[a];
      }
      for (size_t e = 0; e < SS; ++e) GS += G[e] * Sprev[e];
      J->dbeta[(size_t)t * Hv + j] = dbeta;
      J->dg[(size_t)t * Hv + j] = alpha * (GS - b * up);
      for (int c = 0; c < DK; ++c) {
        double gw = 0.0, su = 0.0;
        for (int a = 0; a < DV; ++a) {
          gw += G[(size_t)a * DK + c] * w[a];
          su += Sprev[(size_t)a * DK + c] * u[a];
        }
        dkt[c] += b * (gw - alpha * su);
      }
      /* G <- alpha (G - b u k_t^T) */
      for (int a = 0; a < DV; ++a) {
        double* Grow = G + (size_t)a * DK;
        const double bu = b * u[a];
        for (int c = 0; c < DK; ++c) Grow[c] = alpha * (Grow[c] - bu * kt[c]);
      }
    }
  }
  if (J->dS0) memcpy(J->dS0 + ((size_t)n * Hv + j) * SS, G, SS * sizeof(double));
  free(ckpt); free(states); free(G); free(p); free(u); free(w);
  return 0;
}

static void* worker(void* arg) {
  oracle_job* J = (oracle_job*)arg;
  const size_t SS = (size_t)J->DV * J->DK;
  double* S = (double*)malloc(SS * sizeof(double));
  double* p = (double*)malloc((size_t)J->DV * sizeof(double));
  if (!S || !p) {
    pthread_mutex_lock(&J->lock);
    J->failed = 1;
    pthread_mutex_unlock(&J->lock);
    free(S); free(p);
    return NULL;
  }
  const int G = J->Hv / J->Hk;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    const int unit = J->next_unit++;
    pthread_mutex_unlock(&J->lock);
    if (unit >= J->n_units) break;
    const int n = unit / J->Hk, i = unit % J->Hk;
    for (int jj = 0; jj < G; ++jj) {
      const int j = i * G + jj;
      if (J->backward) {
        if (run_backward_head(J, n, i, j) != 0) {
          pthread_mutex_lock(&J->lock);
          J->failed = 1;
          pthread_mutex_unlock(&J->lock);
        }
      } else {
        run_forward_head(J, n, i, j, S, p);
      }
    }
  }
  free(S); free(p);
  return NULL;
}

static int run_job(oracle_job* J, int nthreads) {
  if (J->num_seqs < 0 || J->Hk <= 0 || J->Hv <= 0 || J->Hv % J->Hk != 0 || J->DK <= 0 ||
      J->DV <= 0)
    return -2;
  J->chunk_offset = (int64_t*)malloc((size_t)(J->num_seqs + 1) * sizeof(int64_t));
  if (!J->chunk_offset) return -1;
  J->chunk_offset[0] = 0;
  for (int n = 0; n < J->num_seqs; ++n) {
    const int64_t L = J->cu[n + 1] - J->cu[n];
    if (L < 0) { free(J->chunk_offset); return -2; }
    J->chunk_offset[n + 1] = J->chunk_offset[n] + (L + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
  }
  J->n_units = J->num_seqs * J->Hk;
  J->next_unit = 0;
  J->failed = 0;
  pthread_mutex_init(&J->lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > J->n_units) nthreads = J->n_units > 0 ? J->n_units : 1;
  pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
  int started = 0;
  if (th) {
    for (int w = 0; w < nthreads; ++w) {
      if (pthread_create(&th[w], NULL, worker, J) != 0) break;
      ++started;
    }
  }
  if (started == 0) worker(J); /* no threads available: run inline */
  for (int w = 0; w < started; ++w) pthread_join(th[w], NULL);
  free(th);
  pthread_mutex_destroy(&J->lock);
  free(J->chunk_offset);
  J->chunk_offset = NULL;
  return J->failed ? -1 : 0;
}

/* Forward.  o, S_T and S_chunks may each be NULL (not computed).  S0 may be
 * NULL (zero initial state).  Returns 0 on success, -1 on allocation failure,
 * -2 on an invalid argument. */
int gdr_oracle_forward(int num_seqs, const int64_t* cu_seqlens, int Hk, int Hv, int DK, int DV,
                       double scale, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, const double* S0, double* o,
                       double* S_T, double* S_chunks, int nthreads) {
  oracle_job J;
  memset(&J, 0, sizeof(J));
  J.num_seqs = num_seqs; J.cu = cu_seqlens;
  J.Hk = Hk; J.Hv = Hv; J.DK = DK; J.DV = DV; J.scale = scale;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.S0 = S0;
  J.o = o; J.S_T = S_T; J.S_chunks = S_chunks;
  J.backward = 0;
  return run_job(&J, nthreads);
}

/* Backward.  dq and dk are overwritten (zeroed here, then summed over the
 * v-heads of each group).  dO and dS_T may be NULL (zero).  dS0 may be NULL
 * (not returned).  Same return codes as the forward. */
int gdr_oracle_backward(int num_seqs, const int64_t* cu_seqlens, int Hk, int Hv, int DK, int DV,
                        double scale, const double* q, const double* k, const double* v,
                        const double* g, const double* beta, const double* S0, const double* dO,
                        const double* dS_T, double* dq, double* dk, double* dv, double* dg,
                        double* dbeta, double* dS0, int nthreads) {
  oracle_job J;
  memset(&J, 0, sizeof(J));
  if (num_seqs < 0) return -2;
  const int64_t T_total = num_seqs > 0 ? cu_seqlens[num_seqs] : 0;
  memset(dq, 0, (size_t)T_total * Hk * DK * sizeof(double));
  memset(dk, 0, (size_t)T_total * Hk * DK * sizeof(double));
  J.num_seqs = num_seqs; J.cu = cu_seqlens;
  J.Hk = Hk; J.Hv = Hv; J.DK = DK; J.DV = DV; J.scale = scale;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.S0 = S0;
  J.dO = dO; J.dS_T = dS_T;
  J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dS0 = dS0;
  J.backward = 1;
  return run_job(&J, nthreads);
}
