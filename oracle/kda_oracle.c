/*
 * kda_oracle.c -- the oracle for the Kimi Delta Attention (KDA) token mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads, links or calls this file:
 * only the test suite, the package smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it is: a plain, slow, obviously correct CPU restatement of what the KDA layer
 * computes, in fp64, one token at a time.  Inputs are read in their storage type (fp32, or
 * bf16 given as raw 16-bit patterns) and widened to double exactly; nothing is rounded on
 * the way.  Sources (web pages, cited by title and section):
 *
 *   [Grouped]  "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches",
 *              section "KDA replaces a token list with a recurrent matrix".
 *   [Headers]  "Ling-3.1-flash: a 560B hybrid-attention MoE, counted from its safetensors
 *              headers", section "How KDA and MLA split the work", the state equation.
 *   [Budget]   "Ling-3.1-flash: What 63 Linear-Attention Layers Do to the KV Budget",
 *              section "The memory math".
 *
 * The per-head recurrence (state S is d_k x d_v; row i = key channel, column j = value
 * channel), for each token t of a sequence:
 *
 *   a   = exp(max(g_t, g_min))          per-channel retention; g_min = -5 is the safe
 *                                        forget gate's log-retention lower bound [Grouped]
 *   S'  = Diag(a) S                     channel-wise decay, Diag(alpha_t) S_{t-1} [Headers]
 *   p   = S'^T k                        the state's prediction for the current key
 *   S   = S' + beta * k (v - p)^T       delta-rule write: the prediction for k is corrected
 *                                        toward v, not an uncorrected k v^T add [Grouped]
 *   o   = scale * S^T q                 read after the write, o_t = S_t^T q_t [Headers]
 *
 * q and k are L2-normalised per head first when requested ("The KDA kernel normalizes
 * queries and keys" [Grouped]); when output-gate logits are given, the output is
 * RMS-normalised over d_v, scaled by the norm weight and by a sigmoid gate ("An output
 * normalization and sigmoid gate precede the projection" [Grouped]).
 *
 * The short convolution ("Each projection passes through its own causal short
 * convolution of width four with SiLU activation" [Grouped]) is oracle_prologue below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

/* Widen one stored element to double.  bf16 is the top half of an IEEE-754 binary32. */
static double load_elem(const void *base, int dtype, int64_t idx) {
  if (dtype == ORACLE_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  if (dtype == ORACLE_F64) return ((const double *)base)[idx];
  return (double)((const float *)base)[idx];
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------------------ */
/* Recurrence                                                                            */
/* ------------------------------------------------------------------------------------ */

typedef struct {
  int H, dk, dv;
  int n_seqs;
  const int32_t *cu_seqlens; /* [n_seqs + 1], token offsets of each packed sequence   */
  const void *q, *k, *v;     /* [T_tot, H, dk|dk|dv]                                  */
  int qkv_dtype;             /* ORACLE_F32, ORACLE_BF16 or ORACLE_F64                  */
  const float *g;            /* [T_tot, H, dk] log-retention before the clamp          */
  const float *beta;         /* [T_tot, H] write strength, already in (0, 1)           */
  const void *init_state;    /* [n_seqs, H, dk, dv] or NULL (zeros)                    */
  int state_dtype;
  const void *gate;          /* [T_tot, H, dv] output-gate logits, or NULL (no norm)   */
  int gate_dtype;
  const float *norm_w;       /* [dv] output-norm weight, or NULL (ones)                */
  double scale, l2_eps, norm_eps, g_min;
  int qk_l2norm;
  int n_units;               /* work list: (sequence, head) pairs                      */
  const int32_t *units;      /* [n_units][2]                                           */
  const int64_t *out_offset; /* [n_units] offset, in doubles, of the unit's [len, dv]   */
  double *out;               /* outputs                                                */
  double *final_state;       /* [n_units, dk, dv] or NULL                              */
  double *state_norm;        /* [sum of lens] Frobenius norm of S after each token,    */
                             /* laid out like out / dv; or NULL                        */
  int n_threads;
} oracle_kda_args;

typedef struct {
  const oracle_kda_args *a;
  int first, step;
} worker_arg;

static void run_unit(const oracle_kda_args *a, int u, double *S, double *qv, double *kv,
                     double *vv, double *p, double *o) {
  const int H = a->H, dk = a->dk, dv = a->dv;
  const int n = a->units[2 * u], h = a->units[2 * u + 1];
  const int64_t bos = a->cu_seqlens[n], eos = a->cu_seqlens[n + 1];

  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j)
      S[i * dv + j] = a->init_state
                          ? load_elem(a->init_state, a->state_dtype,
                                      (((int64_t)n * H + h) * dk + i) * dv + j)
                          : 0.0;

  for (int64_t t = bos; t < eos; ++t) {
    const int64_t qk_base = (t * H + h) * dk, v_base = (t * H + h) * dv;
    for (int i = 0; i < dk; ++i) {
      qv[i] = load_elem(a->q, a->qkv_dtype, qk_base + i);
      kv[i] = load_elem(a->k, a->qkv_dtype, qk_base + i);
    }
    for (int j = 0; j < dv; ++j) vv[j] = load_elem(a->v, a->qkv_dtype, v_base + j);

    if (a->qk_l2norm) { /* x / sqrt(sum x^2 + eps) */
      double sq = 0.0, sk = 0.0;
      for (int i = 0; i < dk; ++i) {
        sq += qv[i] * qv[i];
        sk += kv[i] * kv[i];
      }
      const double rq = 1.0 / sqrt(sq + a->l2_eps), rk = 1.0 / sqrt(sk + a->l2_eps);
      for (int i = 0; i < dk; ++i) {
        qv[i] *= rq;
        kv[i] *= rk;
      }
    }
    const double b = (double)a->beta[t * H + h];

    /* decay: S' = Diag(exp(max(g, g_min))) S */
    for (int i = 0; i < dk; ++i) {
      double gi = (double)a->g[qk_base + i];
      if (gi < a->g_min) gi = a->g_min;
      const double alpha = exp(gi);
      for (int j = 0; j < dv; ++j) S[i * dv + j] *= alpha;
    }
    /* prediction p = S'^T k */
    for (int j = 0; j < dv; ++j) p[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) p[j] += S[i * dv + j] * kv[i];
    /* delta-rule write: S = S' + beta k (v - p)^T */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += b * kv[i] * (vv[j] - p[j]);
    /* read after write: o = scale S^T q */
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) o[j] += S[i * dv + j] * qv[i];
    for (int j = 0; j < dv; ++j) o[j] *= a->scale;

    if (a->gate) { /* o / sqrt(mean(o^2) + eps) * w * sigmoid(gate) */
      double ms = 0.0;
      for (int j = 0; j < dv; ++j) ms += o[j] * o[j];
      ms /= dv;
      const double r = 1.0 / sqrt(ms + a->norm_eps);
      for (int j = 0; j < dv; ++j) {
        const double w = a->norm_w ? (double)a->norm_w[j] : 1.0;
        o[j] = o[j] * r * w * sigmoid(load_elem(a->gate, a->gate_dtype, v_base + j));
      }
    }

    double *dst = a->out + a->out_offset[u] + (t - bos) * dv;
    for (int j = 0; j < dv; ++j) dst[j] = o[j];

    if (a->state_norm) {
      double f = 0.0;
      for (int i = 0; i < dk * dv; ++i) f += S[i] * S[i];
      a->state_norm[a->out_offset[u] / dv + (t - bos)] = sqrt(f);
    }
  }

  if (a->final_state) memcpy(a->final_state + (int64_t)u * dk * dv, S, sizeof(double) * dk * dv);
}

static void *worker(void *arg) {
  const worker_arg *w = (const worker_arg *)arg;
  const oracle_kda_args *a = w->a;
  double *S = (double *)malloc(sizeof(double) * a->dk * a->dv);
  double *qv = (double *)malloc(sizeof(double) * a->dk);
  double *kv = (double *)malloc(sizeof(double) * a->dk);
  double *vv = (double *)malloc(sizeof(double) * a->dv);
  double *p = (double *)malloc(sizeof(double) * a->dv);
  double *o = (double *)malloc(sizeof(double) * a->dv);
  for (int u = w->first; u < a->n_units; u += w->step) run_unit(a, u, S, qv, kv, vv, p, o);
  free(S), free(qv), free(kv), free(vv), free(p), free(o);
  return NULL;
}

/* Runs every (sequence, head) unit of the work list.  Returns 0, or -1 on bad arguments. */
int oracle_kda_forward(const oracle_kda_args *a) {
  if (!a || a->H < 1 || a->dk < 1 || a->dv < 1 || a->n_seqs < 0 || !a->cu_seqlens || !a->q ||
      !a->k || !a->v || !a->g || !a->beta || !a->out || !a->out_offset || a->n_units < 0)
    return -1;
  for (int u = 0; u < a->n_units; ++u) {
    const int n = a->units[2 * u], h = a->units[2 * u + 1];
    if (n < 0 || n >= a->n_seqs || h < 0 || h >= a->H) return -1;
  }
  int nt = a->n_threads < 1 ? 1 : a->n_threads;
  if (nt > a->n_units) nt = a->n_units < 1 ? 1 : a->n_units;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
  worker_arg *wa = (worker_arg *)malloc(sizeof(worker_arg) * nt);
  for (int i = 0; i < nt; ++i) {
    wa[i].a = a, wa[i].first = i, wa[i].step = nt;
    pthread_create(&th[i], NULL, worker, &wa[i]);
  }
  for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
  free(th), free(wa);
  return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Prologue: width-4 causal short convolution + SiLU, q/k L2 norm, gate activations      */
/* ------------------------------------------------------------------------------------ */

typedef struct {
  int n_seqs;
  const int32_t *cu_seqlens; /* [n_seqs + 1]                                              */
  int H, d;                  /* channels C = 3 * H * d: q streams, then k, then v        */
  const void *x;             /* [T_tot, C] raw projections                               */
  int x_dtype;
  const void *w;             /* [C, 4]; w[c][j] multiplies x[t - 3 + j][c]                */
  int w_dtype;
  const void *conv_state_in; /* [n_seqs, 3, C] the 3 inputs before each sequence, oldest */
                             /* first, same storage type as x; or NULL (zeros)            */
  void *conv_state_out;      /* [n_seqs, 3, C] the last 3 inputs (raw copies) or NULL    */
  int l2norm_qk;             /* L2-normalise the q and k streams per head after SiLU     */
  double l2_eps;
  double *y;                 /* [T_tot, C] output                                        */
  /* gate activations (optional; all NULL to skip) */
  const float *beta_logit;   /* [T_tot, H]                                                */
  double *beta;              /* [T_tot, H] sigmoid(beta_logit)                            */
  const float *g_raw;        /* [T_tot, H, d]                                             */
  double *g;                 /* [T_tot, H, d] max(g_raw, g_min)                           */
  double g_min;
} oracle_prologue_args;

int oracle_prologue(const oracle_prologue_args *a) {
  if (!a || a->n_seqs < 0 || !a->cu_seqlens || a->H < 1 || a->d < 1 || !a->x || !a->w || !a->y)
    return -1;
  const int64_t C = 3LL * a->H * a->d;
  const size_t esz = a->x_dtype == ORACLE_BF16 ? 2 : 4;
  for (int n = 0; n < a->n_seqs; ++n) {
    const int64_t bos = a->cu_seqlens[n], eos = a->cu_seqlens[n + 1];
    for (int64_t t = bos; t < eos; ++t) {
      for (int64_t c = 0; c < C; ++c) {
        double acc = 0.0;
        for (int j = 0; j < 4; ++j) {
          const int64_t src = t - 3 + j; /* token feeding tap j */
          double xv;
          if (src >= bos)
            xv = load_elem(a->x, a->x_dtype, src * C + c);
          else if (a->conv_state_in) /* history row: 3 + (src - bos) in [0, 3) */
            xv = load_elem(a->conv_state_in, a->x_dtype, ((int64_t)n * 3 + 3 + (src - bos)) * C + c);
          else
            xv = 0.0;
          acc += load_elem(a->w, a->w_dtype, c * 4 + j) * xv;
        }
        a->y[t * C + c] = acc * sigmoid(acc); /* SiLU */
      }
      if (a->l2norm_qk) {
        for (int s = 0; s < 2; ++s) /* q and k streams */
          for (int h = 0; h < a->H; ++h) {
            double *row = a->y + t * C + ((int64_t)s * a->H + h) * a->d;
            double ss = 0.0;
            for (int i = 0; i < a->d; ++i) ss += row[i] * row[i];
            const double r = 1.0 / sqrt(ss + a->l2_eps);
            for (int i = 0; i < a->d; ++i) row[i] *= r;
          }
      }
    }
    if (a->conv_state_out) { /* the last three raw inputs, reaching into the old state */
      for (int r = 0; r < 3; ++r) {
        const int64_t src = eos - 3 + r;
        char *dst = (char *)a->conv_state_out + (((int64_t)n * 3 + r) * C) * esz;
        if (src >= bos)
          memcpy(dst, (const char *)a->x + src * C * esz, C * esz);
        else if (a->conv_state_in)
          memcpy(dst, (const char *)a->conv_state_in + (((int64_t)n * 3 + 3 + (src - bos)) * C) * esz,
                 C * esz);
        else
          memset(dst, 0, C * esz);
      }
    }
  }
  const int64_t T = a->n_seqs ? a->cu_seqlens[a->n_seqs] : 0;
  if (a->beta_logit && a->beta)
    for (int64_t i = 0; i < T * a->H; ++i) a->beta[i] = sigmoid((double)a->beta_logit[i]);
  if (a->g_raw && a->g)
    for (int64_t i = 0; i < T * a->H * a->d; ++i) {
      const double gi = (double)a->g_raw[i];
      a->g[i] = gi < a->g_min ? a->g_min : gi;
    }
  return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Payload arithmetic [Budget]: bytes of one layer's recurrent state for one sequence.   */
/* ------------------------------------------------------------------------------------ */
int64_t oracle_state_bytes(int H, int dk, int dv, int elem_bytes) {
  return (int64_t)H * dk * dv * elem_bytes;
}

/* Bytes of one layer's convolution tail for one sequence: 3 past inputs of 3*H*d channels. */
int64_t oracle_conv_tail_bytes(int H, int d, int width, int elem_bytes) {
  return (int64_t)(width - 1) * 3 * H * d * elem_bytes;
}
