/*
 * Oracle for the head-wise recurrent scan (fp64, CPU). TEST INFRASTRUCTURE:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * Sources (see rnn_oracle.h for layouts):
 *  - FlashRNN announcement (hottg.com/neural/9889), usage example: the
 *    functional call flashrnn(Wx, R, b, states, function) over Wx[B,T,G,N,D],
 *    R[G,N,D,D], b[G,N,D], states[S,B,1,N,D], returning states[S,B,T,N,D]
 *    and the last states; functions lstm, gru, elman, slstm; heads independent.
 *  - developnotes "deep learning operators", section 5.3 LSTM, MyLSTM.forward:
 *    gates = x.W_ih + h.W_hh + (bias_ih + bias_hh), slices i, f, g, o;
 *    sigmoid, sigmoid, tanh, sigmoid; c = f*c + i*g; h = o*tanh(c); zero
 *    initial states when none are given.
 *
 * Readings where the pages are silent (each repeated beside its cell):
 *  - GRU gates r, z, n; the reset gate multiplies the whole recurrent branch
 *    of n including its bias: n = tanh(x_n + r*(h.R_n + b_n));
 *    h' = (1-z)*n + z*h.
 *  - Elman: h' = tanh(x + h.R + b).
 *  - sLSTM gates i, f, z, o; states h, c, n, m; exponential input and forget
 *    gates (log f = a_f) with the stabiliser m:
 *    m' = max(a_f + m, a_i), i' = exp(a_i - m'), f' = exp(a_f + m - m'),
 *    c' = f' c + i' tanh(a_z), n' = f' n + i', h' = sigmoid(a_o) c'/n'.
 *    At a tie of the max the derivative goes to the a_f + m branch.
 *  - The sigmoid-forget sLSTM (function 4) is the other reading of that gate:
 *    log f = log sigmoid(a_f) in place of a_f in every formula above.
 *
 * The backward is back-propagation through time written by hand: the exact
 * derivative of the forward formulas above, step by step in reverse.
 */
#include "rnn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MAXG 4
#define MAXS 4

int oracle_num_gates(int fn) {
  switch (fn) {
    case ORACLE_LSTM: return 4;
    case ORACLE_GRU: return 3;
    case ORACLE_ELMAN: return 1;
    case ORACLE_SLSTM: return 4;
    case ORACLE_SLSTM_LOGSIG: return 4;
  }
  return -1;
}

int oracle_num_states(int fn) {
  switch (fn) {
    case ORACLE_LSTM: return 2;
    case ORACLE_GRU: return 1;
    case ORACLE_ELMAN: return 1;
    case ORACLE_SLSTM: return 4;
    case ORACLE_SLSTM_LOGSIG: return 4;
  }
  return -1;
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }
/* log sigmoid(v) = -log(1 + exp(-v)), written so that neither branch overflows */
static double log_sigmoid(double v) { return (v < 0.0 ? v : 0.0) - log1p(exp(-fabs(v))); }

/* ---- one cell, one unit --------------------------------------------------
 * x[g]   : the input pre-activation Wx[b,t,g,n,j]
 * rec[g] : the recurrent branch h_{t-1}.R[g,n][:,j] + bias[g,n,j]
 * sp[s]  : the states before the step, sn[s]: after (s = 0 is always h)
 */
static void cell_fwd(int fn, const double *x, const double *rec,
                     const double *sp, double *sn) {
  if (fn == ORACLE_LSTM) {
    /* developnotes 5.3: i, f, g, o; c = f c + i g; h = o tanh(c) */
    double i = sigmoid(x[0] + rec[0]);
    double f = sigmoid(x[1] + rec[1]);
    double g = tanh(x[2] + rec[2]);
    double o = sigmoid(x[3] + rec[3]);
    double c = f * sp[1] + i * g;
    sn[1] = c;
    sn[0] = o * tanh(c);
  } else if (fn == ORACLE_GRU) {
    /* reading: reset gate applied to the recurrent branch of n (with b_n) */
    double r = sigmoid(x[0] + rec[0]);
    double z = sigmoid(x[1] + rec[1]);
    double nn = tanh(x[2] + r * rec[2]);
    sn[0] = (1.0 - z) * nn + z * sp[0];
  } else if (fn == ORACLE_ELMAN) {
    sn[0] = tanh(x[0] + rec[0]);
  } else { /* ORACLE_SLSTM, ORACLE_SLSTM_LOGSIG */
    double ai = x[0] + rec[0], af = x[1] + rec[1];
    double az = x[2] + rec[2], ao = x[3] + rec[3];
    double mp = sp[3];
    double lf = (fn == ORACLE_SLSTM_LOGSIG) ? log_sigmoid(af) : af; /* log f */
    double m = (lf + mp >= ai) ? lf + mp : ai;
    double ig = exp(ai - m);
    double fg = exp(lf + mp - m);
    double c = fg * sp[1] + ig * tanh(az);
    double n = fg * sp[2] + ig;
    sn[1] = c;
    sn[2] = n;
    sn[3] = m;
    sn[0] = sigmoid(ao) * c / n;
  }
}

/* Backward of cell_fwd for one unit. dsn[s] is the total gradient reaching the
 * state after the step. Outputs: dx[g] (gradient of x), drec[g] (gradient of
 * the recurrent branch), dsp[s] (gradient of the previous states through the
 * cell itself; the part of dh_{t-1} through R is added by the caller). */
static void cell_bwd(int fn, const double *x, const double *rec,
                     const double *sp, const double *sn, const double *dsn,
                     double *dx, double *drec, double *dsp) {
  int s;
  for (s = 0; s < MAXS; ++s) dsp[s] = 0.0;
  if (fn == ORACLE_LSTM) {
    double i = sigmoid(x[0] + rec[0]);
    double f = sigmoid(x[1] + rec[1]);
    double g = tanh(x[2] + rec[2]);
    double o = sigmoid(x[3] + rec[3]);
    double tc = tanh(sn[1]);
    double dh = dsn[0];
    double dc = dsn[1] + dh * o * (1.0 - tc * tc);
    double d_o = dh * tc;
    double di = dc * g, df = dc * sp[1], dg = dc * i;
    dx[0] = di * i * (1.0 - i);
    dx[1] = df * f * (1.0 - f);
    dx[2] = dg * (1.0 - g * g);
    dx[3] = d_o * o * (1.0 - o);
    for (s = 0; s < 4; ++s) drec[s] = dx[s];
    dsp[1] = dc * f;
  } else if (fn == ORACLE_GRU) {
    double r = sigmoid(x[0] + rec[0]);
    double z = sigmoid(x[1] + rec[1]);
    double nn = tanh(x[2] + r * rec[2]);
    double dh = dsn[0];
    double dn = dh * (1.0 - z);
    double dz = dh * (sp[0] - nn);
    double dan = dn * (1.0 - nn * nn);
    double dr = dan * rec[2];
    dx[0] = dr * r * (1.0 - r);
    dx[1] = dz * z * (1.0 - z);
    dx[2] = dan;
    drec[0] = dx[0];
    drec[1] = dx[1];
    drec[2] = dan * r;
    dsp[0] = dh * z;
  } else if (fn == ORACLE_ELMAN) {
    double h = sn[0];
    dx[0] = dsn[0] * (1.0 - h * h);
    drec[0] = dx[0];
  } else { /* ORACLE_SLSTM, ORACLE_SLSTM_LOGSIG */
    double ai = x[0] + rec[0], af = x[1] + rec[1];
    double az = x[2] + rec[2], ao = x[3] + rec[3];
    double cp = sp[1], np = sp[2], mp = sp[3];
    double c = sn[1], n = sn[2], m = sn[3];
    double lf = (fn == ORACLE_SLSTM_LOGSIG) ? log_sigmoid(af) : af; /* log f */
    double ig = exp(ai - m);
    double fg = exp(lf + mp - m);
    double zt = tanh(az);
    double o = sigmoid(ao);
    double dh = dsn[0];
    double dy = dh * o;
    double dc = dsn[1] + dy / n;
    double dn = dsn[2] - dy * c / (n * n);
    double dm = dsn[3];
    double d_o = dh * c / n;
    double dfg = dc * cp + dn * np;
    double dig = dc * zt + dn;
    double dzt = dc * ig;
    double dai = dig * ig;
    double dlf = dfg * fg; /* gradient reaching log f */
    double dmp = dfg * fg;
    dm -= dig * ig + dfg * fg;
    if (lf + mp >= ai) { /* tie goes to the forget branch */
      dlf += dm;
      dmp += dm;
    } else {
      dai += dm;
    }
    dx[0] = dai;
    /* d log sigmoid(a) / da = sigmoid(-a) */
    dx[1] = (fn == ORACLE_SLSTM_LOGSIG) ? dlf * sigmoid(-af) : dlf;
    dx[2] = dzt * (1.0 - zt * zt);
    dx[3] = d_o * o * (1.0 - o);
    for (s = 0; s < 4; ++s) drec[s] = dx[s];
    dsp[1] = dc * fg;
    dsp[2] = dn * fg;
    dsp[3] = dmp;
  }
}

/* ---- one (b, n) sequence -------------------------------------------------- */

typedef struct {
  int fn, B, T, N, D, G, S, flags;
  const double *Wx, *R, *bias, *s0, *dstates, *dlast;
  double *states, *last, *dWx, *dR, *db, *ds0;
} problem_t;

#define IDX_WX(p, b, t, g, n, j) \
  ((((((size_t)(b) * (p)->T + (t)) * (p)->G + (g)) * (p)->N + (n)) * (p)->D) + (j))
#define IDX_R(p, g, n, i, j) \
  (((((size_t)(g) * (p)->N + (n)) * (p)->D + (i)) * (p)->D) + (j))
#define IDX_B(p, g, n, j) ((((size_t)(g) * (p)->N + (n)) * (p)->D) + (j))
/* states-like tensor with time extent TT: [S][B][TT][N][D] */
#define IDX_ST(p, TT, s, b, t, n, j) \
  ((((((size_t)(s) * (p)->B + (b)) * (TT) + (t)) * (p)->N + (n)) * (p)->D) + (j))

/* bfloat16 storage mode (ORACLE_ROUND_BF16): the operands of the recurrent
 * contractions are bfloat16 values, the arithmetic stays exact (fp64 here).
 * The value is first rounded to binary32 (as an fp32 computation would hold
 * it) and then to bfloat16 with round-to-nearest-even on the 16 dropped bits. */
static double round_bf16(double v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, sizeof(u));
  if ((u & 0x7f800000u) != 0x7f800000u) { /* finite: round, else keep */
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
  }
  memcpy(&f, &u, sizeof(f));
  return (double)f;
}

static double operand(const problem_t *p, double v) {
  return (p->flags & ORACLE_ROUND_BF16) ? round_bf16(v) : v;
}

/* rec[g*D + j] = h . R[g,n][:, j] + bias[g,n,j] */
static void recurrent_branch(const problem_t *p, int n, const double *h,
                             double *rec) {
  int g, i, j, D = p->D;
  for (g = 0; g < p->G; ++g) {
    for (j = 0; j < D; ++j) rec[g * D + j] = p->bias[IDX_B(p, g, n, j)];
    for (i = 0; i < D; ++i) {
      double hi = operand(p, h[i]);
      const double *row = p->R + IDX_R(p, g, n, i, 0);
      for (j = 0; j < D; ++j) rec[g * D + j] += hi * row[j];
    }
  }
}

/* Runs the forward of sequence (b, n). If tape_x/tape_rec/tape_s are given,
 * records x, rec and the states after every step (for the backward). */
static void seq_fwd(const problem_t *p, int b, int n, double *tape_x,
                    double *tape_rec, double *tape_s) {
  int D = p->D, G = p->G, S = p->S, t, g, s, j;
  double *cur = (double *)calloc((size_t)S * D, sizeof(double));
  double *nxt = (double *)calloc((size_t)S * D, sizeof(double));
  double *rec = (double *)calloc((size_t)G * D, sizeof(double));
  double xg[MAXG], rg[MAXG], sp[MAXS], sn[MAXS];
  if (p->s0)
    for (s = 0; s < S; ++s)
      for (j = 0; j < D; ++j) cur[s * D + j] = p->s0[IDX_ST(p, 1, s, b, 0, n, j)];
  for (t = 0; t < p->T; ++t) {
    recurrent_branch(p, n, cur, rec); /* cur[0..D) is h_{t-1} */
    for (j = 0; j < D; ++j) {
      for (g = 0; g < G; ++g) {
        xg[g] = p->Wx[IDX_WX(p, b, t, g, n, j)];
        rg[g] = rec[g * D + j];
        if (tape_x) {
          tape_x[((size_t)t * G + g) * D + j] = xg[g];
          tape_rec[((size_t)t * G + g) * D + j] = rg[g];
        }
      }
      for (s = 0; s < S; ++s) sp[s] = cur[s * D + j];
      cell_fwd(p->fn, xg, rg, sp, sn);
      for (s = 0; s < S; ++s) nxt[s * D + j] = sn[s];
    }
    for (s = 0; s < S; ++s)
      for (j = 0; j < D; ++j) {
        double v = nxt[s * D + j];
        cur[s * D + j] = v;
        if (p->states) p->states[IDX_ST(p, p->T, s, b, t, n, j)] = v;
        if (tape_s) tape_s[((size_t)t * S + s) * D + j] = v;
      }
  }
  if (p->last)
    for (s = 0; s < S; ++s)
      for (j = 0; j < D; ++j) p->last[IDX_ST(p, 1, s, b, 0, n, j)] = cur[s * D + j];
  free(cur);
  free(nxt);
  free(rec);
}

/* Backward of sequence (b, n); accumulates into dR_acc / db_acc. */
static void seq_bwd(const problem_t *p, int b, int n, double *dR_acc,
                    double *db_acc) {
  int D = p->D, G = p->G, S = p->S, T = p->T, t, g, s, i, j;
  double *tx = (double *)malloc(sizeof(double) * ((size_t)T * G * D + 1));
  double *tr = (double *)malloc(sizeof(double) * ((size_t)T * G * D + 1));
  double *ts = (double *)malloc(sizeof(double) * ((size_t)T * S * D + 1));
  double *init = (double *)calloc((size_t)S * D, sizeof(double));
  double *carry = (double *)calloc((size_t)S * D, sizeof(double));
  double *ncarry = (double *)calloc((size_t)S * D, sizeof(double));
  double *drec = (double *)calloc((size_t)G * D, sizeof(double));
  double xg[MAXG], rg[MAXG], sp[MAXS], sn[MAXS], dsn[MAXS];
  double dxg[MAXG], drg[MAXG], dsp[MAXS];
  problem_t q = *p;
  q.states = NULL;
  q.last = NULL;
  if (p->s0)
    for (s = 0; s < S; ++s)
      for (j = 0; j < D; ++j) init[s * D + j] = p->s0[IDX_ST(p, 1, s, b, 0, n, j)];
  seq_fwd(&q, b, n, tx, tr, ts);

  for (t = T - 1; t >= 0; --t) {
    const double *prev = (t > 0) ? ts + (size_t)(t - 1) * S * D : init;
    const double *now = ts + (size_t)t * S * D;
    memset(ncarry, 0, sizeof(double) * S * D);
    for (j = 0; j < D; ++j) {
      for (g = 0; g < G; ++g) {
        xg[g] = tx[((size_t)t * G + g) * D + j];
        rg[g] = tr[((size_t)t * G + g) * D + j];
      }
      for (s = 0; s < S; ++s) {
        sp[s] = prev[s * D + j];
        sn[s] = now[s * D + j];
        dsn[s] = carry[s * D + j];
        if (p->dstates) dsn[s] += p->dstates[IDX_ST(p, T, s, b, t, n, j)];
        if (p->dlast && t == T - 1) dsn[s] += p->dlast[IDX_ST(p, 1, s, b, 0, n, j)];
      }
      cell_bwd(p->fn, xg, rg, sp, sn, dsn, dxg, drg, dsp);
      for (g = 0; g < G; ++g) {
        if (p->dWx) p->dWx[IDX_WX(p, b, t, g, n, j)] = dxg[g];
        drec[g * D + j] = operand(p, drg[g]);
        db_acc[IDX_B(p, g, n, j)] += drec[g * D + j];
      }
      for (s = 0; s < S; ++s) ncarry[s * D + j] = dsp[s];
    }
    /* through the recurrent branch: dR += h_{t-1}^T drec ; dh_{t-1} += drec . R^T */
    for (g = 0; g < G; ++g)
      for (i = 0; i < D; ++i) {
        double hi = operand(p, prev[i]); /* s = 0 is h */
        const double *row = p->R + IDX_R(p, g, n, i, 0);
        double *drow = dR_acc + IDX_R(p, g, n, i, 0);
        double acc = 0.0;
        for (j = 0; j < D; ++j) {
          drow[j] += hi * drec[g * D + j];
          acc += row[j] * drec[g * D + j];
        }
        ncarry[i] += acc;
      }
    memcpy(carry, ncarry, sizeof(double) * S * D);
  }
  if (T == 0 && p->dlast) /* last == s0 */
    for (s = 0; s < S; ++s)
      for (j = 0; j < D; ++j) carry[s * D + j] = p->dlast[IDX_ST(p, 1, s, b, 0, n, j)];
  if (p->ds0)
    for (s = 0; s < S; ++s)
      for (j = 0; j < D; ++j) p->ds0[IDX_ST(p, 1, s, b, 0, n, j)] = carry[s * D + j];
  free(tx);
  free(tr);
  free(ts);
  free(init);
  free(carry);
  free(ncarry);
  free(drec);
}

/* ---- threading over independent sequences -------------------------------- */

typedef struct {
  const problem_t *p;
  int first, count, backward;
  double *dR_acc, *db_acc;
} job_t;

static void *run_job(void *arg) {
  job_t *jb = (job_t *)arg;
  int k;
  for (k = jb->first; k < jb->first + jb->count; ++k) {
    int b = k / jb->p->N, n = k % jb->p->N;
    if (jb->backward)
      seq_bwd(jb->p, b, n, jb->dR_acc, jb->db_acc);
    else
      seq_fwd(jb->p, b, n, NULL, NULL, NULL);
  }
  return NULL;
}

static int run(problem_t *p, int backward, int nthreads) {
  int nseq = p->B * p->N, k, w;
  size_t nR = (size_t)p->G * p->N * p->D * p->D, nb = (size_t)p->G * p->N * p->D;
  job_t *jobs;
  pthread_t *tids;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nseq) nthreads = nseq > 0 ? nseq : 1;
  jobs = (job_t *)calloc(nthreads, sizeof(job_t));
  tids = (pthread_t *)calloc(nthreads, sizeof(pthread_t));
  for (w = 0, k = 0; w < nthreads; ++w) {
    int cnt = nseq / nthreads + (w < nseq % nthreads ? 1 : 0);
    jobs[w].p = p;
    jobs[w].first = k;
    jobs[w].count = cnt;
    jobs[w].backward = backward;
    if (backward) {
      jobs[w].dR_acc = (double *)calloc(nR + 1, sizeof(double));
      jobs[w].db_acc = (double *)calloc(nb + 1, sizeof(double));
    }
    k += cnt;
  }
  if (nthreads == 1) {
    run_job(&jobs[0]);
  } else {
    for (w = 0; w < nthreads; ++w) pthread_create(&tids[w], NULL, run_job, &jobs[w]);
    for (w = 0; w < nthreads; ++w) pthread_join(tids[w], NULL);
  }
  if (backward) {
    size_t e;
    if (p->dR) memset(p->dR, 0, nR * sizeof(double));
    if (p->db) memset(p->db, 0, nb * sizeof(double));
    for (w = 0; w < nthreads; ++w) {
      if (p->dR)
        for (e = 0; e < nR; ++e) p->dR[e] += jobs[w].dR_acc[e];
      if (p->db)
        for (e = 0; e < nb; ++e) p->db[e] += jobs[w].db_acc[e];
      free(jobs[w].dR_acc);
      free(jobs[w].db_acc);
    }
  }
  free(jobs);
  free(tids);
  return 0;
}

static int setup(problem_t *p, int fn, int B, int T, int N, int D, int flags) {
  memset(p, 0, sizeof(*p));
  p->flags = flags;
  if (fn < 0 || fn > 4 || B < 0 || T < 0 || N < 0 || D < 0) return -1;
  p->fn = fn;
  p->B = B;
  p->T = T;
  p->N = N;
  p->D = D;
  p->G = oracle_num_gates(fn);
  p->S = oracle_num_states(fn);
  return 0;
}

int oracle_fwd(int fn, int B, int T, int N, int D, const double *Wx,
               const double *R, const double *bias, const double *s0,
               double *states, double *last, int flags, int nthreads) {
  problem_t p;
  if (setup(&p, fn, B, T, N, D, flags)) return -1;
  if ((T > 0 && !Wx) || !R || !bias) return -1;
  p.Wx = Wx;
  p.R = R;
  p.bias = bias;
  p.s0 = s0;
  p.states = states;
  p.last = last;
  return run(&p, 0, nthreads);
}

int oracle_bwd(int fn, int B, int T, int N, int D, const double *Wx,
               const double *R, const double *bias, const double *s0,
               const double *dstates, const double *dlast, double *dWx,
               double *dR, double *db, double *ds0, int flags, int nthreads) {
  problem_t p;
  if (setup(&p, fn, B, T, N, D, flags)) return -1;
  if ((T > 0 && !Wx) || !R || !bias) return -1;
  p.Wx = Wx;
  p.R = R;
  p.bias = bias;
  p.s0 = s0;
  p.dstates = dstates;
  p.dlast = dlast;
  p.dWx = dWx;
  p.dR = dR;
  p.db = db;
  p.ds0 = ds0;
  return run(&p, 1, nthreads);
}
