/*
 * Oracle for the head-wise recurrent scan: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code. The CUDA library shares nothing with it.
 *
 * What it computes follows the FlashRNN announcement (hottg.com/neural/9889,
 * "FlashRNN: optimising RNNs on modern hardware", usage example): per batch
 * row b and head n, for t = 0..T-1,
 *     rec_g = h_{t-1} . R[g,n] + b[g,n]       (row vector h times a D x D block)
 *     x_g   = Wx[b,t,g,n,:]
 * followed by the pointwise update of one of four cells. The LSTM cell and
 * the row-vector orientation follow developnotes "deep learning operators",
 * section 5.3 LSTM (MyLSTM.forward: gates = x.Wi + h.Wh + bias, sliced
 * i, f, g, o). GRU, Elman and sLSTM are not written out on the pages; the
 * readings used here are listed in rnn_oracle.c beside each cell.
 *
 * Layouts (row-major, dense):
 *   Wx      [B][T][G][N][D]     R  [G][N][D][D] (R[g][n][i][j], i = input unit)
 *   bias    [G][N][D]           s0 [S][B][1][N][D]
 *   states  [S][B][T][N][D]     last [S][B][1][N][D]
 * s0 == NULL means all-zero initial states. Output `states` holds the state
 * after each of the T steps (the initial state is not repeated in it).
 *
 * Backward: dstates [S][B][T][N][D] (may be NULL), dlast [S][B][1][N][D]
 * (may be NULL, added to step T-1), outputs dWx, dR, db, ds0 in the layouts of
 * their primal inputs; any output pointer may be NULL.
 *
 * Return value: 0 on success, -1 on bad arguments.
 */
#ifndef RNN_ORACLE_H
#define RNN_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_LSTM = 0, ORACLE_GRU = 1, ORACLE_ELMAN = 2, ORACLE_SLSTM = 3, ORACLE_SLSTM_LOGSIG = 4 };

/* flags: ORACLE_ROUND_BF16 = the bfloat16 storage mode, in which the operands
 * of every recurrent contraction (h_{t-1} in h.R, the recurrent-branch
 * gradient in dh = dr.R^T and in dR, db) are bfloat16 values; arithmetic and
 * carried states stay fp64. 0 = plain fp64 throughout. */
enum { ORACLE_ROUND_BF16 = 1 };

int oracle_num_gates(int fn);
int oracle_num_states(int fn);

int oracle_fwd(int fn, int B, int T, int N, int D,
               const double *Wx, const double *R, const double *bias,
               const double *s0, double *states, double *last, int flags,
               int nthreads);

int oracle_bwd(int fn, int B, int T, int N, int D,
               const double *Wx, const double *R, const double *bias,
               const double *s0, const double *dstates, const double *dlast,
               double *dWx, double *dR, double *db, double *ds0, int flags,
               int nthreads);

#ifdef __cplusplus
}
#endif
#endif
