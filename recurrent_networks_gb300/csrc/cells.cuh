// Pointwise cells of the head-wise recurrent scan, fp32 arithmetic.
//
// LSTM: developnotes "deep learning operators", section 5.3 LSTM
// (MyLSTM.forward): gates i,f,g,o with sigmoid, sigmoid, tanh, sigmoid;
// c = f c + i g; h = o tanh(c). GRU (r,z,n; reset gate on the recurrent
// branch of n including its bias; h' = (1-z) n + z h), Elman (h' = tanh a) and
// sLSTM (i,f,z,o; states h,c,n,m; exponential gates with stabiliser m, log f =
// a_f; the max's derivative goes to the forget branch on a tie) are the
// readings the FlashRNN announcement's function list (lstm, gru, elman,
// slstm) leaves to us. SLSTM_LS is the other reading of the sLSTM forget
// gate, a sigmoid: log f = log sigmoid(a_f), the rest unchanged.
//
// Tape record of one (t, b, n, unit), fp32, K = G + S (+1 for GRU) values:
//   LSTM  a_i a_f a_g a_o | h c
//   GRU   a_r a_z x_n q   | h        (q = rec_n, the recurrent branch of n)
//   Elman a               | h
//   sLSTM a_i a_f a_z a_o | h c n m   (also the sigmoid-forget sLSTM, SLSTM_LS)
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace rnn {

enum { LSTM = 0, GRU = 1, ELMAN = 2, SLSTM = 3, SLSTM_LS = 4 };

template <int FN> struct FnInfo;
template <> struct FnInfo<LSTM> { static constexpr int G = 4, S = 2, P = 4; };
template <> struct FnInfo<GRU> { static constexpr int G = 3, S = 1, P = 4; };
template <> struct FnInfo<ELMAN> { static constexpr int G = 1, S = 1, P = 1; };
template <> struct FnInfo<SLSTM> { static constexpr int G = 4, S = 4, P = 4; };
template <> struct FnInfo<SLSTM_LS> { static constexpr int G = 4, S = 4, P = 4; };
// P = number of "pre" values on the tape; tape width K = P + S.

__host__ __device__ constexpr int fn_gates(int fn) { return fn == 0 ? 4 : fn == 1 ? 3 : fn == 2 ? 1 : 4; }
__host__ __device__ constexpr int fn_states(int fn) { return fn == 0 ? 2 : fn == 1 ? 1 : fn == 2 ? 1 : 4; }
__host__ __device__ constexpr int fn_pre(int fn) { return fn == 1 ? 4 : fn_gates(fn); }
__host__ __device__ constexpr int fn_tape(int fn) { return fn_pre(fn) + fn_states(fn); }

// ---- transcendentals ------------------------------------------------------
// FAST = true builds the functions from the PTX base-2 exponential and
// reciprocal approximations (ex2.approx.ftz.f32, rcp.approx.ftz.f32, each
// within a few ulp of fp32):  sigmoid(x) = 1 / (1 + 2^(-x log2 e)),
// tanh(x) = 1 - 2 / (1 + 2^(2x log2 e)); absolute error ~1e-7, so a bf16
// rounding of h almost never lands on the other side of a tie because of it
// (tanh.approx.f32, at ~2^-11 relative error, flipped ~1 in 4 roundings).
// FAST = false calls CUDA's accurate tanhf / expf.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <bool FAST> __device__ __forceinline__ float f_tanh(float x) {
  if (FAST) return fmaf(-2.0f, rcp_fast(1.0f + exp2_fast(2.8853900817779268f * x)), 1.0f);
  return tanhf(x);
}
template <bool FAST> __device__ __forceinline__ float f_sigmoid(float x) {
  if (FAST) return rcp_fast(1.0f + exp2_fast(-1.4426950408889634f * x));
  return 1.0f / (1.0f + expf(-x));
}
template <bool FAST> __device__ __forceinline__ float f_exp(float x) {
  if (FAST) return exp2_fast(x * 1.4426950408889634f);
  return expf(x);
}
// log sigmoid(x) = min(x, 0) - log(1 + exp(-|x|)), in a form that neither
// overflows nor cancels; FAST uses the exp / log intrinsics (absolute error
// ~1e-7, far below the bf16 rounding of the states it feeds).
template <bool FAST> __device__ __forceinline__ float f_logsigmoid(float x) {
  if (FAST) return fminf(x, 0.0f) - __logf(1.0f + __expf(-fabsf(x)));
  return fminf(x, 0.0f) - log1pf(expf(-fabsf(x)));
}

// ---- forward --------------------------------------------------------------
// x[g]: Wx pre-activation; r[g]: recurrent branch (h.R + b); sp: previous
// states; sn: new states; pre: tape pre values.
template <int FN, bool FAST>
__device__ __forceinline__ void cell_fwd(const float* x, const float* r, const float* sp,
                                         float* sn, float* pre) {
  if constexpr (FN == LSTM) {
    float ai = x[0] + r[0], af = x[1] + r[1], ag = x[2] + r[2], ao = x[3] + r[3];
    float i = f_sigmoid<FAST>(ai), f = f_sigmoid<FAST>(af);
    float g = f_tanh<FAST>(ag), o = f_sigmoid<FAST>(ao);
    float c = fmaf(f, sp[1], i * g);
    sn[1] = c;
    sn[0] = o * f_tanh<FAST>(c);
    pre[0] = ai; pre[1] = af; pre[2] = ag; pre[3] = ao;
  } else if constexpr (FN == GRU) {
    float ar = x[0] + r[0], az = x[1] + r[1];
    float rg = f_sigmoid<FAST>(ar), z = f_sigmoid<FAST>(az);
    float n = f_tanh<FAST>(fmaf(rg, r[2], x[2]));
    sn[0] = fmaf(z, sp[0] - n, n);  // (1-z) n + z h
    pre[0] = ar; pre[1] = az; pre[2] = x[2]; pre[3] = r[2];
  } else if constexpr (FN == ELMAN) {
    float a = x[0] + r[0];
    sn[0] = f_tanh<FAST>(a);
    pre[0] = a;
  } else {  // SLSTM (log f = a_f) and SLSTM_LS (log f = log sigmoid(a_f))
    float ai = x[0] + r[0], af = x[1] + r[1], az = x[2] + r[2], ao = x[3] + r[3];
    float mp = sp[3];
    const float lf = FN == SLSTM_LS ? f_logsigmoid<FAST>(af) : af;
    float fm = lf + mp;
    float m = fm >= ai ? fm : ai;
    float ig = f_exp<FAST>(ai - m), fg = f_exp<FAST>(fm - m);
    float c = fmaf(fg, sp[1], ig * f_tanh<FAST>(az));
    float n = fmaf(fg, sp[2], ig);
    sn[1] = c; sn[2] = n; sn[3] = m;
    sn[0] = f_sigmoid<FAST>(ao) * c / n;
    pre[0] = ai; pre[1] = af; pre[2] = az; pre[3] = ao;
  }
}

// ---- backward -------------------------------------------------------------
// pre: tape pre values of the step; sp: states before it; sn: after it;
// dsn: total gradient reaching sn. Outputs dx (gradient of Wx), dr (gradient
// of the recurrent branch, what dR, db and dh_{t-1} through R see) and dsp
// (gradient of the previous states through the cell itself).
//
// The derivative comes in two parts: cell_bwd_act evaluates what does not
// depend on the incoming gradient (the gate activations, from the tape), and
// cell_bwd_grad finishes with dsn. A kernel can so evaluate the
// transcendentals while the gradient of h is still on its way.
constexpr int CELL_BWD_ACT = 8;
template <int FN, bool FAST>
__device__ __forceinline__ void cell_bwd_act(const float* pre, const float* sp, const float* sn, float* act) {
  if constexpr (FN == LSTM) {
    act[0] = f_sigmoid<FAST>(pre[0]);  // i
    act[1] = f_sigmoid<FAST>(pre[1]);  // f
    act[2] = f_tanh<FAST>(pre[2]);     // g
    act[3] = f_sigmoid<FAST>(pre[3]);  // o
    act[4] = f_tanh<FAST>(sn[1]);      // tanh(c)
  } else if constexpr (FN == GRU) {
    act[0] = f_sigmoid<FAST>(pre[0]);                     // r
    act[1] = f_sigmoid<FAST>(pre[1]);                     // z
    act[2] = f_tanh<FAST>(fmaf(act[0], pre[3], pre[2]));  // n
  } else if constexpr (FN == ELMAN) {
    act[0] = sn[0];
  } else {  // SLSTM and SLSTM_LS
    const float ai = pre[0], af = pre[1];
    const float lf = FN == SLSTM_LS ? f_logsigmoid<FAST>(af) : af;
    const float m = sn[3], mp = sp[3];
    act[0] = f_exp<FAST>(ai - m);                            // i'
    act[1] = f_exp<FAST>(lf + mp - m);                       // f'
    act[2] = f_tanh<FAST>(pre[2]);                           // z
    act[3] = f_sigmoid<FAST>(pre[3]);                        // o
    act[4] = 1.0f / sn[2];                                   // 1 / n
    act[5] = sn[1] * act[4];                                 // y = c / n
    act[6] = lf + mp >= ai ? 1.0f : 0.0f;                    // the max took the forget branch
    act[7] = FN == SLSTM_LS ? f_sigmoid<FAST>(-af) : 1.0f;  // d log f / d a_f
  }
}

template <int FN, bool FAST>
__device__ __forceinline__ void cell_bwd_grad(const float* act, const float* pre, const float* sp,
                                              const float* dsn, float* dx, float* dr, float* dsp) {
  if constexpr (FN == LSTM) {
    const float i = act[0], f = act[1], g = act[2], o = act[3], tc = act[4];
    float dh = dsn[0];
    float dc = fmaf(dh * o, 1.0f - tc * tc, dsn[1]);
    dx[0] = dc * g * i * (1.0f - i);
    dx[1] = dc * sp[1] * f * (1.0f - f);
    dx[2] = dc * i * (1.0f - g * g);
    dx[3] = dh * tc * o * (1.0f - o);
    dr[0] = dx[0]; dr[1] = dx[1]; dr[2] = dx[2]; dr[3] = dx[3];
    dsp[0] = 0.0f;
    dsp[1] = dc * f;
  } else if constexpr (FN == GRU) {
    const float rg = act[0], z = act[1], n = act[2];
    float q = pre[3];
    float dh = dsn[0];
    float dan = dh * (1.0f - z) * (1.0f - n * n);
    float drg = dan * q;
    dx[0] = drg * rg * (1.0f - rg);
    dx[1] = dh * (sp[0] - n) * z * (1.0f - z);
    dx[2] = dan;
    dr[0] = dx[0]; dr[1] = dx[1]; dr[2] = dan * rg;
    dsp[0] = dh * z;
  } else if constexpr (FN == ELMAN) {
    const float h = act[0];
    dx[0] = dsn[0] * (1.0f - h * h);
    dr[0] = dx[0];
    dsp[0] = 0.0f;
  } else {  // SLSTM and SLSTM_LS (gradients through log f, then d log f / d a_f)
    const float ig = act[0], fg = act[1], zt = act[2], o = act[3], rn = act[4], y = act[5];
    const float cp = sp[1], np = sp[2];
    float dh = dsn[0];
    float dy = dh * o;
    float dc = fmaf(dy, rn, dsn[1]);
    float dn = dsn[2] - dy * y * rn;
    float dfg = fmaf(dc, cp, dn * np);
    float dig = fmaf(dc, zt, dn);
    float dai = dig * ig;
    float dlf = dfg * fg;
    float dmp = dlf;
    float dm = dsn[3] - dai - dlf;
    if (act[6] != 0.0f) { dlf += dm; dmp += dm; } else { dai += dm; }
    const float daf = FN == SLSTM_LS ? dlf * act[7] : dlf;
    dx[0] = dai; dx[1] = daf;
    dx[2] = dc * ig * (1.0f - zt * zt);
    dx[3] = dh * y * o * (1.0f - o);
    dr[0] = dx[0]; dr[1] = dx[1]; dr[2] = dx[2]; dr[3] = dx[3];
    dsp[0] = 0.0f; dsp[1] = dc * fg; dsp[2] = dn * fg; dsp[3] = dmp;
  }
}

template <int FN, bool FAST>
__device__ __forceinline__ void cell_bwd(const float* pre, const float* sp, const float* sn,
                                         const float* dsn, float* dx, float* dr, float* dsp) {
  float act[CELL_BWD_ACT];
  cell_bwd_act<FN, FAST>(pre, sp, sn, act);
  cell_bwd_grad<FN, FAST>(act, pre, sp, dsn, dx, dr, dsp);
}

// ---- element access --------------------------------------------------------
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
// value as the storage type sees it (bf16 rounding for bf16 storage)
__device__ __forceinline__ float roundas(const float*, float v) { return v; }
__device__ __forceinline__ float roundas(const __nv_bfloat16*, float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Device status word: kernels record the first error here (bounded waits).
enum { STATUS_OK = 0, STATUS_TIMEOUT = 1 };

}  // namespace rnn
