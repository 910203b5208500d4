// Shared-memory layouts of the persistent cluster kernels, used by the
// kernels and by the host planner (plain C++: no CUDA dependency).
#pragma once
#include <stddef.h>

#if defined(__CUDACC__)
#define RNN_HD __host__ __device__
#else
#define RNN_HD
#endif

namespace rnn {

constexpr int FUSED_NS = 4;           // Wx ring depth (steps in flight)
constexpr int FUSED_RED_STRIDE = 20;  // floats per batch row of a partial-sum tile (16 used)
constexpr int FUSED_MAX_KS = 8;       // K-split warps per 16-unit group (warps <= 8)
constexpr int FUSED_MAX_C = 16;       // CTAs per cluster
constexpr int FUSED_PPT = 2;          // (batch row, unit) pairs a thread carries in registers

// Launch shape of a persistent cluster kernel, chosen by the planner.
struct FusedShape {
  int C = 1;      // CTAs per cluster (one cluster per head and batch group)
  int U = 0;      // units owned by one CTA (D / C)
  int NT = 0;     // n-tiles of 8 batch rows (BC = 8 NT rows per cluster)
  int KT = 0;     // k-tiles of 16 per warp
  int KS = 0;     // warps splitting K for one 16-row group
  int MT = 0;     // backward: m-tiles (16 rows of dh) per warp
  bool allg = false;  // forward: a warp holds all G gate tiles (else one gate)
  int warps = 0;  // warps per CTA
  size_t smem = 0;
};

// Forward cluster kernel: per CTA, G gates x U units, BC batch rows, K split in KS.
struct FusedSmem {
  size_t bars, wx, hbuf, red, stage, cst, bias, total;
  RNN_HD static size_t take(size_t& off, size_t bytes) {
    size_t o = off;
    off = (off + bytes + 127) & ~(size_t)127;
    return o;
  }
  RNN_HD static FusedSmem make(int G, int S, int D, int U, int BC, int KS) {
    FusedSmem m;
    size_t off = 0;
    // h_{t-1} is kept per source CTA: hbuf[2][C][BC][U + 8] (bf16, rows padded
    // by 16 bytes so that ldmatrix rows fall on distinct banks); the CTA's own
    // slice of h_t is staged in the same row format, double-buffered.
    const int C = D / U, UP = U + 8;
    m.bars = take(off, 8 * (3 + FUSED_NS));  // h full x2, Wx ring, one never signalled
    m.wx = take(off, (size_t)FUSED_NS * BC * G * U * 2);
    m.hbuf = take(off, (size_t)2 * C * BC * UP * 2);
    m.red = take(off, (size_t)(U / 16) * KS * G * BC * FUSED_RED_STRIDE * 4);
    m.stage = take(off, (size_t)2 * BC * UP * 2);
    m.cst = m.bias = off;  // carried states and biases are held in registers
    (void)S;
    m.total = off;
    return m;
  }
};

// Backward cluster kernel: per CTA, the U units it owns; the reverse scan
// streams tape[t] ([BC][K][U] fp32) and dstates[:, t] ([S][BC][U] bf16) through
// a TMA ring, receives C fp32 partial sums of dh for its units per step
// ([C][U][BC]), and feeds its own recurrent-branch gradients ([BC][G U + 8]
// bf16) to the tensor cores.
constexpr int FUSED_BWD_MAX_KTA = 8;  // k-tiles G*U/16 a CTA may own

struct FusedBwdSmem {
  size_t bars, ring, ring_stage, tape_bytes, dst_off, recv, drb, ds, s0, dbs, total;
  RNN_HD static FusedBwdSmem make(int G, int S, int K, int U, int BC, int C) {
    FusedBwdSmem m;
    size_t off = 0;
    m.bars = FusedSmem::take(off, 8 * (2 + FUSED_NS));
    m.tape_bytes = (size_t)BC * K * U * 4;
    m.dst_off = (m.tape_bytes + 127) & ~(size_t)127;
    m.ring_stage = (m.dst_off + (size_t)S * BC * U * 2 + 127) & ~(size_t)127;
    m.ring = FusedSmem::take(off, FUSED_NS * m.ring_stage);
    m.recv = FusedSmem::take(off, (size_t)2 * C * U * BC * 4);
    m.drb = FusedSmem::take(off, (size_t)2 * BC * (G * U + 8) * 2);
    m.ds = off;  // the carried gradients are held in registers
    m.s0 = FusedSmem::take(off, (size_t)S * BC * U * 4);
    m.dbs = FusedSmem::take(off, (size_t)G * BC * U * 4);  // db sums of the CTA's pairs
    m.total = off;
    return m;
  }
};

// Backward grid kernel: the TMA ring of the cluster backward, the gathered
// recurrent-branch gradients of the whole group ([BC][G D + 8] bf16), the
// K-split partial sums, and the carried and initial states.
struct GridBwdSmem {
  size_t bars, ring, ring_stage, tape_bytes, dst_off, dbuf, red, ds, s0, dbs, total;
  RNN_HD static GridBwdSmem make(int G, int S, int K, int D, int U, int BC, int KS) {
    GridBwdSmem m;
    size_t off = 0;
    m.bars = FusedSmem::take(off, 8 * (FUSED_NS + 1));  // the TMA ring, then the gather
    m.tape_bytes = (size_t)BC * K * U * 4;
    m.dst_off = (m.tape_bytes + 127) & ~(size_t)127;
    m.ring_stage = (m.dst_off + (size_t)S * BC * U * 2 + 127) & ~(size_t)127;
    m.ring = FusedSmem::take(off, FUSED_NS * m.ring_stage);
    m.dbuf = FusedSmem::take(off, (size_t)BC * (G * D + 8) * 2);
    m.red = FusedSmem::take(off, (size_t)(U / 16) * KS * BC * FUSED_RED_STRIDE * 4);
    m.ds = FusedSmem::take(off, (size_t)S * BC * U * 4);
    m.s0 = FusedSmem::take(off, (size_t)S * BC * U * 4);
    m.dbs = FusedSmem::take(off, (size_t)G * BC * U * 4);  // db sums of the CTA's pairs
    m.total = off;
    return m;
  }
};

}  // namespace rnn
