// Kernel planner: an integer constraint solver over the tile and cluster
// parameters of the persistent kernels -- the role the FlashRNN announcement
// gives its ConstrINT tuner (hardware limits written as equalities,
// inequalities and divisibility constraints). Host code only.
#pragma once
#include <stddef.h>

#include "layout.h"

namespace rnn {

struct PlanRequest {
  int B, T, N, D, fn, dtype, path;
  bool bwd;
};

// Limits of one GB300 SM / GPU that the constraints use.
struct DeviceLimits {
  int sms = 152;
  int max_cluster = 16;       // non-portable cluster size limit
  size_t smem_per_cta = 227 * 1024;
  int regs_per_thread = 255;  // launch bounds: 256 threads, 1 CTA per SM
  int max_warps = 8;
};

struct Plan {
  int path = 0;         // rnn_path_t actually used
  FusedShape fs;        // cluster kernels
  int groups = 0;       // independent CTA groups: heads x batch groups
  int regs_R = 0;       // registers per thread holding resident R fragments
  size_t scratch_bytes = 0;  // workspace the path needs beyond the status word
  double model_ns = 0;  // modelled latency of one step
  int candidates = 0;   // feasible points the solver compared
  char why[200] = {0};  // reason when no plan fits
};

// The constraint check for one candidate point of the forward cluster kernel
// (exposed for tests): returns true and fills *out when every constraint holds.
bool fused_fwd_feasible(const PlanRequest& q, int C, int NT, int KT, bool allg, const DeviceLimits& lim,
                        Plan* out);

// Alternating path (csrc/alt.cu): whether the unit tiles divide D, and the
// workspace its ping-pong and carried-state buffers take.
int alt_supported(int fn, int D);
size_t alt_scratch_bytes(int fn, int B, int N, int D, bool bwd);

int plan_select(const PlanRequest& q, Plan* out);  // RNN_OK or RNN_EUNSUPPORTED
void plan_describe(const Plan& p, int rc, char* buf, size_t len);

}  // namespace rnn
