// Kernel planner: an integer constraint solver over the tile and cluster
// parameters of the persistent kernels -- the role the FlashRNN announcement
// gives its ConstrINT tuner (hardware limits written as equalities,
// inequalities and divisibility constraints). Host code only.
#pragma once
#include <stddef.h>

#include "layout.h"

namespace rnn {

// The grid kernels' counter region in the workspace: 16 blocks of 1 KB (under
// die placement a group's counter sits at the start of a block whose L2 home
// is on the group's die), then one line of die tickets; 1 KB of alignment
// slack in front.
constexpr int GRID_CTR_BLOCKS = 16;
constexpr size_t GRID_CTR_BYTES = (size_t)(GRID_CTR_BLOCKS + 1) * 1024 + 256;
// Chunks of steps whose dR the grid backward's spare CTAs compute beside the scan.
constexpr int DR_BESIDE_CHUNKS = 5;

// Limits of the GPU that the constraints use. The defaults are a GB300's
// (152 SMs, 227 KB of opt-in shared memory per CTA, clusters of up to 16 CTAs
// with the non-portable size); the library fills them from the current device.
struct DeviceLimits {
  int sms = 152;
  int max_cluster = 16;       // non-portable cluster size limit
  size_t smem_per_cta = 227 * 1024;
  int regs_per_thread = 255;  // launch bounds: 256 threads, 1 CTA per SM
  int max_warps = 8;
  // Clusters of the cluster kernel for (fn, backward, shape) that the device
  // can hold at once (cudaOccupancyMaxActiveClusters), or -1 when unknown (no
  // device to ask). 0 makes the candidate infeasible; a positive count sets the
  // number of waves the model charges. nullptr: not asked.
  int (*cluster_capacity)(int fn, bool bwd, const FusedShape& fs) = nullptr;
};

struct PlanRequest {
  int B, T, N, D, fn, dtype, path;
  bool bwd;
  const DeviceLimits* lim = nullptr;  // nullptr: the GB300 defaults above
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
bool fused_bwd_feasible(const PlanRequest& q, int C, int NT, int MT, const DeviceLimits& lim, Plan* out);
bool grid_feasible(const PlanRequest& q, int C, int NT, int KT, const DeviceLimits& lim, Plan* out);

// Alternating path (csrc/alt.cu): whether the unit tiles divide D, and the
// workspace its ping-pong and carried-state buffers take.
int alt_supported(int fn, int D);
size_t alt_scratch_bytes(int fn, int B, int N, int D, bool bwd);

int plan_select(const PlanRequest& q, Plan* out);  // RNN_OK or RNN_EUNSUPPORTED
void plan_describe(const Plan& p, int rc, char* buf, size_t len);

}  // namespace rnn
