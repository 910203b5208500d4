// Kernel planner: an integer constraint solver over the tile and cluster
// parameters of the fused and grid kernels (the role the FlashRNN announcement
// gives its ConstrINT tuner: hardware limits written as equalities,
// inequalities and divisibility constraints). Host code only.
#pragma once
#include <stddef.h>

namespace rnn {

struct PlanRequest {
  int B, T, N, D, fn, dtype, path;
  bool bwd;
};

// Limits of one GB300 SM / GPU that the constraints use.
struct DeviceLimits {
  int sms = 152;
  int max_cluster = 16;          // non-portable cluster size limit
  int portable_cluster = 8;
  size_t smem_per_cta = 227 * 1024;
  int regs_per_sm = 65536;
  int max_regs_per_thread = 255;
  int max_threads = 1024;
};

struct Plan {
  int path = 0;         // rnn_path_t
  // fused (cluster) and grid kernels
  int C = 1;            // CTAs cooperating on one head (cluster size, or grid CTAs per head)
  int U = 0;            // units of D owned by one CTA (D / C)
  int Bc = 0;           // batch rows per CTA group (padded to the MMA N tile inside)
  int NT = 0;           // n-tiles of 8 batch rows
  int groups = 0;       // independent CTA groups: heads x batch splits
  int MT = 0;           // m-tiles (16 rows) per warp
  int KT = 0;           // k-tiles (16) per warp
  int ksplit = 0;       // warps sharing one m-tile set along K
  int warps = 0;
  int regs_R = 0;       // registers per thread holding the resident R fragments
  size_t smem = 0;      // dynamic shared memory per CTA
  size_t scratch_bytes = 0;  // workspace the path needs beyond the status word
  double model_ns = 0;  // modelled latency of one step
  char why[200] = {0};  // reason when no plan fits
};

int plan_select(const PlanRequest& q, Plan* out);  // RNN_OK or RNN_EUNSUPPORTED
void plan_describe(const Plan& p, int rc, char* buf, size_t len);

}  // namespace rnn
