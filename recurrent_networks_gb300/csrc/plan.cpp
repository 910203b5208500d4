// Kernel planner (see plan.h).
#include "plan.h"

#include <stdio.h>
#include <string.h>

#include "rnn.h"

namespace rnn {

static int gates_of(int fn) { return fn == 0 ? 4 : fn == 1 ? 3 : fn == 2 ? 1 : 4; }

static void simt_plan(const PlanRequest& q, Plan* p) {
  *p = Plan{};
  p->path = RNN_PATH_SIMT;
  p->Bc = q.B < 8 ? q.B : 8;
  p->groups = q.N * ((q.B + p->Bc - 1) / p->Bc);
}

int plan_select(const PlanRequest& q, Plan* out) {
  Plan p;
  switch (q.path) {
    case RNN_PATH_AUTO:
    case RNN_PATH_SIMT:
      simt_plan(q, &p);
      *out = p;
      return RNN_OK;
    default:
      snprintf(p.why, sizeof(p.why), "path %d not available for fn=%d D=%d", q.path, q.fn, q.D);
      (void)gates_of;
      *out = p;
      return RNN_EUNSUPPORTED;
  }
}

void plan_describe(const Plan& p, int rc, char* buf, size_t len) {
  if (rc != RNN_OK) {
    snprintf(buf, len, "unsupported: %s", p.why);
    return;
  }
  const char* names[] = {"auto", "fused", "alternating", "simt"};
  snprintf(buf, len,
           "path=%s C=%d U=%d Bc=%d NT=%d groups=%d MT=%d KT=%d ksplit=%d warps=%d regs_R=%d "
           "smem=%zu scratch=%zu model_ns=%.0f",
           names[p.path & 3], p.C, p.U, p.Bc, p.NT, p.groups, p.MT, p.KT, p.ksplit, p.warps,
           p.regs_R, p.smem, p.scratch_bytes, p.model_ns);
}

}  // namespace rnn
