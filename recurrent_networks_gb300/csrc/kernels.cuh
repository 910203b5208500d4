// Internal declarations shared by the kernel translation units and the C ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "cells.cuh"

namespace rnn {

// Counts kernel launches for rnn_kernel_launches(); every launcher calls it.
void note_launch(int count = 1);

// Arguments of the plain per-head kernels (and of the weight-gradient pass).
struct SimtArgs {
  int B, T, N, D, BB;
  const void* Wx;
  const void* R;
  const void* bias;
  const void* s0;
  void* states;
  void* last;
  float* tape;  // fwd: out (may be null); bwd: in
  const void* dstates;
  const void* dlast;
  void* dWx;
  void* dr;  // bwd: recurrent-branch gradients [B,T,G,N,D] (storage type)
  void* ds0;
};

int simt_supported(int fn, int B, int D, bool bwd);
cudaError_t simt_run(int fn, int dtype, const SimtArgs& a, bool bwd, cudaStream_t st);

// dR[g,n,i,j] = sum_{b,t} hprev[b,t,n,i] dr[b,t,g,n,j];  db[g,n,j] = sum_{b,t} dr[b,t,g,n,j]
// with hprev[b,t] = states[0,b,t-1] (t > 0) or states0[0,b,0] (t = 0, zeros if null).
struct WgradArgs {
  int B, T, N, D, G;
  const void* states;
  const void* s0;
  const void* dr;
  void* dR;  // may be null
  void* db;  // may be null
};
cudaError_t wgrad_run(int dtype, const WgradArgs& a, cudaStream_t st);

}  // namespace rnn
