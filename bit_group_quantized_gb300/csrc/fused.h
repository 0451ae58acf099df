// fused.h — parameters of the persistent batch-1 decode kernel (fused.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace bgq {

constexpr int kMaxFusedLayers = 128;

struct FusedLayer {
  const uint16_t* router;  // bf16 [E][d]
  const uint16_t* sgate;   // bf16 [d] or null
  const uint32_t* pool_q;
  const uint16_t* pool_sb;
  long long q_stride, sb_stride;
  const uint32_t* shared_q;
  const uint16_t* shared_sb;
  const uint16_t* rho;  // bf16 [d] (stack mode)
};

// Geometry of one launch, computed on the host (fused.cu, fused_geo): the
// work split of every phase and the shared-memory layout.
struct FGeo {
  int nC;              // CTAs (one per SM)
  int qr, rpc;         // warps per router row (1024 columns each), router rows per CTA
  int nRouter;         // CTAs holding router rows
  int nit_d, wpr, gpr; // rows of d (router, gate, up): parts per lane, code words, groups
  int unit;            // shared-memory bytes of one gate+up unit (two rows, their scale/bias)
  int nBmax;           // selected gate/up units per CTA (at most)
  int s1_nr;           // shared gate/up units per CTA without router rows
  int s1_rest0, s1_nparts;  // the other CTAs' split of the remaining shared units
  int rows_c;          // output rows per CTA (at most)
  int wqf, wsf;        // bytes of one down row's codes / scale-bias pairs
  int a_bytes;         // region A: phase-A data (router rows + shared units)
  int b_bytes;         // region B: selected gate/up units, then phase C's down rows and staged inputs
  // shared-memory byte offsets
  int o_misc, o_as, o_sta, o_hres, o_a, o_b, total;
};

struct FusedParams {
  FGeo g;  // filled by launch_fused
  int n_layers, d, f, E, K;
  int stack;  // 1: RMSNorm + residual per layer, x_next output; 0: one layer, out = layer(x)
  float eps;
  long long timeout_ns;
  const uint16_t* x_in;  // bf16 [d]
  // outputs (nullable)
  uint16_t* x_next;    // stack: bf16 [d]
  float* h_out;        // stack: fp32 [d]
  uint16_t* out;       // layer: bf16 [d]
  float* out_f32;      // layer: fp32 [d]
  int32_t* idx_out;    // [n_layers][K]
  float* w_out;        // [n_layers][K]
  float* gamma_out;    // [n_layers]
  // scratch (workspace)
  Ctrl* ctrl;
  float* h;          // [d] residual stream
  float* hk;         // [K+1][f] SwiGLU outputs (slot K: shared expert)
  float* logits;     // [E+1]
  unsigned long long* ltag;  // [E+1] logits as {value bits, tag} words (tag: launch epoch and layer)
  float* part_ss;    // [2][nCTA] per-CTA sums of h^2
  int32_t* route_idx;  // [K]
  float* route_w;      // [K+1] (K: gamma)
  // optional phase timestamps (%globaltimer, ns): [n_layers][nCTA][kTraceEvents]
  unsigned long long* trace;
  FusedLayer layers[kMaxFusedLayers];
};

constexpr int kTraceEvents = 16;

size_t fused_smem_bytes(int d, int f, int K, int bits);
bool fused_supported(int d, int f, int E, int K, int bits);
cudaError_t launch_fused(const FusedParams& P, int bits, cudaStream_t s);
cudaError_t launch_wait_selftest(Ctrl* ctrl, long long timeout_ns, cudaStream_t s);

}  // namespace bgq
