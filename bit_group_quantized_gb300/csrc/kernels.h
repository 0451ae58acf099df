// kernels.h — internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

struct bgq_moe_layer;

namespace bgq {

struct QMat {
  const uint32_t* q;
  const uint16_t* sb;
  int rows, cols, bits;
};

// Device-resolvable reference to one SwiGLU expert.
struct ExpertRef {
  const uint32_t* gate_q;
  const uint16_t* gate_sb;
  const uint32_t* up_q;
  const uint16_t* up_sb;
  const uint32_t* down_q;
  const uint16_t* down_sb;
};

// The experts a plan can name: pool expert e >= 0, or `shared` for e == -1.
struct ExpertSet {
  const uint32_t* pool_q;
  const uint16_t* pool_sb;
  long long q_stride;   // words between experts
  long long sb_stride;  // bf16 elements between experts
  ExpertRef shared;
  int d, f, bits;
};

constexpr int kTaskTok = 8;  // tokens per task (grouped GEMV width)
constexpr int kBigTok = 16;  // smallest tensor-core task (an explicit expert; a layer call uses 32, api.cu)

// One grouped-GEMV task: expert `expert` applied to up to 8 tokens; token i's
// result goes to slot slot[i] of token tok[i].
struct Task {
  int expert;
  int ntok;
  int tok[kTaskTok];
  int slot[kTaskTok];
};

// One tensor-core task: expert `expert` (-1: shared) applied to ntok tokens,
// listed at ptok[first..first+ntok) with their slots at pslot[...]; its
// activations are staged at rows [pad, pad + ntok rounded up to 16).
struct BigTask {
  int expert;
  int ntok;
  int first;
  int pad;
};

// Plan header; followed by Task[max_tasks], BigTask[max_big], int ptok[max_pairs], int pslot[max_pairs].
struct Plan {
  int ntasks;  // grouped-GEMV tasks
  int nbig;    // tensor-core tasks
  int pad[2];
};

__host__ __device__ inline int plan_max_tasks(int B, int K) { return B * K + (B + kTaskTok - 1) / kTaskTok + 1; }
__host__ __device__ inline int plan_max_big(int B, int K) { return (B * K) / kBigTok + 2; }
__host__ __device__ inline int plan_max_pairs(int B, int K) { return B * K + B; }
__host__ __device__ inline Task* plan_tasks(Plan* p) { return reinterpret_cast<Task*>(p + 1); }
__host__ __device__ inline const Task* plan_tasks(const Plan* p) { return reinterpret_cast<const Task*>(p + 1); }
__host__ __device__ inline BigTask* plan_big(Plan* p, int B, int K) {
  return reinterpret_cast<BigTask*>(plan_tasks(p) + plan_max_tasks(B, K));
}
__host__ __device__ inline const BigTask* plan_big(const Plan* p, int B, int K) {
  return reinterpret_cast<const BigTask*>(plan_tasks(p) + plan_max_tasks(B, K));
}
__host__ __device__ inline int* plan_ptok(Plan* p, int B, int K) {
  return reinterpret_cast<int*>(plan_big(p, B, K) + plan_max_big(B, K));
}
__host__ __device__ inline const int* plan_ptok(const Plan* p, int B, int K) {
  return reinterpret_cast<const int*>(plan_big(p, B, K) + plan_max_big(B, K));
}
__host__ __device__ inline int* plan_pslot(Plan* p, int B, int K) { return plan_ptok(p, B, K) + plan_max_pairs(B, K); }
__host__ __device__ inline const int* plan_pslot(const Plan* p, int B, int K) {
  return plan_ptok(p, B, K) + plan_max_pairs(B, K);
}

inline size_t plan_bytes(int batch, int top_k) {
  return sizeof(Plan) + (size_t)plan_max_tasks(batch, top_k) * sizeof(Task) +
         (size_t)plan_max_big(batch, top_k) * sizeof(BigTask) + (size_t)plan_max_pairs(batch, top_k) * 8;
}

// Workspace control block (first 256 bytes of every workspace).
struct Ctrl {
  int status;         // 0 = ok, 4 = a bounded wait timed out
  int pad0[15];
  int route_counter;  // last-CTA detection of the router kernel
  int pad1[15];
  int misc[32];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

size_t qgemv_int_smem(int cols, int bits, int T);
// res (nullable, variant 0): bf16 [batch][rows] added to each fp32 row sum
// before the outputs are written.
cudaError_t launch_qgemv(const QMat& W, const uint16_t* x, int batch, uint16_t* y, float* yf, int variant,
                         cudaStream_t s, const uint16_t* res = nullptr);

// Bytes at the start of a layer workspace that must be zero before a call:
// control block and tagged logits (api.cu).
size_t layer_zero_prefix_bytes(const bgq_moe_layer* L);
// moe_layer_forward's argument checks, split around its workspace check
// (api.cu): BGQ_OK or the status moe_layer_forward returns for the same
// arguments. layer_call_check comes first, layer_location_check (weights in
// device or mapped pinned host memory) after the workspace's.
int layer_call_check(const bgq_moe_layer* L, const uint16_t* x, int batch, const void* out, const void* out_f32);
int layer_location_check(const bgq_moe_layer* L);

// 8-bit GEMV (gemv8.cu). gpr = (scale, bias) pairs per row: cols/64 or 1 (per
// row). q8gemv_max_tokens: inputs staged per launch for `cols` (0: too wide).
int q8gemv_max_tokens(int cols);
cudaError_t launch_q8gemv(const QMat& W, int gpr, const uint16_t* x, int batch, uint16_t* y, cudaStream_t s);

// Router + softmax + top-K (+ optional grouping plan). Experts with at least
// big_min tokens become tensor-core tasks (kBigTok; INT_MAX: none).
cudaError_t launch_route(const uint16_t* router, const uint16_t* sgate, const uint16_t* x, int batch, int d,
                         int E, int K, float* logits_ws, Ctrl* ctrl, int32_t* idx, float* w, float* gamma,
                         float* logits_out, Plan* plan, int big_min, cudaStream_t s);

// Builds the plan of one explicit expert over `batch` tokens (slot 0).
cudaError_t launch_plan_single(Plan* plan, int batch, int big_min, cudaStream_t s);

// Tensor-core (tcgen05) gate/up + SiLU*mul and down projection for the plan's
// big tasks (experts with >= kBigTok tokens). B, K: the plan's batch and top_k.
// `act` holds the staged fp16 activations and their per-row scales
// (tc_act_bytes for a plan of (B, K); written before read). K is split over
// the CTAs of a cluster, whose partial sums meet in distributed shared
// memory: no other scratch, nothing left behind between calls.
// plan == nullptr: one task of all B tokens of the shared-expert view (token
// n in slot 0; K = 0, nslot = 1). Only then may the down call write bf16 `y`
// and/or fp32 `y_f32` rows (token-major, d columns) directly instead of Y:
// the same bits as the combine of that one slot with weight 1.
size_t tc_act_bytes(int d, int f, int B, int K);
// Whether the pools of `es` can feed the tensor-core path (tensor-map
// alignment of the codes and scale/bias rows); host-side check.
bool tc_layer_ok(const ExpertSet& es);
cudaError_t launch_gateup_tc(const ExpertSet& es, const Plan* plan, int B, int K, const uint16_t* x, float* H,
                             int nslot, Ctrl* ctrl, unsigned char* act, cudaStream_t s);
cudaError_t launch_down_tc(const ExpertSet& es, const Plan* plan, int B, int K, const float* H, float* Y, int nslot,
                           Ctrl* ctrl, unsigned char* act, uint16_t* y, float* y_f32, cudaStream_t s);

// plan == nullptr (launch_gateup / launch_down): one explicit expert over all
// `batch` tokens (tasks of 8 consecutive tokens of the shared-expert view,
// slot 0, nslot 1), built by the kernels themselves; allowed when
// grouped_planless_ok() holds (at most kPlanlessTasks tasks and shapes the
// one-CTA-per-SM kernels take).
constexpr int kPlanlessTasks = 32;
bool grouped_planless_ok(const ExpertSet& es, int batch, bool stage_ws);
// Grouped gate/up + SiLU*mul: H[(tok*nslot + slot)*f + row].
// batch: tokens of x, staged all at once in shared memory when they fit, else
// into stage_ws (staged_tokens_bytes(d, bits, batch) bytes of global memory;
// null: the per-task kernels instead).
cudaError_t launch_gateup(const ExpertSet& es, const Plan* plan, int max_tasks, int batch, const uint16_t* x, float* H,
                          int nslot, unsigned char* stage_ws, cudaStream_t s);
// Weighted combine of the K + 1 slots per token (launch_combine's formula),
// done by launch_down when out or out_f32 is set. w: [batch][K] (K may be 0),
// gamma nullable (1).
struct Combine {
  const float* w;
  const float* gamma;
  int K;
  uint16_t* out;
  float* out_f32;
};
// Grouped down projection: Y[(tok*nslot + slot)*d + row]; H holds batch*nslot
// vectors of f (stage_ws: staged_tokens_bytes(f, bits, batch*nslot) bytes).
// Every tensor-core task's Y must be written before (the combine reads them).
cudaError_t launch_down(const ExpertSet& es, const Plan* plan, int max_tasks, int batch, const float* H, float* Y,
                        int nslot, unsigned char* stage_ws, const Combine& cb, cudaStream_t s);
size_t staged_tokens_bytes(int cols, int bits, int T);
// out[t][r] = sum_{k<K} w[t][k] Y[t][k][r] + gamma[t] Y[t][K][r]  (K may be 0; gamma NULL => 1).
cudaError_t launch_combine(const float* Y, const float* w, const float* gamma, int batch, int K, int d,
                           uint16_t* out, float* out_f32, cudaStream_t s);

cudaError_t launch_rmsnorm(const float* h, const uint16_t* rho, int batch, int d, float eps, uint16_t* a,
                           cudaStream_t s);
cudaError_t launch_rmsnorm_bf16(const uint16_t* x, const uint16_t* rho, int batch, int d, float eps, uint16_t* a,
                                cudaStream_t s);
cudaError_t launch_residual_add(float* h, const float* delta, long long n, cudaStream_t s);
cudaError_t launch_widen(const uint16_t* x, float* h, int n, cudaStream_t s);

// Experts copied per layer into HBM slots (stream.cu). Slot buffer layout:
// header (int count, then the expert of each slot), the slots' codes, then
// their scale/bias rows, every region 256-byte aligned.
struct SlotGeo {
  int max_slots;
  long long q_bytes, sb_bytes;  // one expert's codes / scale-bias bytes (gate, up, down)
  long long slot_q, slot_sb;    // slot strides (bytes)
  long long hdr, total;         // header bytes, whole buffer bytes
};
SlotGeo slot_geo(int d, int f, int bits, int max_slots);
// Turn the plan's experts into slot numbers and copy the selected experts of
// `pool` into the slots (two kernels on s).
cudaError_t launch_slot_copy(Plan* plan, int E, const ExpertSet& pool, const SlotGeo& g, void* slots, cudaStream_t s);
// The slots as an expert set (shared expert as in `pool`).
ExpertSet slot_expert_set(const ExpertSet& pool, const SlotGeo& g, void* slots);

int num_sms();

// Longest projection chain of bgq_gemv_chain.
constexpr int kMaxChain = 8;

}  // namespace bgq
