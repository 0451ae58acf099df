// api.cu — the C ABI of libbgq.so (declared in include/bgq.h).
//
// Every entry point validates its arguments before it enqueues anything,
// carves the caller's workspace into the regions its kernels need, and
// launches on the caller's stream. Nothing here allocates or synchronises.
#include <climits>
#include <stdint.h>
#include <string.h>

#include "../../include/bgq.h"
#include "common.cuh"
#include "fused.h"
#include "kernels.h"

namespace bgq {
bool route_shape_ok(int d);
}

using namespace bgq;

namespace {

constexpr int kMaxBatch = 256;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 8;
constexpr int kMaxLayers = 128;

inline bool al(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline cudaStream_t st(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

int check_qmatrix(const bgq_qmatrix* W) {
  if (!W || !W->q || !W->sb) return BGQ_ERR_INVALID_ARG;
  if (W->bits != 4 && W->bits != 2) return BGQ_ERR_INVALID_ARG;
  if (W->group != kGroup) return BGQ_ERR_UNSUPPORTED;
  if (W->rows <= 0 || W->cols <= 0 || W->cols % kGroup) return BGQ_ERR_INVALID_ARG;
  if (!cols_supported(W->cols, W->bits)) return BGQ_ERR_UNSUPPORTED;
  if (!al(W->q, 16) || !al(W->sb, 4)) return BGQ_ERR_INVALID_ARG;
  return BGQ_OK;
}

QMat qm(const bgq_qmatrix* W) { return QMat{W->q, W->sb, W->rows, W->cols, W->bits}; }

// Sequential carving of a 256-byte aligned workspace.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t bytes) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += up256(bytes);
    return p;
  }
};

// A layer call sends an expert to the tensor cores from kLayerTcMinTokens
// tokens: below that the grouped GEMVs finish the whole layer sooner (d_model
// 4096, d_ff 1024, top-4: even at batch 32, GEMVs ahead at 16, tensor cores
// ahead from 64). An explicit expert call uses them from kBigTok, where they
// are ahead at every batch.
constexpr int kLayerTcMinTokens = 32;

struct LayerWs {
  Ctrl* ctrl;
  float* logits;  // [B][E+1] then B*K ints of selected experts
  Plan* plan;
  int32_t* idx;
  float* w;
  float* gamma;
  float* H;  // [B][K+1][f]
  float* Y;  // [B][K+1][d]
  unsigned char* stage;  // inputs staged in global memory when too many for shared memory
  // batch-1 persistent kernel scratch
  float* fh;        // [d] residual stream
  float* fpart;     // [2][1024] per-CTA sums of squares
  int32_t* fidx;    // [16]
  float* fw;        // [16]
  unsigned char* tca;  // staged activations of the tensor-core kernels (batches that can use them)
  unsigned long long* ftag;  // batch-1 persistent kernel: tagged logits [E+1]
  size_t zero_bytes;  // leading bytes that must be zero when a call starts (ctrl, ftag)
  size_t bytes;
};

LayerWs carve_layer(void* ws, int B, int d, int f, int E, int K) {
  Carver c(ws);
  LayerWs L;
  L.ctrl = c.take<Ctrl>(sizeof(Ctrl));
  // the persistent kernel's tagged logits right after the control block: zero
  // between calls like it (layer_zero_prefix_bytes covers both)
  L.ftag = c.take<unsigned long long>((size_t)(E + 1) * 8);
  L.zero_bytes = c.off;  // everything above is left at zero by the kernels; the rest is written before read
  L.logits = c.take<float>((size_t)B * (E + 1) * 4 + (size_t)B * K * 4);
  L.plan = c.take<Plan>(plan_bytes(B, K));
  L.idx = c.take<int32_t>((size_t)B * K * 4);
  L.w = c.take<float>((size_t)B * K * 4);
  L.gamma = c.take<float>((size_t)B * 4);
  L.H = c.take<float>((size_t)B * (K + 1) * f * 4);
  L.Y = c.take<float>((size_t)B * (K + 1) * d * 4);
  {
    const size_t sx = staged_tokens_bytes(d, 4, B), sh = staged_tokens_bytes(f, 4, B * (K + 1));
    L.stage = c.take<unsigned char>(sx > sh ? sx : sh);  // 4-bit staging is the larger
  }
  L.fh = c.take<float>((size_t)d * 4);
  L.fpart = c.take<float>(2 * 1024 * 4);
  L.fidx = c.take<int32_t>(16 * 4);
  L.fw = c.take<float>(16 * 4);
  L.tca = B >= kLayerTcMinTokens ? c.take<unsigned char>(tc_act_bytes(d, f, B, K)) : nullptr;
  L.bytes = c.off;
  return L;
}

int check_layer(const bgq_moe_layer* L) {
  if (!L || !L->router || !L->expert_q || !L->expert_sb || !L->shared_q || !L->shared_sb) return BGQ_ERR_INVALID_ARG;
  if (L->bits != 4 && L->bits != 2) return BGQ_ERR_INVALID_ARG;
  if (L->group != kGroup) return BGQ_ERR_UNSUPPORTED;
  if (L->d_model <= 0 || L->d_ff <= 0 || L->n_experts <= 0 || L->top_k <= 0) return BGQ_ERR_INVALID_ARG;
  if (L->top_k > kMaxTopK || L->n_experts > kMaxExperts || L->top_k > L->n_experts) return BGQ_ERR_UNSUPPORTED;
  if (!cols_supported(L->d_model, L->bits) || !cols_supported(L->d_ff, L->bits)) return BGQ_ERR_UNSUPPORTED;
  if (!route_shape_ok(L->d_model)) return BGQ_ERR_UNSUPPORTED;
  const long long mw = (long long)L->d_model * L->d_ff * L->bits / 32;
  const long long mg = (long long)L->d_model * L->d_ff / kGroup * 2;
  if (L->expert_q_stride < 3 * mw || L->expert_sb_stride < 3 * mg) return BGQ_ERR_INVALID_ARG;
  if (L->expert_q_stride % 4 || L->expert_sb_stride % 2) return BGQ_ERR_INVALID_ARG;
  if (!al(L->router, 16) || !al(L->expert_q, 16) || !al(L->shared_q, 16) || !al(L->expert_sb, 4) ||
      !al(L->shared_sb, 4) || (L->shared_gate && !al(L->shared_gate, 16)))
    return BGQ_ERR_INVALID_ARG;
  return BGQ_OK;
}

ExpertSet expert_set(const bgq_moe_layer* L) {
  ExpertSet es;
  es.pool_q = L->expert_q;
  es.pool_sb = L->expert_sb;
  es.q_stride = L->expert_q_stride;
  es.sb_stride = L->expert_sb_stride;
  const long long mw = (long long)L->d_model * L->d_ff * L->bits / 32;
  const long long mg = (long long)L->d_model * L->d_ff / kGroup * 2;
  es.shared = ExpertRef{L->shared_q, L->shared_sb, L->shared_q + mw, L->shared_sb + mg, L->shared_q + 2 * mw,
                        L->shared_sb + 2 * mg};
  es.d = L->d_model;
  es.f = L->d_ff;
  es.bits = L->bits;
  return es;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? BGQ_OK : BGQ_ERR_CUDA; }

// Where weights live. Device memory is read by every kernel; pinned host
// memory mapped into the device address space (Grace memory over the CPU-GPU
// link) is read by the kernels that use plain loads only: the router, the
// grouped GEMVs and the combine, never the bulk copies of the persistent
// kernel or the tensor-core path.
enum class Where { kDevice, kHost, kBad };
Where where_is(const void* p) {
  if (!p) return Where::kDevice;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return Where::kBad;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return Where::kDevice;
  if (a.type == cudaMemoryTypeHost && a.devicePointer == p) return Where::kHost;
  return Where::kBad;
}
Where layer_where(const bgq_moe_layer* L) {
  const void* ps[] = {L->router, L->shared_gate, L->expert_q, L->expert_sb, L->shared_q, L->shared_sb};
  Where w = Where::kDevice;
  for (const void* p : ps) {
    const Where k = where_is(p);
    if (k == Where::kBad) return Where::kBad;
    if (k == Where::kHost) w = Where::kHost;
  }
  return w;
}
// Tokens an expert needs in a layer call before it runs on tensor cores
// (never for host-resident pools, nor for pools whose rows the tensor maps
// cannot address).
int big_min_for(Where w, const ExpertSet& es) {
  return w == Where::kHost || !tc_layer_ok(es) ? INT_MAX : kLayerTcMinTokens;
}

constexpr long long kFusedTimeoutNs = 2000000000ll;  // bounded waits inside the persistent kernel

// The persistent kernel streams weight rows with 16-byte bulk copies.
bool use_fused(const bgq_moe_layer* L) {
  if (!al(L->router, 16) || !al(L->expert_sb, 16) || !al(L->shared_sb, 16)) return false;
  if (L->shared_gate && !al(L->shared_gate, 16)) return false;
  if (L->expert_sb_stride % 8) return false;
  return fused_supported(L->d_model, L->d_ff, L->n_experts, L->top_k, L->bits) && num_sms() <= 1024;
}

void fill_fused_common(FusedParams& P, const bgq_moe_layer* L0, const LayerWs& W) {
  P.d = L0->d_model;
  P.f = L0->d_ff;
  P.E = L0->n_experts;
  P.K = L0->top_k;
  P.timeout_ns = kFusedTimeoutNs;
  P.ctrl = W.ctrl;
  P.h = W.fh;
  P.hk = W.H;
  P.logits = W.logits;
  P.ltag = W.ftag;
  P.part_ss = W.fpart;
  P.route_idx = W.fidx;
  P.route_w = W.fw;
}

FusedLayer fused_layer(const bgq_moe_layer* L, const uint16_t* rho) {
  FusedLayer f;
  f.router = L->router;
  f.sgate = L->shared_gate;
  f.pool_q = L->expert_q;
  f.pool_sb = L->expert_sb;
  f.q_stride = L->expert_q_stride;
  f.sb_stride = L->expert_sb_stride;
  f.shared_q = L->shared_q;
  f.shared_sb = L->shared_sb;
  f.rho = rho;
  return f;
}

}  // namespace

namespace bgq {
// Bytes at the start of a layer workspace that must be zero before a call:
// the control block, the persistent kernel's tagged logits and the
// tensor-core split-K counters. Their places depend on the layer's shape but
// not on the batch.
size_t layer_zero_prefix_bytes(const bgq_moe_layer* L) {
  return carve_layer(nullptr, 1, L->d_model, L->d_ff, L->n_experts, L->top_k).zero_bytes;
}

// moe_layer_forward's argument checks that come before the workspace's, in
// the same order, so that both layer entry points return the same status for
// the same bad call before anything is enqueued.
int layer_call_check(const bgq_moe_layer* L, const uint16_t* x, int batch, const void* out, const void* out_f32) {
  int r = check_layer(L);
  if (r) return r;
  if (!x || !al(x, 16) || (!out && !out_f32)) return BGQ_ERR_INVALID_ARG;
  if ((out && !al(out, 16)) || (out_f32 && !al(out_f32, 16))) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > kMaxBatch) return BGQ_ERR_INVALID_ARG;
  return BGQ_OK;
}
// The last check (after the workspace's): every weight pointer is device
// memory or pinned host memory mapped into the device address space.
int layer_location_check(const bgq_moe_layer* L) {
  return layer_where(L) == Where::kBad ? BGQ_ERR_INVALID_ARG : BGQ_OK;
}
}  // namespace bgq

extern "C" {

const char* bgq_status_string(int32_t s) {
  switch (s) {
    case BGQ_OK: return "ok";
    case BGQ_ERR_INVALID_ARG: return "invalid argument";
    case BGQ_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case BGQ_ERR_CUDA: return "CUDA launch or query failed";
    case BGQ_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case BGQ_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int32_t bgq_abi_version(void) { return 103; }

static int32_t gemv_common(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, int32_t variant,
                           int want_bits, void* stream) {
  int r = check_qmatrix(W);
  if (r) return r;
  if (want_bits && W->bits != want_bits) return BGQ_ERR_INVALID_ARG;
  if (!x || !y || !al(x, 16) || !al(y, 16)) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > 64) return BGQ_ERR_INVALID_ARG;
  if (variant < BGQ_DQ_INT || variant > BGQ_DQ_HOISTED) return BGQ_ERR_INVALID_ARG;
  return cuda_status(launch_qgemv(qm(W), x, batch, y, nullptr, variant, st(stream)));
}

int32_t q4_gemv(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, void* stream) {
  return gemv_common(W, x, y, batch, BGQ_DQ_INT, 4, stream);
}

int32_t q2_gemv(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, void* stream) {
  return gemv_common(W, x, y, batch, BGQ_DQ_INT, 2, stream);
}

int32_t bgq_qgemv_variant(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, int32_t variant,
                          void* stream) {
  return gemv_common(W, x, y, batch, variant, 0, stream);
}

int32_t q8_gemv(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, void* stream) {
  if (!W || !W->q || !W->sb || !x || !y) return BGQ_ERR_INVALID_ARG;
  if (W->bits != 8) return BGQ_ERR_INVALID_ARG;
  if (W->rows <= 0 || W->cols <= 0 || W->cols % kGroup || W->cols > 65536) return BGQ_ERR_INVALID_ARG;
  if (W->group != kGroup && W->group != W->cols) return BGQ_ERR_UNSUPPORTED;
  if (!cols_supported(W->cols, 8) || q8gemv_max_tokens(W->cols) < 1) return BGQ_ERR_UNSUPPORTED;
  if (!al(W->q, 16) || !al(W->sb, 4) || !al(x, 16) || !al(y, 16)) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > 64) return BGQ_ERR_INVALID_ARG;
  const int gpr = W->group == W->cols ? 1 : W->cols / kGroup;
  return cuda_status(launch_q8gemv(qm(W), gpr, x, batch, y, st(stream)));
}

size_t moe_route_workspace_bytes(int32_t batch, int32_t n_experts) {
  if (batch < 1 || n_experts < 1) return 0;
  return sizeof(Ctrl) + up256((size_t)batch * (n_experts + 1) * 4 + (size_t)batch * kMaxTopK * 4);
}

int32_t moe_route_topk(const uint16_t* router, const uint16_t* shared_gate, const uint16_t* x, int32_t batch,
                       int32_t d_model, int32_t n_experts, int32_t top_k, int32_t* idx, float* w, float* gamma,
                       float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (!router || !x || !idx || !w) return BGQ_ERR_INVALID_ARG;
  if (!al(router, 16) || !al(x, 16) || (shared_gate && !al(shared_gate, 16))) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > kMaxBatch || d_model <= 0 || n_experts <= 0 || top_k <= 0) return BGQ_ERR_INVALID_ARG;
  if (top_k > kMaxTopK || n_experts > kMaxExperts || top_k > n_experts) return BGQ_ERR_UNSUPPORTED;
  if (!route_shape_ok(d_model)) return BGQ_ERR_UNSUPPORTED;
  if (!ws || !al(ws, 256) || ws_bytes < moe_route_workspace_bytes(batch, n_experts)) return BGQ_ERR_WORKSPACE;
  Carver c(ws);
  Ctrl* ctrl = c.take<Ctrl>(sizeof(Ctrl));
  float* lg = c.take<float>((size_t)batch * (n_experts + 1) * 4 + (size_t)batch * top_k * 4);
  return cuda_status(launch_route(router, shared_gate, x, batch, d_model, n_experts, top_k, lg, ctrl, idx, w, gamma,
                                  logits, nullptr, kBigTok, st(stream)));
}

size_t moe_expert_workspace_bytes(const bgq_expert* e, int32_t batch) {
  if (!e || batch < 1) return 0;
  const int d = e->gate.cols, f = e->gate.rows;
  const size_t sx = staged_tokens_bytes(d, 4, batch), sh = staged_tokens_bytes(f, 4, batch);
  return sizeof(Ctrl) + up256(plan_bytes(batch, 0)) + up256((size_t)batch * f * 4) +
         up256((size_t)batch * d * 4) + up256(sx > sh ? sx : sh) +
         (batch >= kBigTok ? tc_act_bytes(d, f, batch, 0) : 0);
}

int32_t moe_expert_swiglu(const bgq_expert* e, const uint16_t* x, int32_t batch, uint16_t* y, float* y_f32,
                          void* ws, size_t ws_bytes, void* stream) {
  if (!e) return BGQ_ERR_INVALID_ARG;
  int r;
  if ((r = check_qmatrix(&e->gate)) || (r = check_qmatrix(&e->up)) || (r = check_qmatrix(&e->down))) return r;
  const int d = e->gate.cols, f = e->gate.rows, bits = e->gate.bits;
  if (e->up.rows != f || e->up.cols != d || e->down.rows != d || e->down.cols != f) return BGQ_ERR_INVALID_ARG;
  if (e->up.bits != bits || e->down.bits != bits) return BGQ_ERR_INVALID_ARG;
  if (!x || !al(x, 16) || (!y && !y_f32) || (y && !al(y, 16)) || (y_f32 && !al(y_f32, 16)))
    return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > kMaxBatch) return BGQ_ERR_INVALID_ARG;
  if (!ws || !al(ws, 256) || ws_bytes < moe_expert_workspace_bytes(e, batch)) return BGQ_ERR_WORKSPACE;
  Carver c(ws);
  Ctrl* ctrl = c.take<Ctrl>(sizeof(Ctrl));
  Plan* plan = c.take<Plan>(plan_bytes(batch, 0));
  float* H = c.take<float>((size_t)batch * f * 4);
  float* Y = c.take<float>((size_t)batch * d * 4);
  const size_t sx = staged_tokens_bytes(d, 4, batch), sh = staged_tokens_bytes(f, 4, batch);
  unsigned char* stage = c.take<unsigned char>(sx > sh ? sx : sh);
  unsigned char* tca = batch >= kBigTok ? c.take<unsigned char>(tc_act_bytes(d, f, batch, 0)) : nullptr;
  ExpertSet es{};
  es.shared = ExpertRef{e->gate.q, e->gate.sb, e->up.q, e->up.sb, e->down.q, e->down.sb};
  es.d = d;
  es.f = f;
  es.bits = bits;
  cudaStream_t s = st(stream);
  const int ntasks = (batch + kTaskTok - 1) / kTaskTok;
  Where where = Where::kDevice;
  for (const void* p : {(const void*)e->gate.q, (const void*)e->gate.sb, (const void*)e->up.q, (const void*)e->up.sb,
                        (const void*)e->down.q, (const void*)e->down.sb}) {
    const Where k = where_is(p);
    if (k == Where::kBad) return BGQ_ERR_INVALID_ARG;
    if (k == Where::kHost) where = Where::kHost;
  }
  const int big_min = where == Where::kHost || !tc_layer_ok(es) ? INT_MAX : kBigTok;  // tensor cores from 16 tokens
  if (batch >= big_min) {
    // one tensor-core task holds every token: no plan (the kernels take token n, slot 0) and the down
    // GEMM's epilogue writes y / y_f32 itself, the combine of one slot of weight 1
    if (launch_gateup_tc(es, nullptr, batch, 0, x, H, 1, ctrl, tca, s) != cudaSuccess) return BGQ_ERR_CUDA;
    return cuda_status(launch_down_tc(es, nullptr, batch, 0, H, Y, 1, ctrl, tca, y, y_f32, s));
  }
  // grouped GEMVs: the kernels build the tasks themselves where they can, else from a plan kernel
  const Plan* gp = grouped_planless_ok(es, batch, true) ? nullptr : plan;
  if (gp && launch_plan_single(plan, batch, big_min, s) != cudaSuccess) return BGQ_ERR_CUDA;
  if (launch_gateup(es, gp, ntasks, batch, x, H, 1, stage, s) != cudaSuccess) return BGQ_ERR_CUDA;
  return cuda_status(launch_down(es, gp, ntasks, batch, H, Y, 1, stage, Combine{nullptr, nullptr, 0, y, y_f32}, s));
}

size_t moe_layer_workspace_bytes(const bgq_moe_layer* L, int32_t max_batch) {
  if (!L || max_batch < 1 || L->top_k < 1 || L->n_experts < 1) return 0;
  return carve_layer(nullptr, max_batch, L->d_model, L->d_ff, L->n_experts, L->top_k).bytes;
}

static int32_t layer_forward_impl(const bgq_moe_layer* L, const uint16_t* x, int32_t batch, uint16_t* out,
                                  float* out_f32, int32_t* idx_out, float* w_out, float* gamma_out, const LayerWs& W,
                                  Where where, cudaStream_t s) {
  const ExpertSet es = expert_set(L);
  const int big_min = big_min_for(where, es);
  const int K = L->top_k, E = L->n_experts;
  int32_t* idx = idx_out ? idx_out : W.idx;
  float* w = w_out ? w_out : W.w;
  float* gamma = gamma_out ? gamma_out : W.gamma;
  if (launch_route(L->router, L->shared_gate, x, batch, L->d_model, E, K, W.logits, W.ctrl, idx, w, gamma, nullptr,
                   W.plan, big_min, s) != cudaSuccess)
    return BGQ_ERR_CUDA;
  const int max_tasks = plan_max_tasks(batch, K);
  // experts with fewer than big_min tokens: grouped GEMV; the others: tensor-core GEMM
  if (launch_gateup(es, W.plan, max_tasks, batch, x, W.H, K + 1, W.stage, s) != cudaSuccess) return BGQ_ERR_CUDA;
  const bool tc = batch >= big_min;
  if (tc && launch_gateup_tc(es, W.plan, batch, K, x, W.H, K + 1, W.ctrl, W.tca, s) != cudaSuccess) return BGQ_ERR_CUDA;
  // tensor-core tasks first: the grouped down kernel ends with the weighted combine
  if (tc && launch_down_tc(es, W.plan, batch, K, W.H, W.Y, K + 1, W.ctrl, W.tca, nullptr, nullptr, s) != cudaSuccess)
    return BGQ_ERR_CUDA;
  return cuda_status(
      launch_down(es, W.plan, max_tasks, batch, W.H, W.Y, K + 1, W.stage, Combine{w, gamma, K, out, out_f32}, s));
}

int32_t moe_layer_forward(const bgq_moe_layer* L, const uint16_t* x, int32_t batch, uint16_t* out, float* out_f32,
                          int32_t* idx_out, float* w_out, float* gamma_out, void* ws, size_t ws_bytes, void* stream) {
  int r = bgq::layer_call_check(L, x, batch, out, out_f32);
  if (r) return r;
  if (!ws || !al(ws, 256) || ws_bytes < moe_layer_workspace_bytes(L, batch)) return BGQ_ERR_WORKSPACE;
  const Where where = layer_where(L);
  if (where == Where::kBad) return BGQ_ERR_INVALID_ARG;
  LayerWs W = carve_layer(ws, batch, L->d_model, L->d_ff, L->n_experts, L->top_k);
  if (batch == 1 && where == Where::kDevice && use_fused(L)) {
    static_assert(sizeof(FusedParams) < 32000, "kernel parameter space");
    FusedParams P{};
    fill_fused_common(P, L, W);
    P.n_layers = 1;
    P.stack = 0;
    P.eps = 0.f;
    P.x_in = x;
    P.out = out;
    P.out_f32 = out_f32;
    P.idx_out = idx_out;
    P.w_out = w_out;
    P.gamma_out = gamma_out;
    P.layers[0] = fused_layer(L, nullptr);
    return cuda_status(launch_fused(P, L->bits, st(stream)));
  }
  return layer_forward_impl(L, x, batch, out, out_f32, idx_out, w_out, gamma_out, W, where, st(stream));
}

size_t moe_stream_slots_bytes(const bgq_moe_layer* L, int32_t batch) {
  if (!L || batch < 1 || L->top_k < 1 || L->n_experts < 1 || L->d_model <= 0 || L->d_ff <= 0) return 0;
  if (L->bits != 4 && L->bits != 2) return 0;
  const long long pairs = (long long)batch * L->top_k;
  const int max_slots = (int)(pairs < L->n_experts ? pairs : L->n_experts);
  return (size_t)slot_geo(L->d_model, L->d_ff, L->bits, max_slots).total;
}

int32_t moe_layer_forward_streamed(const bgq_moe_layer* L, const uint16_t* x, int32_t batch, uint16_t* out,
                                   float* out_f32, int32_t* idx_out, float* w_out, float* gamma_out, void* slots,
                                   size_t slots_bytes, void* ws, size_t ws_bytes, void* stream) {
  int r = check_layer(L);
  if (r) return r;
  if (!x || !al(x, 16) || (!out && !out_f32)) return BGQ_ERR_INVALID_ARG;
  if ((out && !al(out, 16)) || (out_f32 && !al(out_f32, 16))) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > kMaxBatch) return BGQ_ERR_INVALID_ARG;
  if (!ws || !al(ws, 256) || ws_bytes < moe_layer_workspace_bytes(L, batch)) return BGQ_ERR_WORKSPACE;
  if (!slots || !al(slots, 256) || slots_bytes < moe_stream_slots_bytes(L, batch)) return BGQ_ERR_WORKSPACE;
  if (layer_where(L) == Where::kBad || where_is(slots) != Where::kDevice) return BGQ_ERR_INVALID_ARG;
  const LayerWs W = carve_layer(ws, batch, L->d_model, L->d_ff, L->n_experts, L->top_k);
  const cudaStream_t s = st(stream);
  const int K = L->top_k, E = L->n_experts;
  int32_t* idx = idx_out ? idx_out : W.idx;
  float* w = w_out ? w_out : W.w;
  float* gamma = gamma_out ? gamma_out : W.gamma;
  // routing and the grouping plan (grouped GEMVs only: no tensor-core tasks)
  if (launch_route(L->router, L->shared_gate, x, batch, L->d_model, E, K, W.logits, W.ctrl, idx, w, gamma, nullptr,
                   W.plan, INT_MAX, s) != cudaSuccess)
    return BGQ_ERR_CUDA;
  // fetch: the selected experts into the slots, then compute on the slots
  const ExpertSet pool = expert_set(L);
  const long long pairs = (long long)batch * K;
  const SlotGeo g = slot_geo(L->d_model, L->d_ff, L->bits, (int)(pairs < E ? pairs : E));
  if (launch_slot_copy(W.plan, E, pool, g, slots, s) != cudaSuccess) return BGQ_ERR_CUDA;
  const ExpertSet es = slot_expert_set(pool, g, slots);
  const int max_tasks = plan_max_tasks(batch, K);
  if (launch_gateup(es, W.plan, max_tasks, batch, x, W.H, K + 1, W.stage, s) != cudaSuccess) return BGQ_ERR_CUDA;
  return cuda_status(
      launch_down(es, W.plan, max_tasks, batch, W.H, W.Y, K + 1, W.stage, Combine{w, gamma, K, out, out_f32}, s));
}

int32_t bgq_rmsnorm(const float* h, const uint16_t* rho, int32_t batch, int32_t d, float eps, uint16_t* a,
                    void* stream) {
  if (!h || !a || !al(h, 16) || !al(a, 16) || (rho && !al(rho, 16))) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || d <= 0 || d % 256 || !(eps >= 0.f)) return BGQ_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm(h, rho, batch, d, eps, a, st(stream)));
}

int32_t bgq_residual_add(float* h, const float* delta, int64_t n, void* stream) {
  if (!h || !delta || n < 0) return BGQ_ERR_INVALID_ARG;
  if (n == 0) return BGQ_OK;
  return cuda_status(launch_residual_add(h, delta, n, st(stream)));
}

static int chain_check(const bgq_qmatrix* W, int32_t n, int32_t batch) {
  if (!W || n < 1 || n > kMaxChain) return BGQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > 8) return BGQ_ERR_INVALID_ARG;
  int max_cols = 0;
  for (int i = 0; i < n; ++i) {
    int r = check_qmatrix(&W[i]);
    if (r) return r;
    if (W[i].bits != W[0].bits) return BGQ_ERR_INVALID_ARG;
    if (i > 0 && W[i].cols != W[i - 1].rows) return BGQ_ERR_INVALID_ARG;
    if (W[i].cols > max_cols) max_cols = W[i].cols;
  }
  // every step's GEMV stages at least one token's input in shared memory
  if (qgemv_int_smem(max_cols, W[0].bits, 1) > (size_t)227 * 1024) return BGQ_ERR_UNSUPPORTED;
  return BGQ_OK;
}
// Row stride of the intermediate vectors (the normalised input, the inner
// steps' outputs): the widest, a multiple of 8.
static int chain_ldb(const bgq_qmatrix* W, int32_t n) {
  int m = W[0].cols > 8 ? W[0].cols : 8;
  for (int i = 0; i + 1 < n; ++i)
    if (W[i].rows > m) m = W[i].rows;
  return (m + 7) & ~7;
}

size_t bgq_gemv_chain_workspace_bytes(const bgq_qmatrix* W, int32_t n, int32_t batch) {
  if (chain_check(W, n, batch)) return 0;
  return sizeof(Ctrl) + 256 + 2 * up256((size_t)batch * chain_ldb(W, n) * 2);
}

// The chain as programmatic dependent launches of the standalone kernels
// (RMSNorm, then one GEMV per step, the residual added in the last GEMV's
// epilogue): each waits for the one before it, and its weight loads start
// while that one finishes. A single persistent launch with grid-wide waits
// between the steps was built and measured slower on this GPU (a grid-wide
// wait on 152 SMs costs more than a dependent launch's boundary).
int32_t bgq_gemv_chain(const bgq_qmatrix* W, int32_t n, const uint16_t* x, int32_t batch, int32_t norm,
                       const uint16_t* rho, float eps, int32_t residual, uint16_t* out, float* out_f32, void* ws,
                       size_t ws_bytes, void* stream) {
  int r = chain_check(W, n, batch);
  if (r) return r;
  if (!x || !al(x, 16) || (!out && !out_f32) || (out && !al(out, 16)) || (out_f32 && !al(out_f32, 16)))
    return BGQ_ERR_INVALID_ARG;
  if (norm && !(eps > 0.f && eps < 1e30f)) return BGQ_ERR_INVALID_ARG;
  if (residual && W[n - 1].rows != W[0].cols) return BGQ_ERR_INVALID_ARG;
  if (!ws || !al(ws, 256) || ws_bytes < bgq_gemv_chain_workspace_bytes(W, n, batch)) return BGQ_ERR_WORKSPACE;
  Carver c(ws);
  c.take<Ctrl>(sizeof(Ctrl));  // the status word, as in every workspace (nothing here waits on the device)
  c.take<int>(256);
  const int ldb = chain_ldb(W, n);
  uint16_t* buf[2] = {c.take<uint16_t>((size_t)batch * ldb * 2), c.take<uint16_t>((size_t)batch * ldb * 2)};
  cudaStream_t s = st(stream);
  const uint16_t* cur = x;
  int k = 0;
  if (norm) {
    if (launch_rmsnorm_bf16(x, rho, batch, W[0].cols, eps, buf[0], s) != cudaSuccess) return BGQ_ERR_CUDA;
    cur = buf[0];
    k = 1;
  }
  for (int i = 0; i < n; ++i) {
    const bool last = i == n - 1;
    if (launch_qgemv(qm(&W[i]), cur, batch, last ? out : buf[k], last ? out_f32 : nullptr, 0, s,
                     last && residual ? x : nullptr) != cudaSuccess)
      return BGQ_ERR_CUDA;
    cur = buf[k];  // vectors packed at the step's own row stride
    k ^= 1;
  }
  return BGQ_OK;
}

size_t moe_stack_workspace_bytes(const bgq_moe_layer* layers, int32_t n_layers) {
  if (!layers || n_layers < 1) return 0;
  const bgq_moe_layer* L = &layers[0];
  size_t b = moe_layer_workspace_bytes(L, 1);
  if (!b) return 0;
  return b + up256((size_t)L->d_model * 4) * 2 + up256((size_t)L->d_model * 2);
}

static int32_t stack_decode_impl(const bgq_moe_layer* layers, const uint16_t* const* rho, int32_t n_layers,
                                 float eps, const uint16_t* x, uint16_t* x_next, float* h_out, int32_t* idx_out,
                                 void* ws, size_t ws_bytes, uint64_t* trace, void* stream);

int32_t moe_stack_decode(const bgq_moe_layer* layers, const uint16_t* const* rho, int32_t n_layers, float eps,
                         const uint16_t* x, uint16_t* x_next, float* h_out, int32_t* idx_out, void* ws,
                         size_t ws_bytes, void* stream) {
  return stack_decode_impl(layers, rho, n_layers, eps, x, x_next, h_out, idx_out, ws, ws_bytes, nullptr, stream);
}

size_t moe_stack_trace_entries(const bgq_moe_layer* layers, int32_t n_layers) {
  if (!layers || n_layers < 1 || !use_fused(&layers[0])) return 0;
  return (size_t)n_layers * num_sms() * kTraceEvents;
}

int32_t moe_stack_decode_traced(const bgq_moe_layer* layers, const uint16_t* const* rho, int32_t n_layers, float eps,
                                const uint16_t* x, uint16_t* x_next, float* h_out, int32_t* idx_out, void* ws,
                                size_t ws_bytes, uint64_t* trace, void* stream) {
  if (!trace || !al(trace, 16)) return BGQ_ERR_INVALID_ARG;
  if (!layers || n_layers < 1 || !use_fused(&layers[0])) return BGQ_ERR_UNSUPPORTED;
  return stack_decode_impl(layers, rho, n_layers, eps, x, x_next, h_out, idx_out, ws, ws_bytes, trace, stream);
}

static int32_t stack_decode_impl(const bgq_moe_layer* layers, const uint16_t* const* rho, int32_t n_layers,
                                 float eps, const uint16_t* x, uint16_t* x_next, float* h_out, int32_t* idx_out,
                                 void* ws, size_t ws_bytes, uint64_t* trace, void* stream) {
  if (!layers || !rho || n_layers < 1 || n_layers > kMaxLayers) return BGQ_ERR_INVALID_ARG;
  const bgq_moe_layer* L0 = &layers[0];
  for (int l = 0; l < n_layers; ++l) {
    int r = check_layer(&layers[l]);
    if (r) return r;
    const bgq_moe_layer* L = &layers[l];
    if (L->d_model != L0->d_model || L->d_ff != L0->d_ff || L->n_experts != L0->n_experts ||
        L->top_k != L0->top_k || L->bits != L0->bits)
      return BGQ_ERR_INVALID_ARG;
    if (!rho[l] || !al(rho[l], 16)) return BGQ_ERR_INVALID_ARG;
  }
  if (!x || !al(x, 16) || (x_next && !al(x_next, 16)) || (h_out && !al(h_out, 16))) return BGQ_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || L0->d_model % 256) return BGQ_ERR_INVALID_ARG;
  if (!ws || !al(ws, 256) || ws_bytes < moe_stack_workspace_bytes(layers, n_layers)) return BGQ_ERR_WORKSPACE;
  const int d = L0->d_model, K = L0->top_k;
  Where wl[kMaxLayers];
  bool all_device = true;
  for (int l = 0; l < n_layers; ++l) {
    wl[l] = layer_where(&layers[l]);
    const Where wr = where_is(rho[l]);
    if (wl[l] == Where::kBad || wr == Where::kBad) return BGQ_ERR_INVALID_ARG;
    all_device = all_device && wl[l] == Where::kDevice && wr == Where::kDevice;
  }
  LayerWs W = carve_layer(ws, 1, d, L0->d_ff, L0->n_experts, K);
  if (trace && !(all_device && use_fused(L0))) return BGQ_ERR_UNSUPPORTED;  // phase timestamps: persistent kernel only
  if (all_device && use_fused(L0)) {
    FusedParams P{};
    fill_fused_common(P, L0, W);
    P.n_layers = n_layers;
    P.stack = 1;
    P.eps = eps;
    P.x_in = x;
    P.x_next = x_next;
    P.h_out = h_out;
    P.idx_out = idx_out;
    P.trace = reinterpret_cast<unsigned long long*>(trace);
    for (int l = 0; l < n_layers; ++l) P.layers[l] = fused_layer(&layers[l], rho[l]);
    return cuda_status(launch_fused(P, L0->bits, st(stream)));
  }
  Carver c(static_cast<char*>(ws) + W.bytes);
  float* h = c.take<float>((size_t)d * 4);
  float* o = c.take<float>((size_t)d * 4);
  uint16_t* a = c.take<uint16_t>((size_t)d * 2);
  cudaStream_t s = st(stream);
  if (launch_widen(x, h, d, s) != cudaSuccess) return BGQ_ERR_CUDA;
  for (int l = 0; l < n_layers; ++l) {
    if (launch_rmsnorm(h, rho[l], 1, d, eps, a, s) != cudaSuccess) return BGQ_ERR_CUDA;
    int r = layer_forward_impl(&layers[l], a, 1, nullptr, o, idx_out ? idx_out + (size_t)l * K : nullptr, nullptr,
                               nullptr, W, wl[l], s);
    if (r) return r;
    if (launch_residual_add(h, o, d, s) != cudaSuccess) return BGQ_ERR_CUDA;
  }
  if (x_next && launch_rmsnorm(h, nullptr, 1, d, eps, x_next, s) != cudaSuccess) return BGQ_ERR_CUDA;
  if (h_out && cudaMemcpyAsync(h_out, h, (size_t)d * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return BGQ_ERR_CUDA;
  return BGQ_OK;
}

int32_t bgq_wait_selftest(void* ws, size_t ws_bytes, int64_t timeout_ns, void* stream) {
  if (!ws || !al(ws, 256) || ws_bytes < sizeof(Ctrl)) return BGQ_ERR_WORKSPACE;
  if (timeout_ns < 1000 || timeout_ns > 1000000000ll) return BGQ_ERR_INVALID_ARG;
  cudaStream_t s = st(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(Ctrl), s) != cudaSuccess) return BGQ_ERR_CUDA;
  return cuda_status(launch_wait_selftest(static_cast<Ctrl*>(ws), timeout_ns, s));
}

int32_t bgq_read_device_status(void* ws, void* stream) {
  if (!ws || !al(ws, 256)) return BGQ_ERR_INVALID_ARG;
  int v = 0;
  cudaStream_t s = st(stream);
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return BGQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BGQ_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpyAsync(ws, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) return BGQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BGQ_ERR_CUDA;
  }
  return v == 0 ? BGQ_OK : (v == BGQ_ERR_TIMEOUT ? BGQ_ERR_TIMEOUT : BGQ_ERR_CUDA);
}

}  // extern "C"
