/*
 * bgq.h — C ABI of libbgq.so: 4-bit / 2-bit group-quantized Mixture-of-Experts
 * decode on one NVIDIA GB300 (sm_103a).
 *
 * Method (source: "397B参数的模型跑在48GB笔记本上：Flash-MoE用纯C打爆Python推理框架",
 * blog.js-css.com/topics/2026/03/23/519):
 *   - layer shape, section "先搞清楚为什么这件事很难": 512 routed experts per layer,
 *     each token uses 4 of them plus 1 shared expert;
 *   - per-token pipeline, section "架构设计：SSD当显存用": routing logits, softmax +
 *     top-K, the selected experts' forward pass, combine, norm;
 *   - weight format, section "FMA Dequant：一条指令省12%": every weight is
 *     nibble*scale + bias, and the product with x is reordered into
 *     fma(nibble, scale*x, bias*x);
 *   - section "2-bit vs 4-bit": the same layer at 2 bits per weight.
 * Values the page leaves open are fixed by the workload definition: a group of
 * 64 consecutive columns shares one bf16 scale and one bf16 bias; codes are
 * packed least-significant-first, 8 (4-bit) or 16 (2-bit) per uint32 along a
 * row; the top-K weights are renormalised to sum to 1; equal router logits go
 * to the lower expert index; the shared expert is scaled by sigmoid(g . x);
 * every accumulation is fp32 and API outputs are rounded once to bf16.
 *
 * Conventions for every entry point
 *   - All array pointers are DEVICE pointers owned by the caller, unless the
 *     argument is documented as a host pointer. The library allocates no
 *     memory, keeps no state between calls (moe_layer_forward_noalloc's fixed
 *     scratch array is the one exception) and never synchronises the host.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Outputs are valid once the stream reaches that point.
 *   - Arguments are validated before anything is enqueued; a failed check
 *     returns BGQ_ERR_INVALID_ARG / BGQ_ERR_UNSUPPORTED / BGQ_ERR_WORKSPACE and
 *     launches nothing. A failed launch returns BGQ_ERR_CUDA.
 *   - Conditions only the GPU can see (a bounded wait that ran out) are written
 *     to the workspace status word; read it with bgq_read_device_status().
 *     A workspace whose call ended in BGQ_ERR_TIMEOUT must be zero-filled again
 *     before it is reused (counters and exchange words are left mid-call).
 *   - Device pointers must be 16-byte aligned (codes, x, outputs) and 4-byte
 *     aligned (scale/bias). Workspaces must be 256-byte aligned and zero-filled
 *     once before first use (the kernels leave their counters at zero).
 *   - bf16 values are passed as their uint16 bit patterns.
 *   - Calls sharing one workspace must not run concurrently.
 *   - Weights of moe_layer_forward, moe_stack_decode and moe_expert_swiglu
 *     (router, shared gate, expert pools, RMSNorm weights) may also live in
 *     pinned host memory mapped into the device address space (e.g. Grace
 *     memory on a GB300 node, read over the CPU-GPU link): the Flash-MoE
 *     page's idea of keeping the experts outside GPU memory and streaming
 *     only the selected ones (section "架构设计：SSD当显存用"). Such layers
 *     run on the kernels that read weights with plain loads (router, grouped
 *     GEMVs, combine): every expert row is read once per call, directly from
 *     host memory. Pointers the CUDA runtime does not know (unregistered
 *     pageable memory) are rejected with BGQ_ERR_INVALID_ARG.
 */
#ifndef BGQ_H
#define BGQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum {
  BGQ_OK = 0,
  BGQ_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, misalignment, bad enum */
  BGQ_ERR_UNSUPPORTED = 2, /* valid but not implemented shape (see each call) */
  BGQ_ERR_CUDA = 3,        /* a CUDA launch or query failed */
  BGQ_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (status word) */
  BGQ_ERR_WORKSPACE = 5    /* workspace pointer NULL or smaller than required */
};

/* Dequantisation variants of the GEMV (bgq_qgemv_variant).
 * BGQ_DQ_INT       production: per group, y += s*sum(q*x) + b*sum(x), the inner
 *                  sum in exact integer arithmetic on x held as 24-bit fixed point
 *                  with one power-of-two exponent per group of 64 (dp4a): every
 *                  bf16 input within 2^15 of its group's largest magnitude is
 *                  exact, an fp32 input keeps 23 bits below it.
 * BGQ_DQ_STANDARD  per weight: acc += (q*s + b) * x        (the page's "standard").
 * BGQ_DQ_REORDERED per weight: acc += fma(q, s*x, b*x)     (the page's reordering).
 * BGQ_DQ_HOISTED   per group:  y += s*sum(q*x) + b*sum(x), fp32 FMAs per weight
 *                  (the reordering summed over a group, where s and b are constant). */
enum { BGQ_DQ_INT = 0, BGQ_DQ_STANDARD = 1, BGQ_DQ_REORDERED = 2, BGQ_DQ_HOISTED = 3 };

/* One group-quantized matrix W [rows x cols] (host struct, device arrays).
 *   q  : codes, uint32 [rows][cols*bits/32]; column k of a row is in word
 *        k/(32/bits) at bit offset bits*(k%(32/bits)).
 *   sb : bf16 pairs [rows][cols/64][2] = (scale, bias) of each group of 64.
 *   W[n][k] = q[n][k]*scale[n][k/64] + bias[n][k/64].
 *   bits is 4 or 2; group must be 64; cols a multiple of 64 such that
 *   P = cols*bits/128 divides 32 or is a multiple of 32 (e.g. 64..1024 by powers
 *   of two, and any multiple of 1024 (4-bit) / 2048 (2-bit)). */
typedef struct bgq_qmatrix {
  const uint32_t* q;
  const uint16_t* sb;
  int32_t rows;
  int32_t cols;
  int32_t bits;
  int32_t group;
} bgq_qmatrix;

/* One SwiGLU expert: y = down( silu(gate x) * (up x) ).
 * gate and up are [d_ff x d_model], down is [d_model x d_ff]. */
typedef struct bgq_expert {
  bgq_qmatrix gate;
  bgq_qmatrix up;
  bgq_qmatrix down;
} bgq_expert;

/* One MoE layer (host struct, device arrays).
 *   router      : bf16 [n_experts][d_model].
 *   shared_gate : bf16 [d_model]; gamma = sigmoid(shared_gate . x). NULL: gamma = 1.
 *   expert_q/sb : pool of routed experts. Expert e starts at
 *                 expert_q + e*expert_q_stride (uint32 words) and
 *                 expert_sb + e*expert_sb_stride (bf16 elements). Inside an
 *                 expert the matrices follow each other: gate, up, down, each
 *                 in the bgq_qmatrix layout (gate at word 0, up at word
 *                 d_ff*d_model*bits/32, down at twice that; the same order for
 *                 sb with d_ff*(d_model/64)*2 elements per matrix).
 *   shared_q/sb : the shared expert, same internal layout.
 *   Limits: 1 <= top_k <= 8, top_k <= n_experts <= 1024, d_model and d_ff
 *   valid bgq_qmatrix column counts, bits 4 or 2, group 64. */
typedef struct bgq_moe_layer {
  int32_t d_model;
  int32_t d_ff;
  int32_t n_experts;
  int32_t top_k;
  int32_t bits;
  int32_t group;
  const uint16_t* router;
  const uint16_t* shared_gate;
  const uint32_t* expert_q;
  const uint16_t* expert_sb;
  int64_t expert_q_stride;
  int64_t expert_sb_stride;
  const uint32_t* shared_q;
  const uint16_t* shared_sb;
} bgq_moe_layer;

/* Human-readable name of a status code (static string). */
const char* bgq_status_string(int32_t status);

/* ABI version of this header (major*100 + minor): 103. */
int32_t bgq_abi_version(void);

/* Overlapped launch of the GEMVs (q4_gemv, q2_gemv, bgq_qgemv_variant, q8_gemv):
 * their kernels are launched with programmatic dependent launch, so a GEMV may
 * start while the kernel before it on the stream is still running. Before it
 * waits for that kernel it reads only W (q and sb): W must not be written by
 * the kernels enqueued just before the call on the same stream (weights are
 * normally written once, long before). x is read and y written only after
 * every earlier kernel on the stream has completed, as with a plain launch. */

/* y[b][n] = bf16( sum_k W[n][k] * x[b][k] ), b < batch, fp32 accumulation.
 * The standalone GEMV of the format (Flash-MoE page, "FMA Dequant").
 * W->bits must be 4 for q4_gemv and 2 for q2_gemv. x: bf16 [batch][cols],
 * y: bf16 [batch][rows]. 1 <= batch <= 64. Production variant BGQ_DQ_INT. */
int32_t q4_gemv(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, void* stream);
int32_t q2_gemv(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, void* stream);

/* The same GEMV with an explicit dequantisation variant (BGQ_DQ_*), for the
 * page's standard-vs-reordered comparison. Any bits (4 or 2). */
int32_t bgq_qgemv_variant(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch,
                          int32_t variant, void* stream);

/* y[b][n] = bf16( sum_k W[n][k] * x[b][k] ), b < batch, fp32 accumulation, for
 * 8-bit weights: the int8 format of dense MLP and QKV projections.
 * Source: "Redis 之父下场手写推理引擎：antirez 用约 24000 行原生代码驯服视频生成模型"
 * (text-matrix.pages.dev), the paragraph on --use-int8-row-fc2: MLP weights are
 * int8 with one scale per group, and FC2 can instead carry one scale per row.
 *   W->bits must be 8: codes q in 0..255, four per uint32, code k of a row in
 *     word k/4 at bit offset 8*(k%4); W[n][k] = q[n][k]*scale + bias.
 *   W->group = 64: sb is bf16 [rows][cols/64][2], one (scale, bias) per group;
 *   W->group = W->cols: the per-row format, sb is bf16 [rows][1][2].
 *   Symmetric signed int8 c (W = c*scale) is stored as q = c + 128 with
 *   bias = -128*scale (exact in bf16).
 *   cols: 64, 128, 256 or a multiple of 512, at most 65536.
 *   x: bf16 [batch][cols], y: bf16 [batch][rows], 1 <= batch <= 64 (inputs
 *   are staged in groups of up to 8 per launch, fewer for cols > 8192; W is
 *   read once per group). Alignment: q, x, y 16 bytes; sb 4 bytes.
 * Errors: BGQ_ERR_INVALID_ARG (NULL, bits != 8, bad sizes, misalignment),
 * BGQ_ERR_UNSUPPORTED (group neither 64 nor cols, cols shape), BGQ_ERR_CUDA. */
int32_t q8_gemv(const bgq_qmatrix* W, const uint16_t* x, uint16_t* y, int32_t batch, void* stream);

/* Router of a batch of tokens (Flash-MoE page, "架构设计": routing, then
 * softmax + top-K on the logits).
 *   logits_l[b][e] = router[e] . x[b] (fp32), p = softmax_fp32(l[b]),
 *   idx[b][0..top_k) = the top_k experts by logit, largest first, equal logits
 *   to the lower index; w[b][k] = p[idx] / sum_j p[idx_j];
 *   gamma[b] = sigmoid(shared_gate . x[b]) (1 if shared_gate is NULL).
 * x: bf16 [batch][d_model]. idx: int32 [batch][top_k]. w: fp32 [batch][top_k].
 * gamma (nullable): fp32 [batch]. logits (nullable): fp32 [batch][n_experts].
 * ws: workspace of moe_route_workspace_bytes(batch, n_experts) bytes.
 * 1 <= batch <= 256; d_model a multiple of 256. */
size_t moe_route_workspace_bytes(int32_t batch, int32_t n_experts);
int32_t moe_route_topk(const uint16_t* router, const uint16_t* shared_gate, const uint16_t* x,
                       int32_t batch, int32_t d_model, int32_t n_experts, int32_t top_k,
                       int32_t* idx, float* w, float* gamma, float* logits,
                       void* ws, size_t ws_bytes, void* stream);

/* One SwiGLU expert on a batch (Flash-MoE page, "架构设计": expert forward):
 *   h = silu(gate x) * (up x) (fp32, never rounded), y = down h.
 * x: bf16 [batch][d_model]; y (nullable): bf16 [batch][d_model];
 * y_f32 (nullable): fp32 [batch][d_model]. 1 <= batch <= 256.
 * ws: moe_expert_workspace_bytes(e, batch) bytes.
 * Paths: batch < 16 runs the integer group dot products (exact sums of the
 * 24-bit fixed-point inputs); batch >= 16 (device-resident weights whose rows
 * are 16-byte aligned) the tensor cores, with weights dequantised to fp16
 * and each token scaled by a power of two into fp16's range (relative error
 * about 5e-4 beyond the bf16 output rounding). Either path is deterministic;
 * the two do not give the same bits. */
size_t moe_expert_workspace_bytes(const bgq_expert* e, int32_t batch);
int32_t moe_expert_swiglu(const bgq_expert* e, const uint16_t* x, int32_t batch,
                          uint16_t* y, float* y_f32, void* ws, size_t ws_bytes, void* stream);

/* One MoE layer on a batch of decode tokens:
 *   out[b] = sum_k w[b][k] * expert_{idx[b][k]}(x[b]) + gamma[b] * shared(x[b]),
 * summed in fp32 in the order k = 0..top_k-1, then the shared expert.
 * For batch > 1 the (token, expert) pairs are grouped by expert so each expert's
 * weights are read once per call; an expert (the shared one included) that
 * receives 32 or more tokens in a call runs on the tensor cores (see
 * moe_expert_swiglu), the others on the integer group dot products. A
 * token's result does not depend on the other tokens of the batch as long as
 * its experts stay on the same path.
 * x: bf16 [batch][d_model]. out (nullable): bf16 [batch][d_model].
 * out_f32 (nullable): fp32 [batch][d_model] (unrounded). idx_out (nullable):
 * int32 [batch][top_k]. w_out (nullable): fp32 [batch][top_k].
 * gamma_out (nullable): fp32 [batch]. 1 <= batch <= 256.
 * ws: moe_layer_workspace_bytes(L, batch) bytes. */
size_t moe_layer_workspace_bytes(const bgq_moe_layer* L, int32_t max_batch);
int32_t moe_layer_forward(const bgq_moe_layer* L, const uint16_t* x, int32_t batch,
                          uint16_t* out, float* out_f32, int32_t* idx_out, float* w_out,
                          float* gamma_out, void* ws, size_t ws_bytes, void* stream);

/* moe_layer_forward without a workspace argument. The Flash-MoE page has no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory at the point where they run a layer (a plugin inside a framework that
 * owns the allocator and gives it no workspace, a process whose memory budget
 * is fixed after start-up, a foreign-function caller that can pass buffers but
 * not create them).
 * Same arguments, kernels and results as moe_layer_forward; the scratch memory
 * is a 4 MiB array inside the library (held on every GPU that loads the
 * library until the process exits), enough for batch <= 31 at d_model 4096,
 * d_ff 1024, 512 experts, top-4. A call whose moe_layer_workspace_bytes(L,
 * batch) exceeds 4 MiB returns BGQ_ERR_WORKSPACE and launches nothing.
 * Every argument check of moe_layer_forward runs first, in the same order,
 * with the same status codes; nothing is enqueued when one fails.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it; make that
 * first call before any stream capture, and do not call this entry point again
 * after cudaDeviceReset in the same process. Each call clears, on `stream`,
 * the leading bytes of the array that the kernels expect at zero (the
 * 256-byte control block and the batch-1 kernel's (n_experts + 1) tagged
 * logit words, each rounded up to 256 bytes; their sizes depend on the
 * layer's shape, not on the batch), then runs
 * the layer. Every other region is written before it is read, so calls of
 * different layer shapes may follow each other, and a call that ended in
 * BGQ_ERR_TIMEOUT needs no clean-up before the next one. All calls on a device
 * share the one array, which keeps the last call's contents: calls that can
 * overlap on the GPU (on different streams, or from different host threads)
 * race and must be serialised by the caller. Allocates nothing. */
int32_t moe_layer_forward_noalloc(const bgq_moe_layer* L, const uint16_t* x, int32_t batch, uint16_t* out,
                                  float* out_f32, int32_t* idx_out, float* w_out, float* gamma_out, void* stream);

/* moe_layer_forward with the selected experts fetched first (Flash-MoE page,
 * section "架构设计：SSD当显存用": the pool stays outside GPU memory; after
 * routing, each layer reads only its selected experts into fixed buffers and
 * runs the expert kernels on those, fetch and compute one after the other).
 * Here the routed pool is normally in pinned host memory (see above) and the
 * buffers are `slots`, device memory of moe_stream_slots_bytes(L, batch)
 * bytes, 256-byte aligned, caller-owned: a header, then min(batch * top_k,
 * n_experts) expert slots of the pool's codes and scale/bias rows (gate, up,
 * down). Every distinct selected expert is copied once per call, then the
 * grouped expert kernels read the slots. The same layer through
 * moe_layer_forward reads the host-resident experts directly while computing
 * (fetch overlapped with compute); both give bit-identical results for
 * batches below 16 tokens per expert. Other arguments as moe_layer_forward.
 * Errors: as moe_layer_forward; slots NULL, misaligned or too small =>
 * BGQ_ERR_WORKSPACE; slots not device memory => BGQ_ERR_INVALID_ARG. */
size_t moe_stream_slots_bytes(const bgq_moe_layer* L, int32_t batch);
int32_t moe_layer_forward_streamed(const bgq_moe_layer* L, const uint16_t* x, int32_t batch, uint16_t* out,
                                   float* out_f32, int32_t* idx_out, float* w_out, float* gamma_out, void* slots,
                                   size_t slots_bytes, void* ws, size_t ws_bytes, void* stream);

/* a[b] = bf16( h[b] / sqrt(mean(h[b]^2) + eps) * rho ) — the RMSNorm placed
 * before each layer of a decode stack (Flash-MoE page, "架构设计": "norm").
 * h: fp32 [batch][d]; rho (nullable => 1): bf16 [d]; a: bf16 [batch][d].
 * d a multiple of 256, 1 <= batch <= 65535. */
int32_t bgq_rmsnorm(const float* h, const uint16_t* rho, int32_t batch, int32_t d, float eps,
                    uint16_t* a, void* stream);

/* h[b] += delta[b] (fp32 residual add between layers), n = batch*d elements. */
int32_t bgq_residual_add(float* h, const float* delta, int64_t n, void* stream);

/* A chain of dependent group-quantized GEMVs: the decoder's projections
 * around the MoE block (Flash-MoE page, section "架构设计：SSD当显存用":
 * attention input projections in CMD1, o_proj + norm in CMD2; the attention
 * mixing itself is not part of this library, so each projection feeds the
 * next):
 *   v_0 = norm ? bf16(rmsnorm(x) * rho) : x        (rho NULL => 1; as bgq_rmsnorm)
 *   v_i = bf16(W_i v_{i-1}),  i = 1..n-1            (as q4_gemv / q2_gemv)
 *   out_f32 = W_n v_{n-1} (+ x when residual), out = bf16(out_f32)
 * W: HOST array of n bgq_qmatrix, 1 <= n <= 8, all of the same bits (4 or 2),
 * group 64; W[0].cols = d, W[i].cols = W[i-1].rows; residual needs
 * W[n-1].rows = d. x: bf16 [batch][d], 16-byte aligned; out (bf16) and
 * out_f32 (fp32), [batch][W[n-1].rows], nullable but not both, 16-byte
 * aligned. 1 <= batch <= 8; one staged input of the widest W[i].cols must
 * fit in 227 KB of shared memory (3 bytes per value + 8 per 32 values: up to
 * about 71,000 columns) else BGQ_ERR_UNSUPPORTED. eps > 0 when norm.
 * ws: bgq_gemv_chain_workspace_bytes(W, n, batch) bytes, 256-byte aligned,
 * written before read (the intermediate vectors). The steps run as
 * programmatic dependent launches of the RMSNorm and GEMV kernels on
 * `stream` (each step's weight loads start while the previous step
 * finishes; the residual is added in the last GEMV). The result has the bits
 * of the separate calls (bgq_rmsnorm on the widened x, then q4_gemv per
 * step, the last step's fp32 sum plus x). As for every GEMV, the weights
 * must not be written by the kernel just before the call on its stream. */
size_t bgq_gemv_chain_workspace_bytes(const bgq_qmatrix* W, int32_t n, int32_t batch);
int32_t bgq_gemv_chain(const bgq_qmatrix* W, int32_t n, const uint16_t* x, int32_t batch, int32_t norm,
                       const uint16_t* rho, float eps, int32_t residual, uint16_t* out, float* out_f32, void* ws,
                       size_t ws_bytes, void* stream);

/* One decode token through a stack of n_layers resident layers (batch 1):
 *   h = x (widened to fp32); for each layer l:
 *     a = bf16(rmsnorm(h, rho[l], eps)); h += layer_l(a)  (fp32, unrounded);
 *   x_next = bf16(rmsnorm(h, none, eps)).
 * layers: HOST array of n_layers bgq_moe_layer (all with the same shape).
 * rho: HOST array of n_layers device pointers to bf16 [d_model].
 * x: bf16 [d_model]. x_next (nullable): bf16 [d_model]. h_out (nullable):
 * fp32 [d_model]. idx_out (nullable): int32 [n_layers][top_k].
 * 1 <= n_layers <= 128. ws: moe_stack_workspace_bytes(layers, n_layers). */
size_t moe_stack_workspace_bytes(const bgq_moe_layer* layers, int32_t n_layers);
int32_t moe_stack_decode(const bgq_moe_layer* layers, const uint16_t* const* rho, int32_t n_layers,
                         float eps, const uint16_t* x, uint16_t* x_next, float* h_out,
                         int32_t* idx_out, void* ws, size_t ws_bytes, void* stream);

/* moe_stack_decode that also records when each phase of each layer starts on
 * each SM (the device-side counterpart of a per-layer --timing report).
 * trace: device uint64 [n_layers][n_sm][16] of %globaltimer values (ns),
 * moe_stack_trace_entries(layers, n_layers) entries, 16-byte aligned. Events,
 * in the order they happen: 0 layer start, 1 previous layer complete
 * (grid-wide), 2 input normalised, 3 router rows done, 12 input staged,
 * 4 shared gate/up done, 5 all logits visible, 11 experts selected,
 * 6 selected gate/up done, 7 all SwiGLU outputs visible, 13 SwiGLU outputs
 * staged, 9 down rows landed, 10 down rows done, 8 combine done; 14 and 15:
 * the first and the last chunk of the selected gate/up rows landed.
 * Available when the layers take the persistent batch-1 kernel (otherwise
 * moe_stack_trace_entries returns 0 and the call BGQ_ERR_UNSUPPORTED). */
size_t moe_stack_trace_entries(const bgq_moe_layer* layers, int32_t n_layers);
int32_t moe_stack_decode_traced(const bgq_moe_layer* layers, const uint16_t* const* rho, int32_t n_layers,
                                float eps, const uint16_t* x, uint16_t* x_next, float* h_out, int32_t* idx_out,
                                void* ws, size_t ws_bytes, uint64_t* trace, void* stream);

/* Self-test of the bounded device-side wait used by the persistent decode
 * kernel: clears the control block of `ws` (>= 256 bytes) and launches two
 * CTAs that wait on a counter nothing increments. The wait gives up after
 * timeout_ns (1e3 .. 1e9), writes BGQ_ERR_TIMEOUT to the status word and the
 * kernel returns; bgq_read_device_status(ws) then reports BGQ_ERR_TIMEOUT.
 * Nothing faults or hangs. Leaves the workspace needing a re-zero. */
int32_t bgq_wait_selftest(void* ws, size_t ws_bytes, int64_t timeout_ns, void* stream);

/* Synchronises `stream`, then returns the status word that the kernels of the
 * calls above left in workspace `ws` (BGQ_OK or BGQ_ERR_TIMEOUT), and clears it. */
int32_t bgq_read_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BGQ_H */
