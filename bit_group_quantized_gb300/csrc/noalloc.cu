// noalloc.cu — moe_layer_forward_noalloc: the MoE layer forward without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory when they need a layer forward:
// a plugin hosted inside a framework that owns the CUDA allocator and offers
// it no workspace hook, a process that must not allocate after start-up
// because its memory budget is fixed, or a foreign-function caller that can
// pass tensors but has no way to create one. For them this entry point runs
// the same kernels as moe_layer_forward with its scratch memory taken from a
// fixed array that lives in the library itself.
//
// The array is a file-scope __device__ variable of kStaticScratchBytes. Every
// GPU that loads the library holds one copy of it until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and keeps it for later calls on that device.
#include <mutex>

#include "../../include/bgq.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_layer_scratch[kStaticScratchBytes];

std::mutex g_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_layer_scratch on the current device (set up once per device).
int32_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BGQ_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layer_scratch) != cudaSuccess || !p) return BGQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return BGQ_OK;
}

}  // namespace

extern "C" {

int32_t moe_layer_forward_noalloc(const bgq_moe_layer* L, const uint16_t* x, int32_t batch, uint16_t* out,
                                  float* out_f32, int32_t* idx_out, float* w_out, float* gamma_out, void* stream) {
  if (!L) return BGQ_ERR_INVALID_ARG;
  const size_t need = moe_layer_workspace_bytes(L, batch);
  if (need == 0) return BGQ_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return BGQ_ERR_WORKSPACE;  // this batch/shape needs more than the fixed array
  void* ws = nullptr;
  int32_t r = scratch_for_current_device(&ws);
  if (r != BGQ_OK) return r;
  // The array keeps whatever the previous call left; only its first bytes (the
  // control block: status word and counters, and the batch-1 kernel's tagged
  // routing logits) have to start at zero (every other region is written
  // before it is read).
  if (cudaMemsetAsync(ws, 0, bgq::layer_zero_prefix_bytes(L->n_experts), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return BGQ_ERR_CUDA;
  return moe_layer_forward(L, x, batch, out, out_f32, idx_out, w_out, gamma_out, ws, kStaticScratchBytes, stream);
}

}  // extern "C"
