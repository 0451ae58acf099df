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
// that device current) and keeps it for later calls on that device. The kept
// address belongs to the device's current context: after cudaDeviceReset the
// entry point must not be used again in the process.
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
  // The same checks, in the same order, as moe_layer_forward (the fixed array
  // standing in for the workspace), all before anything is enqueued.
  int32_t r = bgq::layer_call_check(L, x, batch, out, out_f32);
  if (r != BGQ_OK) return r;
  if (moe_layer_workspace_bytes(L, batch) > kStaticScratchBytes) return BGQ_ERR_WORKSPACE;
  r = bgq::layer_location_check(L);
  if (r != BGQ_OK) return r;
  void* ws = nullptr;
  r = scratch_for_current_device(&ws);
  if (r != BGQ_OK) return r;
  // The array keeps whatever the previous call (of any layer shape) left. The
  // leading bytes that the kernels expect at zero (the control block with its
  // status word and counters, the batch-1 kernel's tagged routing logits and
  // the tensor-core split-K tile counters) are cleared on every call; every
  // other region is written before it is read. A call that ended in
  // BGQ_ERR_TIMEOUT therefore leaves nothing that the next call would read.
  if (cudaMemsetAsync(ws, 0, bgq::layer_zero_prefix_bytes(L), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return BGQ_ERR_CUDA;
  return moe_layer_forward(L, x, batch, out, out_f32, idx_out, w_out, gamma_out, ws, kStaticScratchBytes, stream);
}

}  // extern "C"
