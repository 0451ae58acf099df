// stream.cu — experts kept outside HBM, copied per layer into HBM slots.
//
// Flash-MoE page, section "架构设计：SSD当显存用": the expert pool does not fit
// in GPU memory, so after routing each layer reads only its K selected experts
// (about 6.75 MB each at 4-bit) into fixed buffers, and the expert kernels run
// on those buffers; the page found that fetching serially, not overlapped with
// GPU work, was best on its unified-memory machine. Here the pool lives in
// pinned host memory (Grace LPDDR behind NVLink-C2C), the buffers are HBM
// "slots", and the fetch is a copy kernel:
//   k_slot_plan   the grouping plan's experts become slot numbers (experts in
//                 ascending order, one slot each) and the list of experts to
//                 copy is written to the slot header;
//   k_copy_slots  every selected expert's codes and scale/bias rows are copied
//                 from the pool into its slot (16-byte loads for the codes,
//                 4-byte loads for scale/bias, whose rows are 4-byte aligned).
// The expert kernels then read the slots as an ordinary expert set.
#include "../../include/bgq.h"
#include "common.cuh"
#include "kernels.h"

namespace bgq {

constexpr int kSlotThreads = 1024;  // one CTA; E <= 1024

// Plan tasks refer to experts 0..E-1 (shared expert: -1). Replace each routed
// expert by its slot (the rank of the expert among the distinct experts of the
// plan) and write hdr[0] = number of slots, hdr[1 + s] = expert of slot s.
__global__ void __launch_bounds__(kSlotThreads) k_slot_plan(Plan* plan, int E, int* hdr) {
  __shared__ int flag[kSlotThreads];
  __shared__ int wsum[kSlotThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Task* tasks = plan_tasks(plan);
  const int ntasks = plan->ntasks;
  flag[tid] = 0;
  __syncthreads();
  for (int i = tid; i < ntasks; i += kSlotThreads)
    if (tasks[i].expert >= 0) flag[tasks[i].expert] = 1;  // idempotent stores
  __syncthreads();
  // exclusive scan of the flags over experts 0..1023
  const int v = flag[tid];
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = wsum[lane];
    int in2 = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(kFull, in2, o);
      if (lane >= o) in2 += u;
    }
    wsum[lane] = in2 - t;  // exclusive
    if (lane == 31) hdr[0] = in2;
  }
  __syncthreads();
  const int slot = wsum[warp] + incl - v;
  __syncthreads();
  flag[tid] = slot;
  if (v && tid < E) hdr[1 + slot] = tid;
  __syncthreads();
  for (int i = tid; i < ntasks; i += kSlotThreads)
    if (tasks[i].expert >= 0) tasks[i].expert = flag[tasks[i].expert];
}

// Copy the experts listed in hdr (hdr[0] of them) from the pool into slots:
// codes q16 16-byte words per expert (pool stride q_stride16), scale/bias sb4
// 4-byte words per expert (pool stride sb_stride4). Slot by slot, the whole
// grid strides over the slot's words with four loads in flight per thread.
__global__ void k_copy_slots(const uint4* __restrict__ pool_q, long long q_stride16, const uint32_t* __restrict__ pool_sb,
                             long long sb_stride4, const int* __restrict__ hdr, int max_slots, long long q16,
                             long long sb4, uint4* __restrict__ slot_q, long long slot_q16, uint32_t* __restrict__ slot_sb,
                             long long slot_sb4) {
  const int n = min(hdr[0], max_slots);
  const long long step = (long long)gridDim.x * blockDim.x;
  const long long g0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (int sl = 0; sl < n; ++sl) {
    const long long e = hdr[1 + sl];
    const uint4* src = pool_q + e * q_stride16;
    uint4* dst = slot_q + sl * slot_q16;
    for (long long i = g0; i < q16; i += 4 * step) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j * step < q16) v[j] = ldg_stream16(src + i + j * step);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i + j * step < q16) dst[i + j * step] = v[j];
    }
    const uint32_t* ss = pool_sb + e * sb_stride4;
    uint32_t* sd = slot_sb + sl * slot_sb4;
    for (long long i = g0; i < sb4; i += step) sd[i] = ldg_stream4(ss + i);
  }
}

SlotGeo slot_geo(int d, int f, int bits, int max_slots) {
  SlotGeo g;
  const long long mw = (long long)d * f * bits / 32;  // code words of one matrix
  const long long mg = (long long)d * f / kGroup * 2;  // bf16 scale/bias values of one matrix
  g.max_slots = max_slots;
  g.q_bytes = 3 * mw * 4;
  g.sb_bytes = 3 * mg * 2;
  g.slot_q = (g.q_bytes + 255) / 256 * 256;
  g.slot_sb = (g.sb_bytes + 255) / 256 * 256;
  g.hdr = ((long long)(1 + max_slots) * 4 + 255) / 256 * 256;
  g.total = g.hdr + (long long)max_slots * (g.slot_q + g.slot_sb);
  return g;
}

cudaError_t launch_slot_copy(Plan* plan, int E, const ExpertSet& pool, const SlotGeo& g, void* slots, cudaStream_t s) {
  int* hdr = static_cast<int*>(slots);
  k_slot_plan<<<1, kSlotThreads, 0, s>>>(plan, E, hdr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  unsigned char* base = static_cast<unsigned char*>(slots);
  uint4* slot_q = reinterpret_cast<uint4*>(base + g.hdr);
  uint32_t* slot_sb = reinterpret_cast<uint32_t*>(base + g.hdr + (long long)g.max_slots * g.slot_q);
  k_copy_slots<<<num_sms() * 4, 256, 0, s>>>(reinterpret_cast<const uint4*>(pool.pool_q), pool.q_stride / 4,
                                             reinterpret_cast<const uint32_t*>(pool.pool_sb), pool.sb_stride / 2, hdr,
                                             g.max_slots, g.q_bytes / 16, g.sb_bytes / 4, slot_q, g.slot_q / 16,
                                             slot_sb, g.slot_sb / 4);
  return cudaGetLastError();
}

ExpertSet slot_expert_set(const ExpertSet& pool, const SlotGeo& g, void* slots) {
  unsigned char* base = static_cast<unsigned char*>(slots);
  ExpertSet es = pool;
  es.pool_q = reinterpret_cast<const uint32_t*>(base + g.hdr);
  es.pool_sb = reinterpret_cast<const uint16_t*>(base + g.hdr + (long long)g.max_slots * g.slot_q);
  es.q_stride = g.slot_q / 4;
  es.sb_stride = g.slot_sb / 2;
  return es;
}

}  // namespace bgq
