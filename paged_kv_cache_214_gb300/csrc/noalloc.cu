// noalloc.cu — decode attention that needs no caller-provided workspace.
//
// paged_decode_attention needs device scratch (split partials and arrival
// counters) that its caller allocates.  Some callers cannot allocate device
// memory: a plugin whose host framework owns every device allocation and hands
// the library only its input and output tensors, or a runtime working under a
// fixed memory plan in which no call may allocate.  This entry point serves
// them with scratch that the library itself carries: a fixed-size array in
// device global memory (16 MiB, see PKV_NOALLOC_SCRATCH_BYTES), created when the
// library is loaded on a device and held until the process exits.
//
// The array is a device symbol.  Host code cannot use its name as an address
// (on the host the name is only a stand-in), so the device address is looked up
// with cudaGetSymbolAddress once per device, the first time the entry point is
// called on that device, and cached.  The cached address belongs to the
// device's current context: after cudaDeviceReset on a device this entry
// point must not be called on that device again in the same process.

#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevicesNoAlloc = 64;

// Scratch of every no-allocation decode call on this device: arrival counters
// at its start, split partials after them (the layout paged_decode_attention
// uses for a caller's workspace).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevicesNoAlloc];

// Device address of the scratch array on the current device (looked up once
// per device); nullptr if the lookup fails.
void* noalloc_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoAlloc) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_decode_attention_noalloc(void* out, float* lse, const void* q,
                                              const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables,
                                              int max_blocks_per_seq,
                                              const int32_t* context_lens, int B, int Hq,
                                              int Hkv, int D, int block_size,
                                              int64_t num_blocks, float scale, int num_splits,
                                              pkv_stream_t stream) {
  // Every argument check of the decode call runs first: a refused call
  // queues nothing on the stream (not even the counter clear below).
  const DecodeArgs args{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                        context_lens, B, Hq, Hkv, num_blocks, scale, nullptr, 0,
                        num_splits, 0};
  int st = check_decode_args(args, D, block_size);
  if (st || B == 0) return st;
  DecodePlan plan;
  st = plan_decode(B, Hq, Hkv, max_blocks_per_seq, num_splits, device_sm_count(), 0, &plan);
  if (st) return st;
  // This call's partials and counters must fit the fixed scratch array.
  if (plan.workspace_bytes > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
  void* scratch = noalloc_scratch();
  if (!scratch) return PKV_ERR_LAUNCH;
  if (plan.workspace_bytes) {
    // The array keeps whatever the previous call left.  The counters must start
    // at zero; clear this call's counters (the start of the array) on its stream.
    const size_t counters = static_cast<size_t>(B) * Hkv * plan.head_groups * sizeof(unsigned);
    if (cudaMemsetAsync(scratch, 0, counters, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return PKV_ERR_LAUNCH;
  }
  return paged_decode_attention(out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, B, Hq, Hkv, D, block_size, num_blocks, scale,
                                scratch, kNoAllocScratchBytes, num_splits, stream);
}
