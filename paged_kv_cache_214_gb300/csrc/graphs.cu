// Decode steps replayed from CUDA graphs captured per batch bucket
// ("Nano-vLLM System Architecture Analysis", §2 Core Components, "CUDA
// Graphs"; comparison table, "Variable-batch CUDA Graphs").  The runner sits on
// the library's public calls: each graph is the capture of one
// paged_decode_attention_store (or its E4M3 form) over a bucket's rows of the
// caller's static buffers, after a one-block kernel that marks the rows past
// the step's batch as empty.  The batch size reaches that kernel as a launch
// argument, rewritten in the instantiated graph before a replay whose batch
// differs from the previous replay's.  A batch that fills its bucket replays a
// second graph of the step alone.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "pkv.h"
#include "pkv_graphs.h"

namespace {

constexpr size_t kCounterBytes = size_t{1} << 20;   // arrival counters of the workspace
constexpr int kPadThreads = 512;

// Rows [from, to): context length 0 and no new token.
__global__ void __launch_bounds__(kPadThreads) decode_graph_pad_kernel(int32_t* context_lens,
                                                                       int32_t* slot_mapping,
                                                                       int from, int to) {
  for (int r = from + static_cast<int>(threadIdx.x); r < to; r += kPadThreads) {
    context_lens[r] = 0;
    slot_mapping[r] = -1;
  }
}

struct Bucket {
  int size = 0;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraph_t full_graph = nullptr;      // the step alone, for B == size
  cudaGraphExec_t full_exec = nullptr;
  cudaGraphNode_t pad = nullptr;   // the pad kernel's node in `graph`
  void* pad_func = nullptr;        // that node's kernel, as the node reports it
  int pad_from = 0;                // its current `from` argument
};

bool valid_list(const int32_t* b, int n) {
  if (!b || n < 1) return false;
  if (b[0] < 1) return false;
  for (int i = 1; i < n; ++i)
    if (b[i] <= b[i - 1]) return false;
  return true;
}

// The step over rows [0, B) of the static buffers.
int step(const pkv_decode_graphs_config& c, int B, cudaStream_t s) {
  const int64_t stride = static_cast<int64_t>(c.Hkv) * c.D;
  if (c.kv_fp8)
    return paged_decode_attention_fp8_store(
        c.out, c.lse, c.q, c.k_new, c.v_new, stride, stride, c.slot_mapping, c.k_cache,
        c.v_cache, c.block_tables, c.max_blocks_per_seq, c.context_lens, B, c.Hq, c.Hkv, c.D,
        c.block_size, c.num_blocks, c.scale, c.k_scale, c.v_scale, c.workspace,
        c.workspace_bytes, 0, s);
  return paged_decode_attention_store(c.out, c.lse, c.q, c.k_new, c.v_new, stride, stride,
                                      c.slot_mapping, c.k_cache, c.v_cache, c.block_tables,
                                      c.max_blocks_per_seq, c.context_lens, B, c.Hq, c.Hkv,
                                      c.D, c.block_size, c.num_blocks, c.scale, c.workspace,
                                      c.workspace_bytes, 0, s);
}

// Launch parameters of the pad node; args[] points at the four argument values.
void pad_params(cudaKernelNodeParams* kp, void* func, void** args, int32_t** lens,
                int32_t** slots, int* from, int* to) {
  std::memset(kp, 0, sizeof(*kp));
  args[0] = lens;
  args[1] = slots;
  args[2] = from;
  args[3] = to;
  kp->func = func;
  kp->gridDim = dim3(1);
  kp->blockDim = dim3(kPadThreads);
  kp->sharedMemBytes = 0;
  kp->kernelParams = args;
  kp->extra = nullptr;
}

}  // namespace

struct pkv_decode_graphs {
  pkv_decode_graphs_config cfg{};
  std::vector<int32_t> sizes;
  std::vector<Bucket> buckets;
  cudaStream_t stream = nullptr;
};

namespace {

void release(pkv_decode_graphs* r) {
  if (!r) return;
  if (r->stream) cudaStreamSynchronize(r->stream);
  for (Bucket& b : r->buckets) {
    if (b.exec) cudaGraphExecDestroy(b.exec);
    if (b.graph) cudaGraphDestroy(b.graph);
    if (b.full_exec) cudaGraphExecDestroy(b.full_exec);
    if (b.full_graph) cudaGraphDestroy(b.full_graph);
  }
  if (r->stream) cudaStreamDestroy(r->stream);
  delete r;
}

// The runner's bucket sizes for a configuration (empty when it is invalid).
std::vector<int32_t> bucket_sizes(const pkv_decode_graphs_config& c) {
  std::vector<int32_t> v;
  if (c.num_buckets == 0) {
    const int n = pkv_decode_graphs_default_buckets(c.max_batch, nullptr, 0);
    if (n <= 0) return v;
    v.resize(n);
    pkv_decode_graphs_default_buckets(c.max_batch, v.data(), n);
    return v;
  }
  if (c.num_buckets < 0 || c.num_buckets > PKV_GRAPHS_MAX_BUCKETS ||
      !valid_list(c.buckets, c.num_buckets) || c.buckets[c.num_buckets - 1] > c.max_batch)
    return v;
  v.assign(c.buckets, c.buckets + c.num_buckets);
  return v;
}

int check_config(const pkv_decode_graphs_config* c) {
  if (!c) return PKV_ERR_ARG;
  if (c->max_batch < 1 || c->max_blocks_per_seq < 1 || c->num_blocks < 1) return PKV_ERR_ARG;
  if (!c->k_cache || !c->v_cache || !c->q || !c->k_new || !c->v_new || !c->slot_mapping ||
      !c->block_tables || !c->context_lens || !c->out)
    return PKV_ERR_ARG;
  if (c->kv_fp8 != 0 && c->kv_fp8 != 1) return PKV_ERR_ARG;
  if (bucket_sizes(*c).empty()) return PKV_ERR_ARG;
  // shapes are checked by the step itself (the workspace query returns 0 for
  // shapes it rejects, so check those here first)
  if (paged_decode_num_splits(1, c->Hq, c->Hkv, c->D, c->max_blocks_per_seq, c->block_size, 0) <
      1)
    return PKV_ERR_SHAPE;
  return PKV_OK;
}

size_t need_bytes(const pkv_decode_graphs_config& c, const std::vector<int32_t>& sizes) {
  size_t need = paged_decode_workspace_bytes(c.max_batch, c.Hq, c.Hkv, c.D,
                                             c.max_blocks_per_seq, c.block_size, 0);
  for (int32_t b : sizes)
    need = std::max(need, paged_decode_workspace_bytes(b, c.Hq, c.Hkv, c.D,
                                                       c.max_blocks_per_seq, c.block_size, 0));
  return need;
}

}  // namespace

extern "C" size_t pkv_decode_graphs_config_bytes(void) { return sizeof(pkv_decode_graphs_config); }

extern "C" int pkv_decode_graphs_default_buckets(int max_batch, int32_t* out, int capacity) {
  if (max_batch < 1 || capacity < 0 || (capacity > 0 && !out)) return PKV_ERR_ARG;
  int n = 0;
  for (int b = 1; b <= PKV_GRAPHS_DEFAULT_MAX_BUCKET && b <= max_batch; b *= 2) {
    if (n < capacity) out[n] = b;
    ++n;
  }
  return n;
}

extern "C" int pkv_decode_graphs_pick_bucket(const int32_t* buckets, int n, int B) {
  if (B < 0 || !valid_list(buckets, n)) return PKV_ERR_ARG;
  if (B == 0 || B > buckets[n - 1]) return 0;
  return *std::lower_bound(buckets, buckets + n, B);
}

extern "C" size_t pkv_decode_graphs_workspace_bytes(const pkv_decode_graphs_config* config) {
  if (check_config(config) != PKV_OK) return 0;
  return need_bytes(*config, bucket_sizes(*config));
}

extern "C" int pkv_decode_graphs_create(const pkv_decode_graphs_config* config,
                                        pkv_decode_graphs** runner) {
  if (!runner) return PKV_ERR_ARG;
  *runner = nullptr;
  int rc = check_config(config);
  if (rc != PKV_OK) return rc;
  const pkv_decode_graphs_config& c = *config;
  const std::vector<int32_t> sizes = bucket_sizes(c);
  const size_t need = need_bytes(c, sizes);
  if (need > 0 && (!c.workspace || c.workspace_bytes < need ||
                   reinterpret_cast<uintptr_t>(c.workspace) % 256 != 0))
    return PKV_ERR_WORKSPACE;

  pkv_decode_graphs* r = new (std::nothrow) pkv_decode_graphs;
  if (!r) return PKV_ERR_LAUNCH;
  r->cfg = c;
  r->cfg.buckets = nullptr;   // the runner keeps its own copy
  r->cfg.num_buckets = static_cast<int>(sizes.size());
  r->sizes = sizes;
  r->buckets.resize(sizes.size());
  auto fail = [&](int status) {
    release(r);
    return status;
  };
  if (cudaStreamCreateWithFlags(&r->stream, cudaStreamNonBlocking) != cudaSuccess)
    return fail(PKV_ERR_LAUNCH);
  cudaStream_t s = r->stream;

  // every row empty, counters clear
  decode_graph_pad_kernel<<<1, kPadThreads, 0, s>>>(c.context_lens, c.slot_mapping, 0,
                                                    c.max_batch);
  if (cudaGetLastError() != cudaSuccess) return fail(PKV_ERR_LAUNCH);
  if (need > 0 &&
      cudaMemsetAsync(c.workspace, 0, std::min(need, kCounterBytes), s) != cudaSuccess)
    return fail(PKV_ERR_LAUNCH);

  for (size_t i = 0; i < sizes.size(); ++i) {
    Bucket& bk = r->buckets[i];
    bk.size = sizes[i];
    bk.pad_from = bk.size;
    // once eagerly over empty rows: loads the kernel this bucket's plan picks
    rc = step(c, bk.size, s);
    if (rc != PKV_OK) return fail(rc);
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(PKV_ERR_LAUNCH);
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return fail(PKV_ERR_LAUNCH);
    decode_graph_pad_kernel<<<1, kPadThreads, 0, s>>>(c.context_lens, c.slot_mapping,
                                                      bk.size, bk.size);
    const bool launched = cudaGetLastError() == cudaSuccess;
    rc = launched ? step(c, bk.size, s) : PKV_ERR_LAUNCH;
    cudaGraph_t graph = nullptr;
    const cudaError_t end = cudaStreamEndCapture(s, &graph);
    bk.graph = graph;
    if (rc != PKV_OK) return fail(rc);
    if (end != cudaSuccess || !graph) return fail(PKV_ERR_LAUNCH);
    // the pad kernel is the graph's only root
    size_t n_roots = 0;
    if (cudaGraphGetRootNodes(graph, nullptr, &n_roots) != cudaSuccess || n_roots != 1)
      return fail(PKV_ERR_LAUNCH);
    cudaGraphNode_t root = nullptr;
    cudaGraphNodeType type;
    if (cudaGraphGetRootNodes(graph, &root, &n_roots) != cudaSuccess ||
        cudaGraphNodeGetType(root, &type) != cudaSuccess || type != cudaGraphNodeTypeKernel)
      return fail(PKV_ERR_LAUNCH);
    cudaKernelNodeParams kp;
    if (cudaGraphKernelNodeGetParams(root, &kp) != cudaSuccess || kp.gridDim.x != 1 ||
        kp.blockDim.x != kPadThreads)
      return fail(PKV_ERR_LAUNCH);
    bk.pad = root;
    bk.pad_func = kp.func;
    if (cudaGraphInstantiate(&bk.exec, graph, 0) != cudaSuccess) {
      bk.exec = nullptr;
      return fail(PKV_ERR_LAUNCH);
    }
    // a batch that fills the bucket needs no padding: the step alone
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return fail(PKV_ERR_LAUNCH);
    rc = step(c, bk.size, s);
    cudaGraph_t full = nullptr;
    const cudaError_t end_full = cudaStreamEndCapture(s, &full);
    bk.full_graph = full;
    if (rc != PKV_OK) return fail(rc);
    if (end_full != cudaSuccess || !full) return fail(PKV_ERR_LAUNCH);
    if (cudaGraphInstantiate(&bk.full_exec, full, 0) != cudaSuccess) {
      bk.full_exec = nullptr;
      return fail(PKV_ERR_LAUNCH);
    }
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return fail(PKV_ERR_LAUNCH);
  *runner = r;
  return PKV_OK;
}

extern "C" int pkv_decode_graphs_buckets(const pkv_decode_graphs* runner, int32_t* out,
                                         int capacity) {
  if (!runner || capacity < 0 || (capacity > 0 && !out)) return PKV_ERR_ARG;
  const int n = static_cast<int>(runner->sizes.size());
  for (int i = 0; i < n && i < capacity; ++i) out[i] = runner->sizes[i];
  return n;
}

extern "C" int pkv_decode_graphs_run(pkv_decode_graphs* runner, int B, pkv_stream_t stream) {
  if (!runner || B < 0 || B > runner->cfg.max_batch) return PKV_ERR_ARG;
  if (B == 0) return PKV_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int size = pkv_decode_graphs_pick_bucket(runner->sizes.data(),
                                                 static_cast<int>(runner->sizes.size()), B);
  if (size < 0) return PKV_ERR_ARG;
  if (size == 0) return step(runner->cfg, B, s);   // above the largest bucket: eager
  Bucket& bk = *std::find_if(runner->buckets.begin(), runner->buckets.end(),
                             [&](const Bucket& b) { return b.size == size; });
  if (B == bk.size) return cudaGraphLaunch(bk.full_exec, s) == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
  if (bk.pad_from != B) {
    // the replays already queued keep their own arguments
    cudaKernelNodeParams kp;
    void* args[4];
    int32_t* lens = runner->cfg.context_lens;
    int32_t* slots = runner->cfg.slot_mapping;
    int from = B, to = bk.size;
    pad_params(&kp, bk.pad_func, args, &lens, &slots, &from, &to);
    if (cudaGraphExecKernelNodeSetParams(bk.exec, bk.pad, &kp) != cudaSuccess)
      return PKV_ERR_LAUNCH;
    bk.pad_from = B;
  }
  return cudaGraphLaunch(bk.exec, s) == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

extern "C" void pkv_decode_graphs_destroy(pkv_decode_graphs* runner) { release(runner); }
