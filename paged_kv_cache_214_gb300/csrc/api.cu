// api.cu — the C ABI entry points declared in include/pkv.h: argument checks,
// per-device state (SM count, the device error word), TMA tensor-map encoding
// and dispatch to the kernels.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;
// Longest wait limit the test hook accepts (the kernels' own limit).
constexpr unsigned long long kWaitLimitTestMaxNs = 2000000000ull;

// The one piece of state the library keeps: a sticky error word per device,
// or-ed by kernels and read-and-cleared by pkv_get_device_error().
__device__ unsigned g_device_error;

std::mutex g_mu;
int g_sm_count[kMaxDevices];
unsigned* g_err_ptr[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

unsigned* device_error_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}

// The driver's tensor-map encoder, looked up once.
bool encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return true;
}

bool encode_pool_map(CUtensorMap* map, const void* base, int64_t num_slots, int Hkv,
                     int box_rows, int box_heads) {
  if (!encoder()) return false;
  // [slots, Hkv, D] with D innermost; a box is 64 dims (128 B, the swizzle
  // span) x box_heads heads x box_rows consecutive slots.
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(num_slots)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                 static_cast<cuuint64_t>(Hkv) * kHeadDim * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_pool_map_u8(CUtensorMap* map, const void* base, int64_t num_slots, int Hkv,
                        int box_rows) {
  if (!encoder()) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(num_slots)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim),
                                 static_cast<cuuint64_t>(Hkv) * kHeadDim};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 1,
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

int check_pool(int Hkv, int D, int block_size, int64_t num_blocks) {
  if (Hkv <= 0 || D <= 0 || block_size <= 0 || num_blocks < 0) return PKV_ERR_ARG;
  if (D != kHeadDim || block_size != kBlockSize) return PKV_ERR_SHAPE;
  // TMA coordinates are 32-bit: every slot index must fit.
  if (num_blocks * kBlockSize > INT32_MAX) return PKV_ERR_SHAPE;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int kv_cache_store(const void* k, const void* v, int64_t k_tok_stride,
                              int64_t v_tok_stride, void* k_cache, void* v_cache,
                              const int32_t* slot_mapping, int64_t T, int Hkv, int D,
                              int block_size, int64_t num_blocks, pkv_stream_t stream) {
  if (T < 0) return PKV_ERR_ARG;
  int st = check_pool(Hkv, D, block_size, num_blocks);
  if (st) return st;
  if (T == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_ARG;
  const int64_t row = static_cast<int64_t>(Hkv) * D;
  if (k_tok_stride < row || v_tok_stride < row) return PKV_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ARG;
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  StoreArgs a{k, v, k_tok_stride, v_tok_stride, k_cache, v_cache, slot_mapping, T,
              static_cast<int>(row), num_blocks * block_size};
  return launch_store(a, err, reinterpret_cast<cudaStream_t>(stream));
}

namespace {
bool valid_scale(float s) { return std::isfinite(s) && s > 0.f; }
}  // namespace

extern "C" int kv_cache_store_fp8(const void* k, const void* v, int64_t k_tok_stride,
                                  int64_t v_tok_stride, void* k_cache, void* v_cache,
                                  const int32_t* slot_mapping, int64_t T, int Hkv, int D,
                                  int block_size, int64_t num_blocks, float k_scale,
                                  float v_scale, pkv_stream_t stream) {
  if (T < 0 || !valid_scale(k_scale) || !valid_scale(v_scale)) return PKV_ERR_ARG;
  int st = check_pool(Hkv, D, block_size, num_blocks);
  if (st) return st;
  if (T == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_ARG;
  const int64_t row = static_cast<int64_t>(Hkv) * D;
  if (k_tok_stride < row || v_tok_stride < row) return PKV_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ARG;
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  StoreArgs a{k, v, k_tok_stride, v_tok_stride, k_cache, v_cache, slot_mapping, T,
              static_cast<int>(row), num_blocks * block_size};
  // the quantizer multiplies by the binary32 reciprocal of each scale
  const float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;
  return launch_store_fp8(a, k_inv, v_inv, err, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int kv_cache_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_blocks,
                                    const int32_t* dst_blocks, int n_pairs, int Hkv, int D,
                                    int block_size, int64_t num_blocks, pkv_stream_t stream) {
  if (n_pairs < 0) return PKV_ERR_ARG;
  int st = check_pool(Hkv, D, block_size, num_blocks);
  if (st) return st;
  if (n_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PKV_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ARG;
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  const int64_t block_bytes = static_cast<int64_t>(block_size) * Hkv * D * 2;
  return launch_copy_blocks(k_cache, v_cache, src_blocks, dst_blocks, n_pairs, block_bytes,
                            num_blocks, err, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t paged_decode_workspace_bytes(int B, int Hq, int Hkv, int D,
                                               int max_blocks_per_seq, int block_size,
                                               int num_splits) {
  if (D != kHeadDim || block_size != kBlockSize || num_splits < 0) return 0;
  DecodePlan plan;
  if (plan_decode(B, Hq, Hkv, max_blocks_per_seq, num_splits, device_sm_count(), 0, &plan))
    return 0;
  return plan.workspace_bytes;
}

extern "C" int paged_decode_num_splits(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                       int block_size, int num_splits) {
  if (D != kHeadDim || block_size != kBlockSize) return PKV_ERR_SHAPE;
  if (num_splits < 0) return PKV_ERR_ARG;
  DecodePlan plan;
  const int st = plan_decode(B, Hq, Hkv, max_blocks_per_seq, num_splits, device_sm_count(), 0, &plan);
  return st ? st : plan.num_splits;
}




namespace {

// The step's new rows for the fused store (see paged_decode_attention_store).
struct NewRows {
  const void* k;
  const void* v;
  int64_t k_stride, v_stride;  // elements
  const int32_t* slots;
};

}  // namespace

int pkv::check_decode_args(const DecodeArgs& a, int D, int block_size) {
  if (a.B < 0 || a.Hq <= 0 || a.max_blocks_per_seq < 0 || a.num_splits < 0) return PKV_ERR_ARG;
  if (a.fp8 && (!valid_scale(a.k_scale) || !valid_scale(a.v_scale))) return PKV_ERR_ARG;
  int st = check_pool(a.Hkv, D, block_size, a.num_blocks);
  if (st) return st;
  if (a.Hq % a.Hkv) return PKV_ERR_SHAPE;
  if (a.B == 0) return PKV_OK;
  if (!a.out || !a.q || !a.k_cache || !a.v_cache || !a.context_lens) return PKV_ERR_ARG;
  if (a.max_blocks_per_seq > 0 && !a.block_tables) return PKV_ERR_ARG;
  if (a.num_blocks == 0 && a.max_blocks_per_seq > 0) return PKV_ERR_ARG;
  if (!aligned16(a.out) || !aligned16(a.q) || !aligned16(a.k_cache) || !aligned16(a.v_cache))
    return PKV_ERR_ARG;
  return PKV_OK;
}

namespace {

// Checks, plan and launch shared by the single-query decode entry points:
// bf16 or E4M3 pools (a.fp8), with or without the fused store (rows).
int decode_entry(DecodeArgs a, int D, int block_size, const NewRows* rows,
                 pkv_stream_t stream) {
  int st = check_decode_args(a, D, block_size);
  if (st || a.B == 0) return st;
  if (rows && (!rows->k || !rows->v || !rows->slots)) return PKV_ERR_ARG;
  if (rows) {
    // new-token rows are read 16 bytes at a time
    if (!aligned16(rows->k) || !aligned16(rows->v)) return PKV_ERR_ARG;
    const int64_t row = static_cast<int64_t>(a.Hkv) * D;
    if (rows->k_stride < row || rows->v_stride < row || rows->k_stride % 8 ||
        rows->v_stride % 8)
      return PKV_ERR_ARG;
    a.new_slots = rows->slots;
    a.k_new = rows->k;
    a.v_new = rows->v;
    a.k_new_stride = rows->k_stride;
    a.v_new_stride = rows->v_stride;
  }
  DecodePlan plan;
  st = plan_decode(a.B, a.Hq, a.Hkv, a.max_blocks_per_seq, a.num_splits, device_sm_count(), 0,
                   &plan);
  if (st) return st;
  if (plan.workspace_bytes) {
    if (!a.workspace || a.workspace_bytes < plan.workspace_bytes ||
        (reinterpret_cast<uintptr_t>(a.workspace) & 255u))
      return PKV_ERR_WORKSPACE;
  }
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  return launch_decode(a, plan, err, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" int paged_decode_attention(void* out, float* lse, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens, int B,
                                      int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      int num_splits, pkv_stream_t stream) {
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits, 0};
  return decode_entry(a, D, block_size, nullptr, stream);
}

extern "C" int paged_decode_attention_flags(void* out, float* lse, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, int max_blocks_per_seq,
                                            const int32_t* context_lens, int B, int Hq, int Hkv,
                                            int D, int block_size, int64_t num_blocks,
                                            float scale, void* workspace,
                                            size_t workspace_bytes, int num_splits,
                                            unsigned flags, pkv_stream_t stream) {
  if (flags & ~static_cast<unsigned>(PKV_DECODE_METADATA_READY)) return PKV_ERR_ARG;
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits, 0};
  a.metadata_ready = (flags & PKV_DECODE_METADATA_READY) ? 1 : 0;
  return decode_entry(a, D, block_size, nullptr, stream);
}

extern "C" int paged_decode_attention_store(
    void* out, float* lse, const void* q, const void* k_new, const void* v_new,
    int64_t k_tok_stride, int64_t v_tok_stride, const int32_t* slot_mapping, void* k_cache,
    void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int B, int Hq, int Hkv, int D, int block_size,
    int64_t num_blocks, float scale, void* workspace, size_t workspace_bytes, int num_splits,
    pkv_stream_t stream) {
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits, 0};
  const NewRows rows{k_new, v_new, k_tok_stride, v_tok_stride, slot_mapping};
  return decode_entry(a, D, block_size, &rows, stream);
}

extern "C" int paged_decode_attention_fp8(void* out, float* lse, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int B, int Hq, int Hkv,
                                          int D, int block_size, int64_t num_blocks, float scale,
                                          float k_scale, float v_scale, void* workspace,
                                          size_t workspace_bytes, int num_splits,
                                          pkv_stream_t stream) {
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits, 0, 1,
               1, k_scale, v_scale};
  return decode_entry(a, D, block_size, nullptr, stream);
}

extern "C" int paged_decode_attention_fp8_store(
    void* out, float* lse, const void* q, const void* k_new, const void* v_new,
    int64_t k_tok_stride, int64_t v_tok_stride, const int32_t* slot_mapping, void* k_cache,
    void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int B, int Hq, int Hkv, int D, int block_size,
    int64_t num_blocks, float scale, float k_scale, float v_scale, void* workspace,
    size_t workspace_bytes, int num_splits, pkv_stream_t stream) {
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits, 0, 1,
               1, k_scale, v_scale};
  const NewRows rows{k_new, v_new, k_tok_stride, v_tok_stride, slot_mapping};
  return decode_entry(a, D, block_size, &rows, stream);
}

// Longest run of query positions per sequence the multi-query decode accepts.
constexpr int kMaxQueryLen = 64;

// Multi-query decode on the tensor-core kernel (one item per (sequence, kv
// head), all g*q_len rows in one tile) when there are more rows per kv head
// than one split-K decode block serves (8: it then reads K/V once too, and
// measured faster), the rows fit one tile and there are at least as many
// items as SMs; otherwise (up to 8 rows, small batches, or a split count the
// caller asks for) on the split-K decode kernel.
bool use_verify_kernel(int B, int q_len, int Hq, int Hkv, int num_splits) {
  if (num_splits != 0 || q_len < 2 || !verify_rows_fit(Hq / Hkv, q_len)) return false;
  if ((Hq / Hkv) * q_len <= 8) return false;
  return static_cast<int64_t>(B) * Hkv >= device_sm_count();
}

extern "C" size_t paged_decode_multiquery_workspace_bytes(int B, int q_len, int Hq, int Hkv,
                                                          int D, int max_blocks_per_seq,
                                                          int block_size, int num_splits) {
  if (D != kHeadDim || block_size != kBlockSize || num_splits < 0) return 0;
  if (q_len < 1 || q_len > kMaxQueryLen) return 0;
  if (Hkv > 0 && Hq % Hkv == 0 && use_verify_kernel(B, q_len, Hq, Hkv, num_splits)) return 0;
  DecodePlan plan;
  if (plan_decode(B, Hq * q_len, Hkv, max_blocks_per_seq, num_splits, device_sm_count(), 0,
                  &plan))
    return 0;
  return plan.workspace_bytes;
}

extern "C" int paged_decode_attention_multiquery(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int B,
    int q_len, int Hq, int Hkv, int D, int block_size, int64_t num_blocks, float scale,
    void* workspace, size_t workspace_bytes, int num_splits, pkv_stream_t stream) {
  if (B < 0 || Hq <= 0 || max_blocks_per_seq < 0 || num_splits < 0) return PKV_ERR_ARG;
  if (q_len < 1 || q_len > kMaxQueryLen) return PKV_ERR_ARG;
  int st = check_pool(Hkv, D, block_size, num_blocks);
  if (st) return st;
  if (Hq % Hkv) return PKV_ERR_SHAPE;
  if (B == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !context_lens) return PKV_ERR_ARG;
  if (max_blocks_per_seq > 0 && !block_tables) return PKV_ERR_ARG;
  if (num_blocks == 0 && max_blocks_per_seq > 0) return PKV_ERR_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ARG;
  if (use_verify_kernel(B, q_len, Hq, Hkv, num_splits)) {
    unsigned* err = device_error_word();
    if (!err) return PKV_ERR_LAUNCH;
    VerifyArgs va{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                  context_lens, B, q_len, Hq, Hkv, num_blocks, scale};
    return launch_verify(va, err, reinterpret_cast<cudaStream_t>(stream));
  }
  DecodePlan plan;
  st = plan_decode(B, Hq * q_len, Hkv, max_blocks_per_seq, num_splits, device_sm_count(), 0,
                   &plan);
  if (st) return st;
  if (plan.workspace_bytes) {
    if (!workspace || workspace_bytes < plan.workspace_bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return PKV_ERR_WORKSPACE;
  }
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits, 0, q_len};
  return launch_decode(a, plan, err, reinterpret_cast<cudaStream_t>(stream));
}


namespace {

int check_shared_prefix(int max_blocks_per_seq, int shared_prefix_tokens) {
  if (shared_prefix_tokens < 0 || shared_prefix_tokens % kBlockSize) return PKV_ERR_ARG;
  if (shared_prefix_tokens / kBlockSize > max_blocks_per_seq) return PKV_ERR_ARG;
  return PKV_OK;
}

}  // namespace

extern "C" size_t paged_decode_shared_prefix_workspace_bytes(int B, int Hq, int Hkv, int D,
                                                             int max_blocks_per_seq,
                                                             int block_size,
                                                             int shared_prefix_tokens,
                                                             int num_splits) {
  if (D != kHeadDim || block_size != kBlockSize || num_splits < 0) return 0;
  if (check_shared_prefix(max_blocks_per_seq, shared_prefix_tokens)) return 0;
  DecodePlan plan;
  if (plan_decode(B, Hq, Hkv, max_blocks_per_seq, num_splits, device_sm_count(),
                  shared_prefix_tokens / kBlockSize, &plan))
    return 0;
  return plan.workspace_bytes;
}

extern "C" int paged_decode_attention_shared_prefix(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int B,
    int Hq, int Hkv, int D, int block_size, int64_t num_blocks, float scale,
    int shared_prefix_tokens, void* workspace, size_t workspace_bytes, int num_splits,
    pkv_stream_t stream) {
  int st = check_shared_prefix(max_blocks_per_seq, shared_prefix_tokens);
  if (st) return st;
  if (shared_prefix_tokens == 0)
    return paged_decode_attention(out, lse, q, k_cache, v_cache, block_tables,
                                  max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size,
                                  num_blocks, scale, workspace, workspace_bytes, num_splits,
                                  stream);
  if (B < 0 || Hq <= 0 || max_blocks_per_seq < 0 || num_splits < 0) return PKV_ERR_ARG;
  st = check_pool(Hkv, D, block_size, num_blocks);
  if (st) return st;
  if (Hq % Hkv) return PKV_ERR_SHAPE;
  if (B == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !context_lens || !block_tables) return PKV_ERR_ARG;
  if (num_blocks == 0) return PKV_ERR_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ARG;
  DecodePlan plan;
  st = plan_decode(B, Hq, Hkv, max_blocks_per_seq, num_splits, device_sm_count(),
                   shared_prefix_tokens / kBlockSize, &plan);
  if (st) return st;
  if (!workspace || workspace_bytes < plan.workspace_bytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_WORKSPACE;
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* pbase = static_cast<uint8_t*>(workspace) + plan.prefix_offset;
  const size_t o_bytes =
      (static_cast<size_t>(B) * Hq * plan.prefix_splits * kHeadDim * sizeof(float) + 255) /
      256 * 256;
  PrefixArgs pa{reinterpret_cast<float*>(pbase), reinterpret_cast<float*>(pbase + o_bytes), q,
                k_cache, v_cache, block_tables, B, Hq, Hkv, shared_prefix_tokens,
                plan.prefix_splits, plan.prefix_kt_per, num_blocks, scale};
  st = launch_prefix_attention(pa, err, cs);
  if (st) return st;
  DecodeArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
               B, Hq, Hkv, num_blocks, scale, workspace, workspace_bytes, num_splits,
               shared_prefix_tokens};
  return launch_decode(a, plan, err, cs);
}

extern "C" int paged_prefill_attention(void* out, float* lse, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                       const int32_t* cu_seqlens_k, int B, int max_seqlen_q,
                                       int max_seqlen_k, int Hq, int Hkv, int D, int block_size,
                                       int64_t num_blocks, float scale, pkv_stream_t stream) {
  if (B < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || Hq <= 0 || max_blocks_per_seq < 0)
    return PKV_ERR_ARG;
  int st = check_pool(Hkv, D, block_size, num_blocks);
  if (st) return st;
  if (Hq % Hkv) return PKV_ERR_SHAPE;
  if (B == 0 || max_seqlen_q == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k) return PKV_ERR_ARG;
  if (max_blocks_per_seq > 0 && !block_tables) return PKV_ERR_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ARG;
  if (static_cast<int64_t>(max_seqlen_k) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PKV_ERR_ARG;
  unsigned* err = device_error_word();
  if (!err) return PKV_ERR_LAUNCH;
  PrefillArgs a{out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_seqlens_q,
                cu_seqlens_k, B, max_seqlen_q, max_seqlen_k, Hq, Hkv, num_blocks, scale};
  return launch_prefill(a, err, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int pkv_get_device_error(pkv_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_LAUNCH;
  unsigned* p = device_error_word();
  if (!p) return PKV_ERR_LAUNCH;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_LAUNCH;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return PKV_ERR_LAUNCH;
  }
  if (v & kErrIndex) return PKV_ERR_DEVICE_INDEX;
  if (v & kErrTimeout) return PKV_ERR_TIMEOUT;
  return PKV_OK;
}

extern "C" int pkv_testing_set_wait_fault(int64_t wait_limit_ns, int withhold_tile) {
  if (wait_limit_ns < 0 || withhold_tile < -1 || (withhold_tile >= 0 && wait_limit_ns == 0) ||
      wait_limit_ns > static_cast<int64_t>(kWaitLimitTestMaxNs))
    return PKV_ERR_ARG;
  const unsigned long long lim = static_cast<unsigned long long>(wait_limit_ns);
  const int w = withhold_tile + 1;
  int st = set_wait_hook_decode(lim, w);
  if (st == PKV_OK) st = set_wait_hook_prefill(lim, w);
  return st;
}

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_ARG: return "PKV_ERR_ARG: invalid argument";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: unsupported shape";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing, small or misaligned";
    case PKV_ERR_LAUNCH: return "PKV_ERR_LAUNCH: CUDA runtime or launch failure";
    case PKV_ERR_DEVICE_INDEX: return "PKV_ERR_DEVICE_INDEX: index out of range on the device";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT: a device wait ran out";
    default: return "unknown pkv status";
  }
}
