// pkv_internal.h — host-side declarations shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// Bits of the device error word (see pkv_get_device_error()).
constexpr unsigned kErrIndex = 1u;    // slot / block id / length out of range
constexpr unsigned kErrTimeout = 2u;  // a bounded wait ran out

// Head dimension and block size that the kernels are built for.
constexpr int kHeadDim = 128;
constexpr int kBlockSize = 256;

// SM count of the current device (cached per device); 0 on failure.
int device_sm_count();

// Address of the device error word on the current device; nullptr on failure.
unsigned* device_error_word();

// Tensor map over one pool tensor viewed as [slots, Hkv, D] (D innermost),
// box = {64 elements of D, box_heads heads, box_rows slots}, 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* base, int64_t num_slots, int Hkv,
                     int box_rows, int box_heads = 1);
// The same for an FP8 pool [slots, Hkv, 128] of bytes: a box is one 128-byte
// row (all 128 dims) of one kv head x box_rows consecutive slots.
bool encode_pool_map_u8(CUtensorMap* map, const void* base, int64_t num_slots, int Hkv,
                        int box_rows);

struct StoreArgs {
  const void* k;
  const void* v;
  int64_t k_tok_stride;
  int64_t v_tok_stride;
  void* k_cache;
  void* v_cache;
  const int32_t* slot_mapping;
  int64_t T;
  int row_elems;  // Hkv * D
  int64_t num_slots;
};
int launch_store(const StoreArgs& a, unsigned* err, cudaStream_t stream);
// FP8 (E4M3) pool: k_inv / v_inv are 1/scale rounded to fp32.
int launch_store_fp8(const StoreArgs& a, float k_inv, float v_inv, unsigned* err,
                     cudaStream_t stream);
int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                       int n_pairs, int64_t block_bytes, int64_t num_blocks, unsigned* err,
                       cudaStream_t stream);

struct DecodeArgs {
  void* out;
  float* lse;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int B, Hq, Hkv;
  int64_t num_blocks;
  float scale;
  void* workspace;
  size_t workspace_bytes;
  int num_splits;  // as requested (0 = automatic)
  int prefix_tokens;  // shared prefix handled by a separate pass (0 = none)
  int q_len = 1;      // query positions per sequence (several: speculative verify)
  int fp8 = 0;        // pools hold E4M3 codes: element = code value * k_scale / v_scale
  float k_scale = 1.f, v_scale = 1.f;
  // Fused store: before attending, the new token of sequence b
  // (rows of k_new / v_new, token stride in elements) goes to new_slots[b]
  // (-1 = none; otherwise the slot of position context_lens[b] - 1).
  const int32_t* new_slots = nullptr;
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  int64_t k_new_stride = 0, v_new_stride = 0;
  // block_tables and context_lens were written before the stream's previous
  // kernel (PKV_DECODE_METADATA_READY): blocks may read them before waiting
  // for that kernel
  int metadata_ready = 0;
};

// Argument checks of a single-query decode call (pointers, alignment, pool
// shape, head grouping); PKV_OK or the status the call returns.  Launches
// nothing.
int check_decode_args(const DecodeArgs& a, int D, int block_size);

// Split plan of one decode call.
struct DecodePlan {
  int heads_per_cta;  // G: query heads per kv head that one thread block serves
  int head_groups;    // (Hq/Hkv) / G
  int split_tokens;   // tokens per split: whole blocks, or whole 64-token tiles
  int num_splits;     // S
  int consumer_groups;  // 2: bf16 single-token decode with two consumer groups per block
  size_t prefix_offset;  // byte offset of the shared-prefix partials (if any)
  int prefix_splits;     // key ranges of the shared-prefix pass
  int prefix_kt_per;     // 128-key tiles per range
  size_t workspace_bytes;
};
// Returns PKV_OK and fills `plan`, or a negative status.  prefix_blocks: blocks
// of a shared prefix reduced separately (the splits cover the rest).
int plan_decode(int B, int Hq, int Hkv, int max_blocks_per_seq, int num_splits,
                int sm_count, int prefix_blocks, DecodePlan* plan);

// Attention of every (sequence, query head) of the batch over a shared prefix
// of prefix_tokens tokens (the first blocks of sequence 0's table), as one
// normalised fp32 partial [B*Hq, 128] plus log2-sum-exp [B*Hq] per row.
struct PrefixArgs {
  float* part_o;
  float* part_lse;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int B, Hq, Hkv;
  int prefix_tokens;
  int splits;   // key ranges; partials are [B*Hq, splits, 128] and [B*Hq, splits]
  int kt_per;   // 128-key tiles per range
  int64_t num_blocks;
  float scale;
};
int launch_prefix_attention(const PrefixArgs& a, unsigned* err, cudaStream_t stream);
// (sequence, head) rows per query tile of the shared-prefix pass for a group of
// g query heads per kv head (whole tokens per tile), or 0 if g is unsupported.
int prefix_rows_per_tile(int g);
int launch_decode(const DecodeArgs& a, const DecodePlan& plan, unsigned* err,
                  cudaStream_t stream);

struct PrefillArgs {
  void* out;
  float* lse;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int B, max_seqlen_q, max_seqlen_k, Hq, Hkv;
  int64_t num_blocks;
  float scale;
};
int launch_prefill(const PrefillArgs& a, unsigned* err, cudaStream_t stream);

// q_len new positions per sequence (speculative verify) on the tensor-core
// kernel: one item per (sequence, kv head) holding its g*q_len (position, head)
// rows; needs g*q_len <= 128 (verify_rows_fit).  q [B, q_len, Hq, 128],
// out like q, lse [B, q_len, Hq] natural log or null.
struct VerifyArgs {
  void* out;
  float* lse;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int B, q_len, Hq, Hkv;
  int64_t num_blocks;
  float scale;
};
int verify_rows_fit(int g, int q_len);

// Test hook of the decode / prefill kernels' bounded waits (see
// pkv_testing_set_wait_fault); 0, 0 turns it off.
int set_wait_hook_decode(unsigned long long limit_ns, int withhold_plus1);
int set_wait_hook_prefill(unsigned long long limit_ns, int withhold_plus1);
int launch_verify(const VerifyArgs& a, unsigned* err, cudaStream_t stream);

}  // namespace pkv
