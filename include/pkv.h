/* pkv.h — C ABI of the paged KV-cache attention library (GB300, sm_103a).
 *
 * Three operations make up the data-parallel hot path of attention over a paged
 * KV cache, as "Nano-vLLM System Architecture Analysis" describes it (§2 Core
 * Components, "Paged KV Cache" and "Attention with Paged Cache"):
 *
 *   kv_cache_store           write new K/V rows into the block pool via slot_mapping
 *   paged_decode_attention   one query row per (sequence, head) over the whole
 *                            cached context, read through block_tables
 *   paged_prefill_attention  causal (chunked) prefill: new query rows over a
 *                            cached prefix plus the new tokens, all read through
 *                            block_tables
 *
 * and, built on them:
 *   paged_decode_attention_flags      the decode with option bits (tables and
 *                                     lengths ready before the previous kernel)
 *   paged_decode_attention_store      a decode step's store and decode in one
 *                                     launch
 *   paged_decode_attention_shared_prefix  decode with a prefix that every
 *                                     sequence shares attended once per kv head
 *   paged_decode_attention_multiquery several new positions per sequence (the
 *                                     verify step of speculative decoding)
 *   kv_cache_store_fp8, paged_decode_attention_fp8(_store)  the same over E4M3
 *                                     (FP8) pools
 *   kv_cache_copy_blocks              copy-on-write block copies
 *   paged_decode_attention_noalloc    decode without a caller workspace
 *   pkv_testing_set_wait_fault        tests only: make a bounded wait run out
 * (the host block manager is declared in pkv_blocks.h).
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them.  Sizes are element counts.
 *   - Data type: K/V/Q/out are bf16 (IEEE binary16-brain, passed as void*),
 *     indices are int32, lse is fp32.  Byte offsets are computed in 64 bits.
 *   - The block pool k_cache / v_cache is one contiguous array per tensor with
 *     layout [num_blocks, block_size, Hkv, D]; a "slot" is
 *     block_id * block_size + offset and addresses one [Hkv, D] row.
 *   - Supported: D == 128, block_size == 256, Hq % Hkv == 0, Hkv >= 1.
 *     Anything else returns PKV_ERR_SHAPE.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream), does
 *     no host synchronisation and no allocation, and returns a status for
 *     errors it can see on the host.  Errors found by a kernel (a slot or block
 *     id out of range, a context longer than its block table, a bounded wait
 *     that ran out) never trap: the kernel skips the bad access, records the
 *     error in the device error word and finishes; read it with
 *     pkv_get_device_error().
 *   - Outputs for rows whose inputs were invalid are unspecified.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t; /* same type as cudaStream_t */

typedef enum {
  PKV_OK = 0,
  PKV_ERR_ARG = -1,          /* null pointer, negative size, misaligned pointer  */
  PKV_ERR_SHAPE = -2,        /* unsupported D / block_size / head counts          */
  PKV_ERR_WORKSPACE = -3,    /* workspace missing, too small or misaligned        */
  PKV_ERR_LAUNCH = -4,       /* a CUDA runtime call or kernel launch failed       */
  PKV_ERR_DEVICE_INDEX = -5, /* device: slot/block id out of range, ctx > table   */
  PKV_ERR_TIMEOUT = -6       /* device: a bounded wait ran out                    */
} pkv_status;

/* kv_cache_store — "Stores computed K/V entries into the paged cache via
 * slot_mapping" (Nano-vLLM System Architecture Analysis, §2 Core Components,
 * "Attention with Paged Cache"; blocks of 256 tokens per "Paged KV Cache").
 *
 * For every token t in [0, T) with s = slot_mapping[t]:
 *   s <  0                        : padding, nothing is written;
 *   0 <= s < num_blocks*block_size: k_cache[s, :, :] = k[t, :, :] and
 *                                   v_cache[s, :, :] = v[t, :, :] (bit copy);
 *   s >= num_blocks*block_size    : skipped, device error PKV_ERR_DEVICE_INDEX.
 * k, v         : bf16 rows [T, Hkv, D]; row t starts at k + t*k_tok_stride
 *                elements (the [Hkv, D] part of a row is contiguous).  Rows
 *                whose start is 16-byte aligned are moved in 16-byte vectors,
 *                others element by element.
 * k_cache/v_cache : pool [num_blocks, block_size, Hkv, D], 16-byte aligned.
 * slot_mapping : int32 [T] on the device.
 * Two tokens with the same non-negative slot: which one lands is unspecified.
 * Returns PKV_OK, PKV_ERR_ARG (null pointer with T > 0, T < 0, stride smaller
 * than Hkv*D, misaligned pool), PKV_ERR_SHAPE or PKV_ERR_LAUNCH.  T == 0 is a
 * no-op. */
int kv_cache_store(const void* k, const void* v, int64_t k_tok_stride,
                   int64_t v_tok_stride, void* k_cache, void* v_cache,
                   const int32_t* slot_mapping, int64_t T, int Hkv, int D,
                   int block_size, int64_t num_blocks, pkv_stream_t stream);

/* kv_cache_copy_blocks — the device half of copy-on-write block sharing
 * ("reference counting for block sharing (copy-on-write semantics)", Nano-vLLM
 * System Architecture Analysis, §2 Core Components, "Paged KV Cache"): for
 * i in [0, n_pairs), block dst_blocks[i] of k_cache and of v_cache becomes a
 * bit copy of block src_blocks[i] (whole blocks: block_size x Hkv x D).  The
 * host block manager (pkv_blocks.h) reports these pairs when a sequence
 * appends to a shared, partly filled block.
 * src_blocks, dst_blocks: int32 [n_pairs] on the device.  Destination blocks
 * must be distinct and must not be any pair's source; otherwise the result is
 * unspecified.  A block id outside [0, num_blocks) skips that pair and is
 * reported as PKV_ERR_DEVICE_INDEX through pkv_get_device_error().
 * Returns PKV_OK, PKV_ERR_ARG, PKV_ERR_SHAPE or PKV_ERR_LAUNCH; n_pairs == 0 is
 * a no-op. */
int kv_cache_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_blocks,
                         const int32_t* dst_blocks, int n_pairs, int Hkv, int D,
                         int block_size, int64_t num_blocks, pkv_stream_t stream);

/* paged_decode_workspace_bytes — bytes of device workspace that a
 * paged_decode_attention call with the same (B, Hq, Hkv, D, max_blocks_per_seq,
 * block_size, num_splits) needs.  0 means the call needs none (a single split).
 * Returns 0 as well for arguments the decode call would reject. */
size_t paged_decode_workspace_bytes(int B, int Hq, int Hkv, int D,
                                    int max_blocks_per_seq, int block_size,
                                    int num_splits);

/* paged_decode_num_splits — the number of context splits a decode call with
 * these arguments uses (num_splits == 0 picks it from the SM count of the
 * current device).  Returns a value >= 1, or a negative pkv_status. */
int paged_decode_num_splits(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                            int block_size, int num_splits);

/* paged_decode_attention — decode attention over the paged cache: "During
 * decode, gathers all cached K/V from paged blocks before calling
 * scaled_dot_product_attention" (Nano-vLLM System Architecture Analysis, §2
 * Core Components, "Attention with Paged Cache"); GQA per §6 "Architecture
 * Support".  The library reads the blocks in place instead of gathering them.
 *
 * For sequence b with L = context_lens[b] (the token stored this step
 * included) and query head h, with kv head kh = h / (Hq/Hkv):
 *   key/value j (0 <= j < L) is row kh of slot
 *       block_tables[b*max_blocks_per_seq + j/block_size]*block_size + j%block_size,
 *   s_j  = scale * <q[b,h,:], K_j>,
 *   out[b,h,:] = sum_j softmax(s)_j * V_j       (bf16, round to nearest even),
 *   lse[b,h]   = ln(sum_j exp(s_j))             (fp32; may be NULL).
 * L == 0 gives out = 0 and lse = -inf.  No mask: the query is the last
 * position of its sequence.
 * q   : bf16 [B, Hq, D] contiguous.   out : bf16 [B, Hq, D] contiguous.
 * block_tables : int32 [B, max_blocks_per_seq]; only entries < ceil(L/bs) are
 *                read.  context_lens : int32 [B].  Both on the device.
 * Accumulation is fp32.  The context is cut into num_splits ranges of whole
 * blocks (0 = automatic; a requested count is raised when a range would
 * exceed 32 blocks, and paged_decode_num_splits() reports the count used);
 * each range is reduced by its own thread block, and the last one to finish
 * merges the partial results by log-sum-exp.
 * workspace : device memory of at least paged_decode_workspace_bytes(...)
 *   bytes, 256-byte aligned; may be NULL when that size is 0.  Its first
 *   1 MiB holds one arrival counter per (sequence, kv head group), at the same
 *   place for every call shape; the rest holds the partial results.  That
 *   first MiB must be zero before the first call that uses a given workspace
 *   (e.g. cudaMemsetAsync once after allocating it); every call leaves it zero
 *   again, so one workspace can serve calls of any shape.  Calls that share a
 *   workspace must not overlap in time (same stream, or ordered by events).
 * Returns PKV_OK, PKV_ERR_ARG, PKV_ERR_SHAPE, PKV_ERR_WORKSPACE or
 * PKV_ERR_LAUNCH.  A context longer than max_blocks_per_seq*block_size or a
 * block id outside [0, num_blocks) is reported as PKV_ERR_DEVICE_INDEX through
 * pkv_get_device_error() (that read is clamped or skipped, never performed). */
int paged_decode_attention(void* out, float* lse, const void* q,
                           const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int B, int Hq, int Hkv,
                           int D, int block_size, int64_t num_blocks, float scale,
                           void* workspace, size_t workspace_bytes,
                           int num_splits, pkv_stream_t stream);

/* paged_decode_attention_flags — paged_decode_attention with option bits.
 * PKV_DECODE_METADATA_READY: the caller states that block_tables and
 * context_lens were written before the previous kernel on `stream` started,
 * and that no kernel still running writes them (for example they came from
 * host copies at the start of the step, and the previous kernel produced q).
 * The decode's blocks may then read them while that kernel finishes, before
 * they wait for it; everything else (q, the pools, out, lse, the workspace)
 * is still touched only after the wait.  Results are bit-identical to
 * paged_decode_attention; if the statement is false they are undefined.
 * Other bits: PKV_ERR_ARG.  Everything else as paged_decode_attention. */
#define PKV_DECODE_METADATA_READY 1u
int paged_decode_attention_flags(void* out, float* lse, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens, int B,
                                 int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 int num_splits, unsigned flags, pkv_stream_t stream);

/* paged_decode_attention_store — kv_cache_store of the step's new tokens and
 * paged_decode_attention over the updated cache in one launch, the way the
 * attention layer stores K/V through slot_mapping and then attends
 * (Nano-vLLM System Architecture Analysis, §2 Core Components, "Attention
 * with Paged Cache").  Results equal kv_cache_store(k_new, v_new, ...,
 * slot_mapping) followed by paged_decode_attention(...) with the same
 * arguments, under one more rule: slot_mapping[b] is -1 (nothing stored) or
 * the slot of sequence b's last position, context_lens[b] - 1, through its
 * block table.  Any other slot is not written and is reported as
 * PKV_ERR_DEVICE_INDEX through pkv_get_device_error().  The blocks that
 * attend over a sequence's last range write its new row, one kv head each,
 * before they read that range; no other block reads that position, so no
 * block waits for another.
 * k_new, v_new : bf16 [B, Hkv, D] rows, token strides k_tok_stride /
 *   v_tok_stride in elements (multiples of 8, >= Hkv*D), 16-byte aligned.
 * slot_mapping : int32 [B] on the device.  Pools are written; everything else
 * (layouts, workspace = paged_decode_workspace_bytes of the same shapes,
 * results, errors) as paged_decode_attention. */
int paged_decode_attention_store(void* out, float* lse, const void* q, const void* k_new,
                                 const void* v_new, int64_t k_tok_stride, int64_t v_tok_stride,
                                 const int32_t* slot_mapping, void* k_cache, void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                                 int block_size, int64_t num_blocks, float scale,
                                 void* workspace, size_t workspace_bytes, int num_splits,
                                 pkv_stream_t stream);

/* paged_decode_shared_prefix_workspace_bytes — workspace bytes that a
 * paged_decode_attention_shared_prefix call with the same arguments needs
 * (0 for arguments that call would reject). */
size_t paged_decode_shared_prefix_workspace_bytes(int B, int Hq, int Hkv, int D,
                                                  int max_blocks_per_seq, int block_size,
                                                  int shared_prefix_tokens, int num_splits);

/* paged_decode_attention_shared_prefix — decode attention for a batch whose
 * sequences all begin with the same prefix, held once in the pool: "a hash
 * table from content hash -> block ID for prefix caching (sharing common
 * prefixes)" with "reference counting for block sharing" (Nano-vLLM System
 * Architecture Analysis, §2 Core Components, "Paged KV Cache").
 *
 * Results are those of paged_decode_attention on the same arguments.  The
 * first shared_prefix_tokens tokens (a multiple of block_size, at most
 * max_blocks_per_seq*block_size) of every sequence must be the same physical
 * blocks: entries [0, shared_prefix_tokens/block_size) of every row of
 * block_tables equal those of row 0, and every context_lens[b] >=
 * shared_prefix_tokens.  The call computes attention over those shared keys
 * once for all B*Hq query rows, as a dense tcgen05 tile product per kv head
 * (query rows = the group's (sequence, head) pairs), then runs the split decode
 * over each sequence's own tokens [shared_prefix_tokens, ctx) and folds the
 * shared part into the log-sum-exp merge.  The shared blocks are read once per
 * kv head instead of once per sequence.
 * workspace: at least paged_decode_shared_prefix_workspace_bytes(...) bytes,
 * with the conventions of paged_decode_attention (first MiB zero before first
 * use; left zero by every call).  Two kernels run on `stream`.
 * shared_prefix_tokens == 0 is exactly paged_decode_attention.  A table row
 * whose prefix entries differ from row 0's, or a context shorter than the
 * prefix, is reported as PKV_ERR_DEVICE_INDEX through pkv_get_device_error().
 * Returns PKV_OK, PKV_ERR_ARG (also for a prefix that is not whole blocks or
 * is longer than the tables), PKV_ERR_SHAPE, PKV_ERR_WORKSPACE or
 * PKV_ERR_LAUNCH. */
int paged_decode_attention_shared_prefix(void* out, float* lse, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables,
                                         int max_blocks_per_seq,
                                         const int32_t* context_lens, int B, int Hq,
                                         int Hkv, int D, int block_size, int64_t num_blocks,
                                         float scale, int shared_prefix_tokens,
                                         void* workspace, size_t workspace_bytes,
                                         int num_splits, pkv_stream_t stream);

/* Size of the fixed device scratch array behind
 * paged_decode_attention_noalloc (16 MiB per device that loads the library). */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* paged_decode_attention_noalloc — the same decode attention as
 * paged_decode_attention, for callers that cannot allocate device memory and so
 * cannot provide its workspace: for example a plugin whose host framework owns
 * every device allocation and passes the library only its input and output
 * tensors, or a runtime with a fixed memory plan in which no call may
 * allocate.  The source pages have no counterpart to this call; it exists only
 * for such callers.
 *
 * Arguments, layouts, results and errors are those of paged_decode_attention
 * without the workspace arguments.  The split partials and arrival counters
 * live in a scratch array inside the library, PKV_NOALLOC_SCRATCH_BYTES long,
 * which every GPU that loads the library holds until the process exits.  The
 * call allocates nothing: it uses no cudaMalloc, cudaFree or allocating
 * library routine.
 *   - A call whose partials would not fit in that array (see
 *     paged_decode_workspace_bytes: it must be <= PKV_NOALLOC_SCRATCH_BYTES)
 *     returns PKV_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address once
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture starts on that device.  The cached address belongs to
 *     the device's context at that time: after cudaDeviceReset on a device,
 *     do not call this entry point on that device again in the same process.
 *   - Argument checks run before anything is queued: a call refused with any
 *     status launches nothing and queues nothing on `stream`.
 *   - Every call on a device uses the same array, which keeps the previous
 *     call's contents; each call clears its own arrival counters (an async
 *     memset on `stream`) before its kernel.  Calls whose work overlaps on the
 *     GPU (different streams not ordered by events, or several host threads)
 *     race on the array and give wrong results: order them. */
int paged_decode_attention_noalloc(void* out, float* lse, const void* q,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int B, int Hq, int Hkv,
                                   int D, int block_size, int64_t num_blocks, float scale,
                                   int num_splits, pkv_stream_t stream);

/* paged_decode_attention_multiquery — decode attention for q_len new tokens
 * per sequence at once: the check of a speculator's proposed tokens in
 * speculative decoding, which turns sequential decode into a parallel
 * "mini-prefill" ("What Is an Inference Engine, Anyway?", Technical details,
 * Speculative Decoding).  Same operation as paged_prefill_attention with
 * Lq = q_len and Lk = context_lens[b] for every sequence.  With
 * num_splits = 0, g*q_len <= 128 (g = Hq/Hkv) and at least one (sequence, kv
 * head) pair per SM, it runs on the tensor cores with all g*q_len (position,
 * head) rows of a kv head in one tile, so each kv head's K/V are read once and
 * no workspace is used (the size query returns 0); otherwise on the split-K
 * decode kernel over g*q_len rows per kv head.
 * q   : bf16 [B, q_len, Hq, D] contiguous.   out : bf16 [B, q_len, Hq, D].
 * lse : f32 [B, q_len, Hq] (natural log) or NULL.
 * context_lens[b] counts every cached token of sequence b, its q_len new ones
 * included (they must already be stored); position i (0 <= i < q_len) sees
 * keys j < context_lens[b] - q_len + 1 + i.
 * 1 <= q_len <= 64.  Other arguments, the workspace rules (size from
 * paged_decode_multiquery_workspace_bytes) and the errors are those of
 * paged_decode_attention; context_lens[b] < q_len is reported as
 * PKV_ERR_DEVICE_INDEX through pkv_get_device_error().  q_len = 1 is exactly
 * paged_decode_attention. */
size_t paged_decode_multiquery_workspace_bytes(int B, int q_len, int Hq, int Hkv, int D,
                                               int max_blocks_per_seq, int block_size,
                                               int num_splits);
int paged_decode_attention_multiquery(void* out, float* lse, const void* q,
                                      const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int B, int q_len, int Hq,
                                      int Hkv, int D, int block_size, int64_t num_blocks,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      int num_splits, pkv_stream_t stream);

/* FP8 KV cache.  The pages name quantized KV only as "compressed transfers"
 * ("Why Understand Inference Engine Architecture?", Tensor Parallelism
 * Optimization); the format here is this library's choice: OCP FP8 E4M3 (1
 * sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals, no infinity,
 * largest finite 448), one byte per element, with one scale per tensor.  A pool
 * is bytes [num_blocks, block_size, Hkv, D], 16-byte aligned; an element's
 * value is code value * scale.
 *
 * kv_cache_store_fp8 — kv_cache_store into FP8 pools: element x of k (v) is
 * stored as the E4M3 code nearest to fp32(x * fp32(1 / k_scale)) (v_scale for
 * v), ties to the even code, magnitudes past 448 saturated to 448.  Slot rules,
 * layouts of k / v and errors as kv_cache_store; k_scale and v_scale must be
 * finite and > 0 (else PKV_ERR_ARG).  Rows whose start is 16-byte aligned are
 * converted 16 elements at a time, others element by element. */
int kv_cache_store_fp8(const void* k, const void* v, int64_t k_tok_stride,
                       int64_t v_tok_stride, void* k_cache, void* v_cache,
                       const int32_t* slot_mapping, int64_t T, int Hkv, int D, int block_size,
                       int64_t num_blocks, float k_scale, float v_scale, pkv_stream_t stream);

/* paged_decode_attention_fp8 — paged_decode_attention over FP8 pools: key j is
 * code value * k_scale and value j is code value * v_scale.  Half the bytes of
 * the bf16 cache per token.  Arguments, workspace (paged_decode_workspace_bytes
 * of the same shapes), results and errors as paged_decode_attention; k_scale
 * and v_scale must be finite and > 0. */
int paged_decode_attention_fp8(void* out, float* lse, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens, int B,
                               int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                               float scale, float k_scale, float v_scale, void* workspace,
                               size_t workspace_bytes, int num_splits, pkv_stream_t stream);

/* paged_decode_attention_fp8_store — kv_cache_store_fp8 of the step's new
 * tokens and paged_decode_attention_fp8 over the updated pools in one launch,
 * as paged_decode_attention_store is for bf16 pools: the same slot rule
 * (slot_mapping[b] is -1 or the slot of position context_lens[b] - 1; any
 * other slot is reported and not written), the same quantization as
 * kv_cache_store_fp8, results bit-identical to the two calls.  Arguments as
 * paged_decode_attention_store plus k_scale, v_scale (finite, > 0). */
int paged_decode_attention_fp8_store(void* out, float* lse, const void* q, const void* k_new,
                                     const void* v_new, int64_t k_tok_stride,
                                     int64_t v_tok_stride, const int32_t* slot_mapping,
                                     void* k_cache, void* v_cache, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* context_lens, int B,
                                     int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                                     float scale, float k_scale, float v_scale, void* workspace,
                                     size_t workspace_bytes, int num_splits,
                                     pkv_stream_t stream);

/* paged_prefill_attention — causal prefill / chunked prefill with a prefix
 * cache: "During prefill with prefix cache, gathers cached K/V from the paged
 * cache and concatenates with newly computed ones" (Nano-vLLM System
 * Architecture Analysis, §2 Core Components, "Attention with Paged Cache");
 * chunked prefill per §2 "Scheduler".
 *
 * Sequence i has Lq = cu_seqlens_q[i+1]-cu_seqlens_q[i] new query rows and
 * Lk = cu_seqlens_k[i+1]-cu_seqlens_k[i] keys: its cached prefix (Lk-Lq tokens)
 * followed by the Lq new tokens.  The new tokens' K/V must already be in the
 * pool (kv_cache_store first): every key is read through block_tables, so the
 * "concatenation" is the block table itself.  Query row r (0 <= r < Lq) of
 * sequence i and head h sees keys j <= Lk - Lq + r (bottom-right causal):
 *   out[cu_seqlens_q[i]+r, h, :] = sum_j softmax(s)_j V_j,  s_j = scale <q, K_j>,
 *   lse[cu_seqlens_q[i]+r, h]    = ln(sum_j exp(s_j))  (may be NULL).
 * q   : bf16 [sum Lq, Hq, D] contiguous.   out : bf16 [sum Lq, Hq, D].
 * cu_seqlens_q / cu_seqlens_k : int32 [B+1], device.  max_seqlen_q bounds every
 * Lq (it sizes the grid) and max_seqlen_k every Lk.
 * QK^T and PV run on the tcgen05 tensor cores with bf16 operands and fp32
 * accumulation in tensor memory; the probabilities P are rounded to bf16 for
 * the PV product.
 * Returns PKV_OK, PKV_ERR_ARG (null pointers, negative sizes), PKV_ERR_SHAPE or
 * PKV_ERR_LAUNCH.  Lk < Lq, Lq > max_seqlen_q or Lk > max_seqlen_k, and
 * out-of-range block ids, are reported as PKV_ERR_DEVICE_INDEX through
 * pkv_get_device_error() and those rows are left unwritten. */
int paged_prefill_attention(void* out, float* lse, const void* q,
                            const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int B, int max_seqlen_q, int max_seqlen_k, int Hq,
                            int Hkv, int D, int block_size, int64_t num_blocks,
                            float scale, pkv_stream_t stream);

/* pkv_get_device_error — synchronises `stream`, then reads and clears the
 * device error word of the current device.  Returns PKV_OK, the first error
 * class recorded (PKV_ERR_DEVICE_INDEX before PKV_ERR_TIMEOUT), or
 * PKV_ERR_LAUNCH if the synchronisation itself failed. */
int pkv_get_device_error(pkv_stream_t stream);

/* pkv_status_string — static, human-readable name of a status code. */
const char* pkv_status_string(int status);

/* pkv_testing_set_wait_fault — FOR TESTS ONLY: exercises the bounded-wait
 * failure path of the kernels without faulting or hanging the GPU.  The pages
 * have no counterpart; every mbarrier wait of this library's kernels is
 * bounded (PKV_ERR_TIMEOUT, then the block waits for its own copies in flight,
 * frees its tensor memory and exits), and this call lets a test make such a
 * wait run out.
 *   wait_limit_ns > 0 : the kernels' wait limit becomes this many ns (at most
 *                       2e9, the built-in limit); 0 restores the built-in limit.
 *   withhold_tile >= 0: the K/V copy producers of paged_decode_attention (and
 *                       its fused / E4M3 / multi-query forms on the split-K
 *                       kernel) stop before that tile of each block's key range
 *                       (64-token tiles), and those of the tensor-core kernel
 *                       (prefill, shared-prefix pass, verify) before that
 *                       128-key tile of each block's running count, so that a
 *                       consumer's wait on it runs out while no copy is
 *                       outstanding on its barrier; -1: copy everything.  Needs
 *                       wait_limit_ns > 0.
 * The setting is per process, applies to every later launch on the current
 * device until changed, and is set synchronously (cudaMemcpyToSymbol).  Call
 * pkv_testing_set_wait_fault(0, -1) to turn it off.  Returns PKV_OK,
 * PKV_ERR_ARG or PKV_ERR_LAUNCH. */
int pkv_testing_set_wait_fault(int64_t wait_limit_ns, int withhold_tile);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
