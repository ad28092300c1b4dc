/* pkv_graphs.h — decode steps replayed from CUDA graphs captured per batch
 * size ("bucket").
 *
 * The pages' remedy for the host cost of launching a decode step: capture the
 * step once into a CUDA graph, then replay it ("Why Understand Inference
 * Engine Architecture?", Computational Acceleration, "CUDA Graph
 * Compilation"); graphs are captured ahead of time for a set of batch sizes and
 * a step runs the graph of the closest size that holds its batch, while
 * batches of more than 512 sequences run eagerly ("Nano-vLLM System
 * Architecture Analysis", §2 Core Components, "CUDA Graphs", and the
 * comparison table's "CUDA Graphs" and "Variable-batch CUDA Graphs" rows).
 *
 * A runner owns, for one pool and one set of shapes, one graph per bucket b of
 * the step "pad rows [B, b), then paged_decode_attention_store (or
 * paged_decode_attention_fp8_store) over rows [0, b)", and one of the step
 * alone for batches of exactly b.  Every graph reads the
 * same static input buffers and writes the same static outputs, which the
 * CALLER allocates once for max_batch rows and hands to the runner.  A step
 * of B sequences:
 *   1. the caller writes rows [0, B) of q, k_new, v_new, slot_mapping,
 *      block_tables and context_lens (rows at and past B may hold anything);
 *   2. pkv_decode_graphs_run(runner, B, stream);
 *   3. rows [0, B) of out and lse hold the results, once `stream` gets there.
 * Padding rows (B <= row < b) get context length 0 and slot -1 inside the
 * graph: they store nothing and their out / lse rows become 0 / -inf.  Rows
 * [0, B) of the results are bit-identical to those of
 * paged_decode_attention_store (or the E4M3 form) called over all b rows, the
 * padding rows included, with num_splits = 0; against a call over B rows they
 * differ only by the rounding of a different split count.
 *
 * The kernels read lengths, tables and slots from device memory, so one graph
 * serves every batch of up to b sequences of any context lengths up to
 * max_blocks_per_seq * block_size.
 *
 * Conventions are those of pkv.h: device pointers owned by the caller, status
 * codes from pkv_status, errors found by a kernel reported through
 * pkv_get_device_error().  Creating a runner captures and instantiates its
 * graphs (host memory for them, nothing on the device beyond what CUDA graph
 * instantiation itself takes); running one allocates nothing.
 */
#ifndef PKV_GRAPHS_H_
#define PKV_GRAPHS_H_

#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest bucket of the default set, and the most buckets a runner takes. */
#define PKV_GRAPHS_DEFAULT_MAX_BUCKET 512
#define PKV_GRAPHS_MAX_BUCKETS 64

typedef struct pkv_decode_graphs pkv_decode_graphs;

typedef struct {
  /* shapes, as for paged_decode_attention_store */
  int Hq, Hkv, D, block_size;
  int max_blocks_per_seq;   /* width of block_tables (every row) */
  int max_batch;            /* rows of every static buffer, >= 1 */
  int64_t num_blocks;       /* blocks in the pool */
  int kv_fp8;               /* 0: bf16 pools; 1: E4M3 pools (k_scale, v_scale) */
  float scale;              /* softmax scale */
  float k_scale, v_scale;   /* E4M3 pools only: finite, > 0 */
  /* buckets: host array of num_buckets strictly increasing sizes in
   * [1, max_batch], at most PKV_GRAPHS_MAX_BUCKETS; num_buckets = 0 takes the
   * default set (pkv_decode_graphs_default_buckets).  Batches larger than the
   * largest bucket (and at most max_batch) run eagerly. */
  int num_buckets;
  const int32_t* buckets;
  /* the pool: bf16 (or E4M3 bytes) [num_blocks, block_size, Hkv, D] */
  void* k_cache;
  void* v_cache;
  /* static inputs, max_batch rows each, contiguous:
   *   q bf16 [max_batch, Hq, D]; k_new, v_new bf16 [max_batch, Hkv, D];
   *   slot_mapping, context_lens int32 [max_batch];
   *   block_tables int32 [max_batch, max_blocks_per_seq] */
  void* q;
  void* k_new;
  void* v_new;
  int32_t* slot_mapping;
  int32_t* block_tables;
  int32_t* context_lens;
  /* static outputs: out bf16 [max_batch, Hq, D]; lse f32 [max_batch, Hq] (or
   * NULL) */
  void* out;
  float* lse;
  /* workspace: at least pkv_decode_graphs_workspace_bytes(config) bytes,
   * 256-byte aligned (NULL when that is 0); the runner clears its first MiB
   * when it is created and every step leaves it clear */
  void* workspace;
  size_t workspace_bytes;
} pkv_decode_graphs_config;

/* pkv_decode_graphs_config_bytes — sizeof(pkv_decode_graphs_config), for
 * bindings that lay the structure out themselves (natural C alignment, the
 * fields in the order above). */
size_t pkv_decode_graphs_config_bytes(void);

/* pkv_decode_graphs_default_buckets — the default bucket set: the sizes the
 * pages list, 1, 2, 4, 8, 16, 32, ..., 512 (read as the powers of two up to
 * 512), keeping those <= max_batch.  Writes at most `capacity` of them to
 * `out` (which may be NULL when capacity is 0) and returns how many there are,
 * or PKV_ERR_ARG for max_batch < 1 or capacity < 0.  Host only. */
int pkv_decode_graphs_default_buckets(int max_batch, int32_t* out, int capacity);

/* pkv_decode_graphs_pick_bucket — the bucket a batch of B sequences runs in:
 * the smallest of the n strictly increasing sizes that is >= B; 0 when B == 0
 * or B exceeds every size (no graph: the step runs eagerly, or not at all).
 * PKV_ERR_ARG for B < 0, n < 1, a NULL list or a list that is not strictly
 * increasing from >= 1.  Host only. */
int pkv_decode_graphs_pick_bucket(const int32_t* buckets, int n, int B);

/* pkv_decode_graphs_workspace_bytes — workspace bytes a runner with this
 * configuration needs (the most any of its buckets, or an eager step of up to
 * max_batch rows, needs); 0 for a configuration that needs none or that
 * pkv_decode_graphs_create would reject.  Host only (the split plan reads the
 * current device's SM count). */
size_t pkv_decode_graphs_workspace_bytes(const pkv_decode_graphs_config* config);

/* pkv_decode_graphs_create — check the configuration, clear context_lens
 * (to 0) and slot_mapping (to -1) in all max_batch rows and the workspace's
 * first MiB, then for each bucket run the step once eagerly over those empty
 * rows (which loads the kernels) and capture it into a graph, on a private
 * stream of the current device.  Synchronises that stream before returning.
 * The pool, the static buffers and the workspace must stay allocated until
 * pkv_decode_graphs_destroy.  Work queued on other streams that writes the
 * static buffers, the workspace or the pool must have finished before the
 * call (the private stream is not ordered after it), and no other work may
 * use them while it runs.  Stores the runner in *runner and returns
 * PKV_OK, or returns PKV_ERR_ARG / PKV_ERR_SHAPE / PKV_ERR_WORKSPACE (bad
 * configuration) or PKV_ERR_LAUNCH (a CUDA call failed) and stores NULL. */
int pkv_decode_graphs_create(const pkv_decode_graphs_config* config,
                             pkv_decode_graphs** runner);

/* pkv_decode_graphs_buckets — the runner's bucket sizes: writes at most
 * `capacity` of them to `out` and returns how many there are (PKV_ERR_ARG for
 * a NULL runner or capacity < 0). */
int pkv_decode_graphs_buckets(const pkv_decode_graphs* runner, int32_t* out, int capacity);

/* pkv_decode_graphs_run — one decode step of B sequences (0 <= B <=
 * max_batch) on `stream`: replays the graph of the smallest bucket >= B, or,
 * for B above the largest bucket, launches the same fused call eagerly over
 * rows [0, B).  B == 0 queues nothing.  Steps of one runner share its
 * buffers and workspace: order them (one stream, or events).  Returns PKV_OK,
 * PKV_ERR_ARG (NULL runner, B out of range) or PKV_ERR_LAUNCH. */
int pkv_decode_graphs_run(pkv_decode_graphs* runner, int B, pkv_stream_t stream);

/* pkv_decode_graphs_destroy — free the graphs and the private stream (waits for
 * the runner's own stream, not for steps queued on other streams: synchronise
 * those first).  NULL is ignored. */
void pkv_decode_graphs_destroy(pkv_decode_graphs* runner);

#ifdef __cplusplus
}
#endif

#endif /* PKV_GRAPHS_H_ */
