/* pkv_blocks.h — host-side block manager for the paged KV cache.
 *
 * "Nano-vLLM System Architecture Analysis", §2 Core Components, "Paged KV
 * Cache": the cache is split into fixed-size blocks of 256 tokens, and a
 * BlockManager keeps a free list of blocks, a hash table from content hash to
 * block id for prefix caching (sharing common prefixes), and reference counts
 * for block sharing with copy-on-write semantics.  §3 "Lifecycle of a Request":
 * prepare_inputs() builds the block tables and slot mappings the attention
 * kernels read.  This is that manager, in C++ on the host; it produces the
 * block_tables / slot_mapping inputs of include/pkv.h and never touches device
 * memory.  The one device-side consequence of copy-on-write, copying a block's
 * K/V to a fresh block, is kv_cache_copy_blocks() in pkv.h.
 *
 * Behaviour
 *   - Blocks are handed out from a free list in FIFO order; a block whose
 *     reference count drops to zero goes to the back of the list and keeps its
 *     content hash, so a later request with the same content can take it back
 *     (a prefix-cache hit) until it is handed out for other content.
 *   - Only full blocks are hashed.  The hash of block i of a sequence chains
 *     the hash of block i-1 with the block's token ids (a 64-bit mix written
 *     for this library; the pages use xxhash, any well-mixed 64-bit hash
 *     serves), and a hit also compares the stored token ids, so a hash
 *     collision never shares wrong content.
 *   - pkv_bm_fork gives a child sequence the parent's blocks (all shared);
 *     appending to a shared, partly filled last block first moves the
 *     appender to a new block and reports the (source, destination) pair that
 *     must be copied on the device before the token's K/V is stored.
 *   - Every function returns PKV_BM_OK or a negative error; no function
 *     aborts.  A manager is not thread-safe; use one per scheduler thread.
 */
#ifndef PKV_BLOCKS_H_
#define PKV_BLOCKS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

enum {
  PKV_BM_OK = 0,
  PKV_BM_ERR_ARG = -1,        /* bad argument (null, negative, block_size < 1)  */
  PKV_BM_ERR_NO_BLOCKS = -2,  /* not enough free blocks; nothing was changed    */
  PKV_BM_ERR_NO_SEQ = -3,     /* unknown sequence id                             */
  PKV_BM_ERR_EXISTS = -4,     /* sequence id already in use                      */
  PKV_BM_ERR_SMALL = -5       /* output array too small                          */
};

/* A manager for a pool of num_blocks blocks of block_size tokens.  NULL on a
 * bad argument or allocation failure. */
pkv_block_manager* pkv_bm_create(int64_t num_blocks, int block_size);
void pkv_bm_destroy(pkv_block_manager* bm);

int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm);

/* Admit a new sequence with its prompt (n_tokens token ids).  Full blocks whose
 * content is already cached are shared (reference count + 1); the rest are
 * taken from the free list.  *num_cached_tokens receives how many leading
 * prompt tokens already have K/V in the pool (a multiple of block_size), so
 * prefill only needs to compute the rest.  All-or-nothing: on
 * PKV_BM_ERR_NO_BLOCKS nothing changes. */
int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                        int64_t n_tokens, int64_t* num_cached_tokens);

/* Append one token (a decode step).  *slot receives the slot its K/V goes to.
 * If the sequence's last block was shared and partly filled, the sequence first
 * moves to a new block: *copy_src / *copy_dst receive the blocks whose K/V must
 * be copied (kv_cache_copy_blocks) before the store; otherwise both are -1. */
int pkv_bm_append_token(pkv_block_manager* bm, int64_t seq_id, int32_t token,
                        int64_t* slot, int32_t* copy_src, int32_t* copy_dst);

/* A child sequence that shares every block of the parent (for example a
 * second sample of the same prompt). */
int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Release a sequence: every block's reference count drops by one; blocks that
 * reach zero go back to the free list with their content hash kept. */
int pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);

/* Number of tokens / blocks of a sequence (negative error if unknown). */
int64_t pkv_bm_num_tokens(const pkv_block_manager* bm, int64_t seq_id);
int64_t pkv_bm_num_blocks(const pkv_block_manager* bm, int64_t seq_id);

/* The sequence's block table: out[0..n) = its physical block ids in logical
 * order, out[n..max_blocks) = -1. */
int pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* out,
                       int64_t max_blocks);

/* Slots of logical positions [begin, end) of a sequence (end <= its length):
 * block_id * block_size + position % block_size. */
int pkv_bm_slot_mapping(const pkv_block_manager* bm, int64_t seq_id, int64_t begin,
                        int64_t end, int32_t* out);

/* Reference count of a physical block (0 if free), or a negative error. */
int64_t pkv_bm_ref_count(const pkv_block_manager* bm, int64_t block_id);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCKS_H_ */
