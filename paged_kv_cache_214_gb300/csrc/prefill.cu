// prefill.cu — paged causal prefill / chunked prefill attention on the sm_103a
// tensor cores (tcgen05, tensor memory, TMA).
//
// Operation: "During prefill with prefix cache, gathers cached K/V from the paged
// cache and concatenates with newly computed ones" (Nano-vLLM System
// Architecture Analysis, §2 Core Components, "Attention with Paged Cache");
// chunked prefill splits a long prompt across steps (§2 "Scheduler").  The new
// tokens are stored into the pool first, so every key is read through the block
// table and the "concatenation" is simply the table.  Query row r of a chunk of
// Lq rows over Lk keys sees keys j <= Lk - Lq + r.  Prefill is the compute-heavy
// phase (same page, "Differences", §3), so both products run on tensor cores.
// The same kernel computes the shared-prefix pass of a decode batch and the
// verify step of speculative decoding (see the modes below).
//
// Work item: one 128-row query tile (one sequence and query head) and its key
// tiles.  The kernel is persistent: one block per SM walks the items, heaviest
// first, so that set-up, the first loads and the output stores of one item
// overlap the next.  Twelve warps, each with one job:
//   warp 8  (TMA)  Q tiles and 128-key K tiles (two 64-dim boxes, 128-byte
//                  swizzle); a K tile never straddles a 256-token block.  The
//                  next item's Q loads right after its first K tile.
//   warp 9  (TMA)  V tiles.
//   warp 10 (MMA)  S_t = Q K_t^T into one of three S buffers in tensor memory.
//   warp 11 (MMA)  O += P_t V_t, A = P_t read from tensor memory, B = V_t
//                  MN-major straight from its TMA tile.
//   warps 0-7      softmax: warp w owns 16 whole rows of every S tile (half of
//                  its TMEM lane quarter, read with the 16-lane access shapes),
//                  keeps the running max in base 2, rescales O only when the
//                  max grew by more than 2^8 (weights below 256 are exact
//                  enough in fp32 / bf16), and writes P as bf16 pairs over the
//                  first 64 columns of the tile's S buffer.  No softmax warp
//                  waits for another, so the exp2 work of one overlaps the
//                  loads and reductions of the other on the same SM quarter.
// The MMAs come from two warps, each running its issue loop with all lanes and
// issuing through one elected lane (issuing from a lone lane-0 branch cost
// ~116 cycles per M=N=128 product, about half the tensor pipe).  S is
// triple-buffered, so the S of tile t+1 (and t+2) is computed while the
// softmax of tile t runs.
// TMEM (512 columns): S_0 | S_1 | S_2 | O.
// K and V each have three 32 KB stages (Q one buffer).  The tensor copies of
// one thread complete one after another, so every tile copy is split in its
// two 64-dim boxes issued by two lanes, and each ring stage has lanes of its
// own: a copy never waits behind the previous tile's.  An item's output is
// written while the next item's first tile is in flight.
// Every wait is bounded: a wait that runs out records an error, the block
// drains what it started, frees its tensor memory and exits.

#include <cuda_bf16.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kM = 128;   // query rows per tile
constexpr int kN = 128;   // keys per tile
constexpr int kSoftmaxWarps = 8;
constexpr int kQKWarp = 8;
constexpr int kVWarp = 9;
constexpr int kSWarp = 10;
constexpr int kPVWarp = 11;
constexpr int kThreads = 12 * 32;
constexpr int kHalf = 128 * 128;           // 128 rows x 64 bf16 (one 128-byte swizzled box)
constexpr int kTile = 2 * kHalf;           // 128 rows x 128 bf16
constexpr int kKStages = 3;
constexpr int kVStages = 3;
constexpr int kOffQ = 0;                              // one buffer
constexpr int kOffK = kOffQ + kTile;                  // kKStages stages
constexpr int kOffV = kOffK + kKStages * kTile;       // kVStages stages
constexpr int kOffBars = kOffV + kVStages * kTile;
constexpr int kSBufs = 3;
// barriers
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;
constexpr int kBarKFull = 2;    // [K stage]
constexpr int kBarKEmpty = 5;   // [K stage]
constexpr int kBarVFull = 8;    // [V stage]
constexpr int kBarVEmpty = 11;  // [V stage]
constexpr int kBarSFull = 14;   // [S buffer]
constexpr int kBarPFull = 17;   // [S buffer], 8 softmax warps
constexpr int kBarPVDone = 20;  // [S buffer]: the PV that read P from it has completed
constexpr int kBarOFull = 23;   // the last PV of an item has completed
constexpr int kBarDrainS = 24;
constexpr int kBarDrainPV = 25;
constexpr int kNumBars = 26;
static_assert(kKStages == 3 && kVStages == 3 && kSBufs == 3, "barrier layout");
constexpr int kOffTmem = kOffBars + kNumBars * 8;
constexpr int kOffFlags = kOffTmem + 8;
constexpr int kSmemBytes = kOffFlags + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "one block per SM must fit in shared memory");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // + 128 * buffer
constexpr uint32_t kColO = 384;
constexpr float kLazyRescale = 8.f;    // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint32_t kFull = 0xffffffffu;

// Kernel modes.  kCausal: (chunked) prefill, one item per (row tile, sequence,
// query head).  kPrefixPass: the shared-prefix pass of a decode batch.
// kVerify: q_len new positions per sequence (speculative verify), one item per
// (sequence, kv head) whose tile holds the g*q_len (position, head) rows.
constexpr int kCausal = 0;
constexpr int kPrefixPass = 1;
constexpr int kVerify = 2;

struct PrefillParams {
  __nv_bfloat16* out;
  float* lse;
  float* part_o;     // shared-prefix mode: [B*Hq, splits, 128] normalised partial
  float* part_lse;   // shared-prefix mode: [B*Hq, splits] log2-sum-exp
  int prefix_tokens; // shared-prefix mode: keys = the first prefix_tokens of table row 0
  int prefix_kt_per; // shared-prefix mode: key tiles per item
  int splits;        // shared-prefix mode: key ranges
  int rows_per_tile; // shared-prefix mode: (sequence, head) rows per query tile
  int n_rt;          // shared-prefix mode: query tiles per kv head
  int q_len;         // verify mode: query positions per sequence
  const int32_t* ctx;  // verify mode: keys per sequence
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* cu_q;
  const int32_t* cu_k;
  unsigned* err;
  int B, Hq, Hkv, maxblk, max_q, max_k;
  int n_qt;          // ceil(max_q / 128)
  int n_items;
  int64_t num_blocks;
  float scale_log2;
};

// One query tile and its keys.
struct Item {
  int n;          // key tiles (0: nothing to do)
  int kt0;        // first key tile
  int rows;       // valid query rows of the tile
  int diag;       // row i sees keys j <= diag + i
  int Lk;         // keys of the sequence
  int kvh;        // kv head
  int h;          // query head (causal mode)
  int q0;         // first query row of the tile (within the sequence, or the group's rows)
  int q_begin;    // row of q / out where the sequence starts (causal mode)
  int z;          // key range (shared-prefix mode)
  const int32_t* table;
};

template <int kMode>
__device__ __forceinline__ Item get_item(const PrefillParams& p, int idx, bool report) {
  Item it;
  const int g = p.Hq / p.Hkv;
  it.n = 0;
  it.h = 0;
  it.q_begin = 0;
  it.z = 0;
  if constexpr (kMode == kVerify) {
    // rows r = position r/g, head kvh*g + r%g of sequence b; row r sees keys
    // j <= Lk - q_len + r/g
    const int b = idx / p.Hkv;
    it.kvh = idx - b * p.Hkv;
    it.h = it.kvh * g;
    it.q_begin = b * p.q_len;
    it.q0 = 0;
    it.kt0 = 0;
    it.z = 0;
    it.table = p.block_tables + static_cast<int64_t>(b) * p.maxblk;
    const int Lk = p.ctx[b];
    it.Lk = Lk;
    it.rows = g * p.q_len;
    it.diag = Lk - p.q_len;
    if (Lk < p.q_len || static_cast<int64_t>(Lk) > static_cast<int64_t>(p.maxblk) * kBlockSize) {
      if (report) record_error(p.err, kErrIndex);
      it.rows = 0;
      return it;
    }
    it.n = (Lk + kN - 1) / kN;
  } else if constexpr (kMode == kPrefixPass) {
    const int grp = idx / p.n_rt;
    const int rt = idx - grp * p.n_rt;
    it.kvh = grp / p.splits;
    it.z = grp - it.kvh * p.splits;
    it.q0 = rt * p.rows_per_tile;
    it.rows = min(p.rows_per_tile, p.B * g - it.q0);
    it.kt0 = it.z * p.prefix_kt_per;
    const int n = min(p.prefix_kt_per, p.prefix_tokens / kN - it.kt0);
    it.n = (it.rows > 0 && n > 0) ? n : 0;
    it.diag = INT32_MAX / 2;   // no mask
    it.Lk = p.prefix_tokens;
    it.table = p.block_tables;
  } else {
    const int per_lvl = p.B * p.Hq;
    const int lvl = idx / per_lvl;             // heavier (later) row tiles first
    const int rem = idx - lvl * per_lvl;
    const int b = rem / p.Hq;
    it.h = rem - b * p.Hq;
    it.kvh = it.h / g;
    it.q_begin = p.cu_q[b];
    const int Lq = p.cu_q[b + 1] - it.q_begin;
    const int Lk = p.cu_k[b + 1] - p.cu_k[b];
    it.Lk = Lk;
    it.kt0 = 0;
    it.table = p.block_tables + static_cast<int64_t>(b) * p.maxblk;
    it.q0 = (p.n_qt - 1 - lvl) * kM;
    it.rows = 0;
    it.diag = 0;
    if (Lq < 0 || Lk < Lq || Lq > p.max_q || Lk > p.max_k ||
        static_cast<int64_t>(Lk) > static_cast<int64_t>(p.maxblk) * kBlockSize) {
      if (report) record_error(p.err, kErrIndex);
      return it;
    }
    it.rows = it.q0 < Lq ? min(kM, Lq - it.q0) : 0;
    it.diag = Lk - Lq + it.q0;
    it.n = it.rows > 0 ? (it.diag + it.rows - 1) / kN + 1 : 0;
  }
  return it;
}

// Item of round k for this block: rounds alternate direction so that every
// block gets a mix of heavy and light items.
__device__ __forceinline__ int item_index(int k) {
  const int c = (k & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                        : static_cast<int>(blockIdx.x);
  return k * static_cast<int>(gridDim.x) + c;
}

// First non-empty item at or after round k (k is advanced to it).
template <int kMode>
__device__ __forceinline__ bool next_item(const PrefillParams& p, int n_rounds, int& k, Item& it,
                                          bool report) {
  for (; k < n_rounds; ++k) {
    const int idx = item_index(k);
    if (idx >= p.n_items) continue;
    it = get_item<kMode>(p, idx, report);
    if (it.n > 0) return true;
  }
  return false;
}

// Wait with every lane of the warp; the result is the same for all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(kFull, mbar_wait(bar, parity));
}

// Running position in an N-slot ring: slot and phase parity.
template <int N>
struct Ring {
  int idx = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++idx == N) {
      idx = 0;
      ph ^= 1u;
    }
  }
};

// Block ids of a table row, 32 at a time across the lanes of a warp.
struct BlockIds {
  int chunk = -1;
  int mine = 0;
  // Block id of table entry blk; every lane of the warp calls this together.
  __device__ __forceinline__ int get(const int32_t* table, int limit, int blk, int lane,
                                     int64_t num_blocks, unsigned* err) {
    if ((blk >> 5) != chunk) {
      chunk = blk >> 5;
      const int bi = chunk * 32 + lane;
      mine = bi < limit ? __ldg(table + bi) : 0;
    }
    int id = __shfl_sync(kFull, mine, blk & 31);
    if (id < 0 || id >= num_blocks) {
      if (lane == 0) record_error(err, kErrIndex);
      id = 0;   // never form an out-of-range address
    }
    return id;
  }
};

// kCausal: causal (chunked) prefill over (row tile, sequence, query head) items.
// kPrefixPass: the shared-prefix pass of a decode batch.  For kv head kvh the
// query rows are the B*g (sequence, query head) pairs of its group (row r =
// sequence r/g, head kvh*g + r%g); every row sees all prefix_tokens keys of the
// blocks that open table row 0, split into key ranges; the output is a
// normalised fp32 partial and its log2-sum-exp per range, merged into the
// decode result afterwards.
// kVerify: for sequence b and kv head kvh the rows are the g*q_len (position,
// head) pairs (row r = position r/g, head kvh*g + r%g), read by one TMA box
// of g heads x q_len tokens; row r sees the keys a decode of position r/g
// would see.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + kOffBars;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffTmem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = p.Hq / p.Hkv;
  const int n_rounds = (p.n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  constexpr bool kPrefix = kMode == kPrefixPass;
  const int table_limit = kPrefix ? p.prefix_tokens / kBlockSize : p.maxblk;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i >= kBarPFull && i < kBarPFull + kSBufs) count = kSoftmaxWarps;
      mbar_init(bar(i), count);
    }
    flags[0] = 0;  // abort
    flags[1] = 0;  // K tiles issued
    flags[2] = 0;  // V tiles issued
    flags[3] = 0;  // Q tiles issued
    fence_barrier_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(sbase + kOffTmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kQKWarp && lane == 0) {
    tma_prefetch_map(&qmap);
    tma_prefetch_map(&kmap);
  }
  if (warp == kVWarp && lane == 0) tma_prefetch_map(&vmap);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kQKWarp) {
    // ------------------------------------------------------------ TMA: Q and K
    // An item's Q goes into the single Q buffer right after its first K tile
    // has been issued, once the S MMAs of the previous item are done with it.
    bool ok = true, stopped = false;
    int gi = 0, gk = 0;
    BlockIds ids;
    Ring<kKStages> rk;
    const int withhold = withheld_tile();   // test hook: K tiles from here on are never copied
    auto load_q = [&](const Item& it, int qi) -> bool {
      const uint32_t qdst = sbase + kOffQ;
      if (qi >= 1 && !warp_wait(bar(kBarQEmpty), (qi - 1) & 1)) return false;
      if (kMode == kCausal && it.rows < kM) {
        // ragged last tile of a sequence: gather its rows (zero-fill the rest)
        const __nv_bfloat16* base =
            p.q + (static_cast<int64_t>(it.q_begin + it.q0) * p.Hq + it.h) * kHeadDim;
        for (int e = lane; e < kM * 16; e += 32) {
          const int r = e >> 4, piece = e & 15;
          const bool valid = r < it.rows;
          const __nv_bfloat16* src =
              base + (valid ? static_cast<int64_t>(r) * p.Hq * kHeadDim + piece * 8 : 0);
          cp_async16(qdst + (piece >> 3) * kHalf + r * 128 + (((piece & 7) ^ (r & 7)) << 4), src,
                     valid ? 16u : 0u);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQFull));
      } else {
        if (lane == 0)
          mbar_arrive_expect_tx(bar(kBarQFull), kMode == kCausal ? kTile : p.rows_per_tile * 256);
        __syncwarp();
        if (lane >= 2 * kKStages && lane < 2 * kKStages + 2) {   // lanes of their own
          const int hf = lane & 1;
          if constexpr (kPrefix) {
            // (sequence, head) rows of the group: box {64 dims, g heads, tokens}
            tma_load_3d(qdst + hf * kHalf, &qmap, bar(kBarQFull), hf * 64, it.kvh * g, it.q0 / g);
          } else if constexpr (kMode == kVerify) {
            // (position, head) rows: box {64 dims, g heads, q_len tokens}
            tma_load_3d(qdst + hf * kHalf, &qmap, bar(kBarQFull), hf * 64, it.h, it.q_begin);
          } else {
            tma_load_3d(qdst + hf * kHalf, &qmap, bar(kBarQFull), hf * 64, it.h,
                        it.q_begin + it.q0);
          }
        }
      }
      if (lane == 0) flags[3] = qi + 1;
      __syncwarp();
      return true;
    };
    int k = 0;
    Item it;
    bool have = next_item<kMode>(p, n_rounds, k, it, false);
    while (have && ok) {
      int k2 = k + 1;
      Item nx;
      const bool have_next = next_item<kMode>(p, n_rounds, k2, nx, false);
      ids.chunk = -1;
      for (int kt = 0; kt < it.n; ++kt, ++gk, rk.next()) {
        if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
        if (gk >= withhold) { stopped = true; break; }
        const int gkt = it.kt0 + kt;
        const int id = ids.get(it.table, table_limit, gkt >> 1, lane, p.num_blocks, p.err);
        const int slot = id * kBlockSize + (gkt & 1) * kN;
        if (gk >= kKStages && !warp_wait(bar(kBarKEmpty + rk.idx), rk.ph ^ 1u)) {
          ok = false;
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(kBarKFull + rk.idx), kTile);
          flags[1] = gk + 1;
        }
        __syncwarp();
        // lanes 2s, 2s+1 load stage s: a lane's next copy never queues behind
        // its previous one
        if ((lane >> 1) == rk.idx)
          tma_load_3d(sbase + kOffK + rk.idx * kTile + (lane & 1) * kHalf, &kmap,
                      bar(kBarKFull + rk.idx), (lane & 1) * 64, it.kvh, slot);
        __syncwarp();
        if (kt == 0 && !load_q(it, gi)) {
          ok = false;
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
      }
      if (!ok || stopped) break;
      ++gi;
      it = nx;
      k = k2;
      have = have_next;
    }
    if (!ok && lane == 0) flags[0] = 1;
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ TMA: V
    bool ok = true;
    int gk = 0;
    BlockIds ids;
    Ring<kVStages> rv;
    int k = 0;
    Item it;
    bool have = next_item<kMode>(p, n_rounds, k, it, false);
    while (have && ok) {
      int k2 = k + 1;
      Item nx;
      const bool have_next = next_item<kMode>(p, n_rounds, k2, nx, false);
      ids.chunk = -1;
      for (int kt = 0; kt < it.n; ++kt, ++gk, rv.next()) {
        if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
        const int gkt = it.kt0 + kt;
        const int id = ids.get(it.table, table_limit, gkt >> 1, lane, p.num_blocks, p.err);
        const int slot = id * kBlockSize + (gkt & 1) * kN;
        if (gk >= kVStages && !warp_wait(bar(kBarVEmpty + rv.idx), rv.ph ^ 1u)) {
          ok = false;
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(kBarVFull + rv.idx), kTile);
          flags[2] = gk + 1;
        }
        __syncwarp();
        if ((lane >> 1) == rv.idx)
          tma_load_3d(sbase + kOffV + rv.idx * kTile + (lane & 1) * kHalf, &vmap,
                      bar(kBarVFull + rv.idx), (lane & 1) * 64, it.kvh, slot);
        __syncwarp();
      }
      it = nx;
      k = k2;
      have = have_next;
    }
    if (!ok && lane == 0) flags[0] = 1;
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ MMA: S = Q K^T
    // (the whole warp runs the loop and waits; an elected lane issues)
    {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kN, 0);   // B = K, K-major
      bool ok = true, timeout = false;
      int gi = 0, gk = 0;
      Ring<kSBufs> sb;
      Ring<kKStages> rk;
      int k = 0;
      Item it;
      bool have = next_item<kMode>(p, n_rounds, k, it, false);
      while (have && ok) {
        int k2 = k + 1;
        Item nx;
        const bool have_next = next_item<kMode>(p, n_rounds, k2, nx, false);
        if (!warp_wait(bar(kBarQFull), gi & 1)) { ok = false; timeout = true; break; }
        const uint32_t q_s = sbase + kOffQ;
        for (int kt = 0; kt < it.n; ++kt, ++gk, sb.next(), rk.next()) {
          if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
          if (!warp_wait(bar(kBarKFull + rk.idx), rk.ph)) { ok = false; timeout = true; break; }
          // S buffer free: the PV that read P from it (three tiles back) is done
          if (gk >= kSBufs && !warp_wait(bar(kBarPVDone + sb.idx), sb.ph ^ 1u)) {
            ok = false;
            timeout = true;
            break;
          }
          tc_fence_after();
          const uint32_t k_s = sbase + kOffK + rk.idx * kTile;
          const uint32_t d_s = tmem + kColS + sb.idx * kN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
            umma_bf16_warp(d_s, smem_desc_sw128(q_s + off, 16, 1024),
                           smem_desc_sw128(k_s + off, 16, 1024), idesc_s, ks > 0);
          }
          umma_commit_warp(bar(kBarSFull + sb.idx));
          umma_commit_warp(bar(kBarKEmpty + rk.idx));
        }
        if (!ok) break;
        umma_commit_warp(bar(kBarQEmpty));
        ++gi;
        it = nx;
        k = k2;
        have = have_next;
      }
      if (timeout && lane == 0) record_error(p.err, kErrTimeout);
      if (!ok && lane == 0) flags[0] = 1;
      // every MMA this warp issued has completed once this arrives
      umma_commit_warp(bar(kBarDrainS));
      (void)warp_wait(bar(kBarDrainS), 0);
    }
  } else if (warp == kPVWarp) {
    // ------------------------------------------------------------ MMA: O += P V
    {
      constexpr uint32_t idesc_o = idesc_bf16_f32(kM, kHeadDim, 1);  // B = V, MN-major
      bool ok = true, timeout = false;
      int gk = 0;
      Ring<kSBufs> sb;
      Ring<kVStages> rv;
      const uint32_t d_o = tmem + kColO;
      int k = 0;
      Item it;
      bool have = next_item<kMode>(p, n_rounds, k, it, false);
      while (have && ok) {
        int k2 = k + 1;
        Item nx;
        const bool have_next = next_item<kMode>(p, n_rounds, k2, nx, false);
        for (int kt = 0; kt < it.n; ++kt, ++gk, sb.next(), rv.next()) {
          if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
          if (!warp_wait(bar(kBarVFull + rv.idx), rv.ph) ||
              !warp_wait(bar(kBarPFull + sb.idx), sb.ph)) {
            ok = false;
            timeout = true;
            break;
          }
          tc_fence_after();
          const uint32_t v_s = sbase + kOffV + rv.idx * kTile;
          const uint32_t p_t = tmem + kColS + sb.idx * kN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // A = P: 16 keys = 8 packed columns per step.  B = V: 64-dim boxes
            // kHalf apart (LBO), 8-key swizzle atoms 1024 bytes apart (SBO).
            umma_bf16_tmem_a_warp(d_o, p_t + ks * 8, smem_desc_sw128(v_s + ks * 2048, kHalf, 1024),
                                  idesc_o, (kt > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit_warp(bar(kBarVEmpty + rv.idx));
          umma_commit_warp(bar(kBarPVDone + sb.idx));
        }
        if (!ok) break;
        umma_commit_warp(bar(kBarOFull));
        it = nx;
        k = k2;
        have = have_next;
      }
      if (timeout && lane == 0) record_error(p.err, kErrTimeout);
      if (!ok && lane == 0) flags[0] = 1;
      umma_commit_warp(bar(kBarDrainPV));
      (void)warp_wait(bar(kBarDrainPV), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w owns 16 whole rows of every tile: TMEM lanes 32(w%4) + 16(w/4) +
    // [0, 16).  Through the 16x256b access shape thread t holds rows
    // ra = .. + t/4 and rb = ra + 8, key columns 8k + 2(t%4) + {0, 1}
    // (k = 0..15); the four threads of a row reduce its max and sum with two
    // shuffles, and no warp waits for another.
    const int qd = warp & 3;
    const int m4 = lane & 3;
    const int ra = qd * 32 + (warp >> 2) * 16 + (lane >> 2);   // rows within the tile
    const int rb = ra + 8;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32 + (warp >> 2) * 16) << 16);
    const uint32_t o_col = lane_base + kColO;
    const f32x2 sc2 = pack2(p.scale_log2, p.scale_log2);
    bool ok = true, timeout = false;
    int gi = 0, gk = 0;
    Ring<kSBufs> sb;
    Ring<kVStages> rv;   // V stage of the current tile (for the ragged-end clearing)
    auto row_max = [&](float v) {
      v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
      return fmaxf(v, __shfl_xor_sync(kFull, v, 2));
    };
    auto row_sum = [&](float v) {
      v += __shfl_xor_sync(kFull, v, 1);
      return v + __shfl_xor_sync(kFull, v, 2);
    };
    // Output of a finished item: O / l for both rows, written row by row.  It
    // runs inside the first tile of the next item, after that tile's P is in
    // place and before P is handed on, so the last PV of the item has long
    // finished and the next item's first PV cannot overwrite O too early.
    auto epilogue = [&](const Item& e, float ema, float emb, f32x2 ela, f32x2 elb,
                        int egi) -> bool {
      const float la = row_sum(lo2(ela) + hi2(ela));
      const float lb = row_sum(lo2(elb) + hi2(elb));
      if (!warp_wait(bar(kBarOFull), egi & 1)) return false;
      tc_fence_after();
      const float ia = 1.f / la, ib = 1.f / lb;
      const bool va = ra < e.rows, vb = rb < e.rows;
      int64_t rowa = 0, rowb = 0;   // output rows (causal) or partial rows (shared prefix)
      if constexpr (kPrefix) {
        const int ga = e.q0 + ra, gb = e.q0 + rb;
        rowa = (static_cast<int64_t>(ga / g) * p.Hq + e.kvh * g + ga % g) * p.splits + e.z;
        rowb = (static_cast<int64_t>(gb / g) * p.Hq + e.kvh * g + gb % g) * p.splits + e.z;
      } else if constexpr (kMode == kVerify) {
        // row r: position r/g of the sequence, head kvh*g + r%g
        rowa = static_cast<int64_t>(e.q_begin + ra / g) * p.Hq + e.h + ra % g;
        rowb = static_cast<int64_t>(e.q_begin + rb / g) * p.Hq + e.h + rb % g;
      } else {
        rowa = static_cast<int64_t>(e.q_begin + e.q0 + ra) * p.Hq + e.h;
        rowb = static_cast<int64_t>(e.q_begin + e.q0 + rb) * p.Hq + e.h;
      }
      // O for both rows in one load: o[4j], o[4j+1] (row ra) and o[4j+2],
      // o[4j+3] (row rb) hold dims 8j + 2 m4 + {0, 1}, j = 0..15.  Lanes m4 and
      // m4 ^ 1 swap one pair per 16-dim group, so that each lane writes 4
      // consecutive dims and the four lanes of a row one whole 32-byte sector
      // per store (fp32 partials: two sectors): even lanes keep group j = 2i
      // (dims 16i + 2 m4 ..), odd lanes j = 2i + 1 (dims 16i + 8 + 2 (m4 - 1) ..).
      uint32_t o[64];
      tmem_ld16x256_x16_wait(o_col, o);
      const bool odd = m4 & 1;
      const int cbase = odd ? 8 + 2 * (m4 - 1) : 2 * m4;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int col = 16 * i + cbase;
        const float ae0 = __uint_as_float(o[8 * i]) * ia, ae1 = __uint_as_float(o[8 * i + 1]) * ia;
        const float be0 = __uint_as_float(o[8 * i + 2]) * ib, be1 = __uint_as_float(o[8 * i + 3]) * ib;
        const float ao0 = __uint_as_float(o[8 * i + 4]) * ia, ao1 = __uint_as_float(o[8 * i + 5]) * ia;
        const float bo0 = __uint_as_float(o[8 * i + 6]) * ib, bo1 = __uint_as_float(o[8 * i + 7]) * ib;
        if constexpr (kPrefix) {
          // send the pair the neighbour keeps; keep own pair first (even) or second (odd)
          const float sa0 = odd ? ae0 : ao0, sa1 = odd ? ae1 : ao1;
          const float sb0 = odd ? be0 : bo0, sb1 = odd ? be1 : bo1;
          const float xa0 = __shfl_xor_sync(kFull, sa0, 1), xa1 = __shfl_xor_sync(kFull, sa1, 1);
          const float xb0 = __shfl_xor_sync(kFull, sb0, 1), xb1 = __shfl_xor_sync(kFull, sb1, 1);
          const float4 va4 = odd ? make_float4(xa0, xa1, ao0, ao1) : make_float4(ae0, ae1, xa0, xa1);
          const float4 vb4 = odd ? make_float4(xb0, xb1, bo0, bo1) : make_float4(be0, be1, xb0, xb1);
          if (va) *reinterpret_cast<float4*>(p.part_o + rowa * kHeadDim + col) = va4;
          if (vb) *reinterpret_cast<float4*>(p.part_o + rowb * kHeadDim + col) = vb4;
        } else {
          const uint32_t ae = pack_bf16x2(ae0, ae1), ao = pack_bf16x2(ao0, ao1);
          const uint32_t be = pack_bf16x2(be0, be1), bo = pack_bf16x2(bo0, bo1);
          const uint32_t xa = __shfl_xor_sync(kFull, odd ? ae : ao, 1);
          const uint32_t xb = __shfl_xor_sync(kFull, odd ? be : bo, 1);
          const uint2 wa = odd ? make_uint2(xa, ao) : make_uint2(ae, xa);
          const uint2 wb = odd ? make_uint2(xb, bo) : make_uint2(be, xb);
          if (va) *reinterpret_cast<uint2*>(p.out + rowa * kHeadDim + col) = wa;
          if (vb) *reinterpret_cast<uint2*>(p.out + rowb * kHeadDim + col) = wb;
        }
      }
      if (m4 == 0) {
        if constexpr (kPrefix) {
          if (va) p.part_lse[rowa] = ema + __log2f(la);
          if (vb) p.part_lse[rowb] = emb + __log2f(lb);
        } else if (p.lse) {
          if (va) p.lse[rowa] = (ema + __log2f(la)) * kLn2;
          if (vb) p.lse[rowb] = (emb + __log2f(lb)) * kLn2;
        }
      }
      return true;
    };
    bool pend = false;        // an item's output is still to be written
    Item pit;
    float pma = 0.f, pmb = 0.f;
    f32x2 pla = 0ull, plb = 0ull;
    int k = 0;
    Item it;
    bool have = next_item<kMode>(p, n_rounds, k, it, warp == 0 && lane == 0);
    while (have && ok) {
      int k2 = k + 1;
      Item nx;
      const bool have_next = next_item<kMode>(p, n_rounds, k2, nx, warp == 0 && lane == 0);
      // last visible keys: row r is query position r (r / g in verify mode)
      const int visa = it.diag + (kMode == kVerify ? ra / g : ra);
      const int visb = it.diag + (kMode == kVerify ? rb / g : rb);
      float ma = -INFINITY, mb = -INFINITY;
      f32x2 la2 = pack2(0.f, 0.f), lb2 = pack2(0.f, 0.f);  // running sums, as pairs
      for (int kt = 0; kt < it.n; ++kt, ++gk, sb.next(), rv.next()) {
        if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
        const uint32_t s_col = lane_base + kColS + sb.idx * kN;
        if (!(ok = warp_wait(bar(kBarSFull + sb.idx), sb.ph))) { timeout = true; break; }
        tc_fence_after();
        uint32_t r[64];
        tmem_ld16x256_x16_wait(s_col, r);
        const int j0 = (it.kt0 + kt) * kN + 2 * m4;   // key of register 0
        if (!kPrefix && (it.kt0 + kt) * kN + kN - 1 > it.diag) {   // causal edge
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int key = j0 + 8 * q;
            if (key > visa) r[4 * q] = __float_as_uint(-INFINITY);
            if (key + 1 > visa) r[4 * q + 1] = __float_as_uint(-INFINITY);
            if (key > visb) r[4 * q + 2] = __float_as_uint(-INFINITY);
            if (key + 1 > visb) r[4 * q + 3] = __float_as_uint(-INFINITY);
          }
        }
        float xa0 = __uint_as_float(r[0]), xa1 = __uint_as_float(r[1]);
        float xb0 = __uint_as_float(r[2]), xb1 = __uint_as_float(r[3]);
#pragma unroll
        for (int q = 1; q < 16; ++q) {
          xa0 = fmaxf(xa0, __uint_as_float(r[4 * q]));
          xa1 = fmaxf(xa1, __uint_as_float(r[4 * q + 1]));
          xb0 = fmaxf(xb0, __uint_as_float(r[4 * q + 2]));
          xb1 = fmaxf(xb1, __uint_as_float(r[4 * q + 3]));
        }
        const float mta = row_max(fmaxf(xa0, xa1)) * p.scale_log2;
        const float mtb = row_max(fmaxf(xb0, xb1)) * p.scale_log2;
        if (kt == 0) {
          ma = mta;
          mb = mtb;
        } else {
          const bool need_a = mta > ma + kLazyRescale, need_b = mtb > mb + kLazyRescale;
          if (__any_sync(kFull, need_a || need_b)) {
            // the previous PV must have finished accumulating into O
            const int pb = sb.idx == 0 ? kSBufs - 1 : sb.idx - 1;
            const uint32_t pph = sb.idx == 0 ? sb.ph ^ 1u : sb.ph;
            if (!(ok = warp_wait(bar(kBarPVDone + pb), pph))) { timeout = true; break; }
            tc_fence_after();
            const float alpha_a = need_a ? ex2(ma - mta) : 1.f;
            const float alpha_b = need_b ? ex2(mb - mtb) : 1.f;
            if (need_a) {
              la2 = mul2(la2, pack2(alpha_a, alpha_a));
              ma = mta;
            }
            if (need_b) {
              lb2 = mul2(lb2, pack2(alpha_b, alpha_b));
              mb = mtb;
            }
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t o[32];
              tmem_ld16x256_x8_wait(o_col + h2 * 64, o);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                o[4 * j] = __float_as_uint(__uint_as_float(o[4 * j]) * alpha_a);
                o[4 * j + 1] = __float_as_uint(__uint_as_float(o[4 * j + 1]) * alpha_a);
                o[4 * j + 2] = __float_as_uint(__uint_as_float(o[4 * j + 2]) * alpha_b);
                o[4 * j + 3] = __float_as_uint(__uint_as_float(o[4 * j + 3]) * alpha_b);
              }
              tmem_st16x256_x8(o_col + h2 * 64, o);
            }
          }
        }
        // P = 2^(scale*s - m) as bf16 pairs: P column 4q + m4 holds keys
        // 8q + 2 m4 + {0, 1} (the 16x128b shape).  Hidden keys hold -inf and
        // get weight exactly 0.
        const f32x2 nma = pack2(-ma, -ma), nmb = pack2(-mb, -mb);
        uint32_t pk[32];
        f32x2 sa = pack2(0.f, 0.f), sb2 = pack2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const f32x2 xa =
              fma2(pack2(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1])), sc2, nma);
          const f32x2 xb =
              fma2(pack2(__uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])), sc2, nmb);
          const float a0 = ex2(lo2(xa)), a1 = ex2(hi2(xa));
          const float b0 = ex2(lo2(xb)), b1 = ex2(hi2(xb));
          pk[2 * q] = pack_bf16x2(a0, a1);
          pk[2 * q + 1] = pack_bf16x2(b0, b1);
          sa = add2(sa, pack2(a0, a1));
          sb2 = add2(sb2, pack2(b0, b1));
        }
        la2 = add2(la2, sa);
        lb2 = add2(lb2, sb2);
        tmem_st16x128_x16(s_col, pk);
        // keys past the end of the sequence in its last tile: zero their V rows
        // so that 0 * (stale data) cannot put a NaN into O (thread s of the 256
        // softmax threads clears row s/2, dims 64(s%2)..)
        if (!kPrefix && kt == it.n - 1 && (it.kt0 + kt) * kN + kN > it.Lk) {
          if (!(ok = warp_wait(bar(kBarVFull + rv.idx), rv.ph))) { timeout = true; break; }
          const int vr = tid >> 1, vh = tid & 1;
          if ((it.kt0 + kt) * kN + vr >= it.Lk) {
            const uint4 zero = make_uint4(0, 0, 0, 0);
            const uint32_t vrow = sbase + kOffV + rv.idx * kTile + vh * kHalf + vr * 128;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) sts128(vrow + cc * 16, zero);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        if (kt == 0 && pend) {
          pend = false;
          if (!(ok = epilogue(pit, pma, pmb, pla, plb, gi - 1))) { timeout = true; break; }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + sb.idx));
      }
      if (!ok) break;
      pend = true;
      pit = it;
      pma = ma;
      pmb = mb;
      pla = la2;
      plb = lb2;
      ++gi;
      it = nx;
      k = k2;
      have = have_next;
    }
    if (ok && pend && !(ok = epilogue(pit, pma, pmb, pla, plb, gi - 1))) timeout = true;
    if (timeout && lane == 0) record_error(p.err, kErrTimeout);
    if (!ok && lane == 0) flags[0] = 1;
  }

  tc_fence_before();
  __syncthreads();
  // After an abort, wait (bounded) for TMA copies that may still be landing:
  // the last two issued tiles of each ring.
  if (flags[0] && tid == kQKWarp * 32) {
    const int kin = flags[1], qin = flags[3];
    for (int x = max(0, kin - kKStages); x < kin; ++x)
      (void)mbar_wait(bar(kBarKFull + x % kKStages), (x / kKStages) & 1);
    if (qin > 0) (void)mbar_wait(bar(kBarQFull), (qin - 1) & 1);
  }
  if (flags[0] && tid == kVWarp * 32) {
    const int vin = flags[2];
    for (int x = max(0, vin - kVStages); x < vin; ++x)
      (void)mbar_wait(bar(kBarVFull + x % kVStages), (x / kVStages) & 1);
  }
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


template <int kMode>
bool set_smem_attr() {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(paged_prefill_kernel<kMode>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return false;
    attr_set[dev] = true;
  }
  return true;
}

int grid_for(int n_items) {
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  return n_items < sms ? n_items : sms;
}

}  // namespace

int set_wait_hook_prefill(unsigned long long limit_ns, int withhold_plus1) {
  const WaitHook h{limit_ns, withhold_plus1, 0};
  return cudaMemcpyToSymbol(g_wait_hook, &h, sizeof h) == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int prefix_rows_per_tile(int g) { return (g >= 1 && g <= kM) ? (kM / g) * g : 0; }

int launch_prefill(const PrefillArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.B == 0 || a.max_seqlen_q == 0) return PKV_OK;
  // The query map spans B * max_seqlen_q rows, at least the real sum of Lq.
  // Only full 128-row tiles go through it, and a full tile never leaves its
  // sequence, so every row it reads exists.
  const int64_t q_rows = static_cast<int64_t>(a.B) * a.max_seqlen_q;
  if (q_rows > INT32_MAX) return PKV_ERR_SHAPE;
  CUtensorMap qm, km, vm;
  const int64_t slots = a.num_blocks * kBlockSize;
  if (!encode_pool_map(&qm, a.q, q_rows, a.Hq, kM) ||
      !encode_pool_map(&km, a.k_cache, slots, a.Hkv, kN) ||
      !encode_pool_map(&vm, a.v_cache, slots, a.Hkv, kN))
    return PKV_ERR_ARG;
  PrefillParams prm = {};
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.lse = a.lse;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_tables = a.block_tables;
  prm.cu_q = a.cu_seqlens_q;
  prm.cu_k = a.cu_seqlens_k;
  prm.err = err;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.maxblk = a.max_blocks_per_seq;
  prm.max_q = a.max_seqlen_q;
  prm.max_k = a.max_seqlen_k;
  prm.n_qt = (a.max_seqlen_q + kM - 1) / kM;
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  const int64_t items = static_cast<int64_t>(prm.n_qt) * a.B * a.Hq;
  if (items > INT32_MAX) return PKV_ERR_SHAPE;
  prm.n_items = static_cast<int>(items);
  if (!set_smem_attr<kCausal>()) return PKV_ERR_LAUNCH;
  paged_prefill_kernel<kCausal><<<grid_for(prm.n_items), kThreads, kSmemBytes, stream>>>(
      qm, km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int launch_prefix_attention(const PrefixArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.B == 0 || a.prefix_tokens == 0) return PKV_OK;
  const int g = a.Hq / a.Hkv;
  const int rpt = prefix_rows_per_tile(g);
  if (rpt == 0) return PKV_ERR_SHAPE;
  CUtensorMap qm, km, vm;
  const int64_t slots = a.num_blocks * kBlockSize;
  // q [B, Hq, 128]: a box is 64 dims x the g heads of one kv head x rpt/g tokens
  if (!encode_pool_map(&qm, a.q, a.B, a.Hq, rpt / g, g) ||
      !encode_pool_map(&km, a.k_cache, slots, a.Hkv, kN) ||
      !encode_pool_map(&vm, a.v_cache, slots, a.Hkv, kN))
    return PKV_ERR_ARG;
  PrefillParams prm = {};
  prm.part_o = a.part_o;
  prm.part_lse = a.part_lse;
  prm.prefix_tokens = a.prefix_tokens;
  prm.prefix_kt_per = a.kt_per;
  prm.splits = a.splits;
  prm.rows_per_tile = rpt;
  prm.n_rt = (a.B * g + rpt - 1) / rpt;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_tables = a.block_tables;
  prm.err = err;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  const int64_t items = static_cast<int64_t>(prm.n_rt) * a.Hkv * a.splits;
  if (items > INT32_MAX) return PKV_ERR_SHAPE;
  prm.n_items = static_cast<int>(items);
  if (!set_smem_attr<kPrefixPass>()) return PKV_ERR_LAUNCH;
  paged_prefill_kernel<kPrefixPass><<<grid_for(prm.n_items), kThreads, kSmemBytes, stream>>>(
      qm, km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int verify_rows_fit(int g, int q_len) { return g >= 1 && q_len >= 1 && g * q_len <= kM; }

int launch_verify(const VerifyArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.B == 0) return PKV_OK;
  const int g = a.Hq / a.Hkv;
  if (!verify_rows_fit(g, a.q_len)) return PKV_ERR_SHAPE;
  const int64_t q_rows = static_cast<int64_t>(a.B) * a.q_len;
  if (q_rows > INT32_MAX) return PKV_ERR_SHAPE;
  CUtensorMap qm, km, vm;
  const int64_t slots = a.num_blocks * kBlockSize;
  // q [B*q_len, Hq, 128]: a box is 64 dims x the g heads of one kv head x q_len positions
  if (!encode_pool_map(&qm, a.q, q_rows, a.Hq, a.q_len, g) ||
      !encode_pool_map(&km, a.k_cache, slots, a.Hkv, kN) ||
      !encode_pool_map(&vm, a.v_cache, slots, a.Hkv, kN))
    return PKV_ERR_ARG;
  PrefillParams prm = {};
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.lse = a.lse;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_tables = a.block_tables;
  prm.ctx = a.context_lens;
  prm.err = err;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.maxblk = a.max_blocks_per_seq;
  prm.q_len = a.q_len;
  prm.rows_per_tile = g * a.q_len;
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  const int64_t items = static_cast<int64_t>(a.B) * a.Hkv;
  if (items > INT32_MAX) return PKV_ERR_SHAPE;
  prm.n_items = static_cast<int>(items);
  if (!set_smem_attr<kVerify>()) return PKV_ERR_LAUNCH;
  paged_prefill_kernel<kVerify><<<grid_for(prm.n_items), kThreads, kSmemBytes, stream>>>(
      qm, km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv
