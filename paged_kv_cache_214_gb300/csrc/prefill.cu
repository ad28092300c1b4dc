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
// The same kernel computes the shared-prefix pass of a decode batch (kPrefix).
//
// Work item: one 128-row query tile (one sequence and query head) and its key
// tiles.  The kernel is persistent: one block per SM walks the items, heaviest
// first, so that set-up, the first loads and the output stores of one item
// overlap the next.  Twelve warps, each with one job:
//   warp 8  (TMA)  Q tiles and 128-key K tiles (two 64-dim boxes, 128-byte
//                  swizzle); a K tile never straddles a 256-token block.
//   warp 9  (TMA)  V tiles.
//   warp 10 (MMA)  S_t = Q K_t^T into one of three S buffers in tensor memory.
//   warp 11 (MMA)  O += P_t V_t, A = P_t read from tensor memory, B = V_t
//                  MN-major straight from its TMA tile.
//   warps 0-7      softmax: warp w owns rows 32(w%4).. (its TMEM lane quarter)
//                  and key columns 64(w/4).. of every S tile.  The two warps of
//                  a row quarter exchange their partial row maxima through
//                  shared memory, keep the running max in base 2, rescale O
//                  only when the max grew by more than 2^8 (weights below 256
//                  are exact enough in fp32 / bf16), and write P as bf16 pairs
//                  over the first 64 columns of the tile's S buffer.
// The MMAs come from two threads: one thread issuing M=N=128 tcgen05.mma in a
// chain waits ~116 cycles per instruction, about half the tensor pipe, while
// two independent chains fill it.  S is triple-buffered, so the S of tile t+1
// (and t+2) is computed while the softmax of tile t runs.
// TMEM (512 columns): S_0 | S_1 | S_2 | O.
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
constexpr int kOffQ = 0;                   // 2 buffers
constexpr int kOffK = kOffQ + 2 * kTile;   // 2 stages
constexpr int kOffV = kOffK + 2 * kTile;   // 2 stages
constexpr int kOffXMax = kOffV + 2 * kTile;          // f32 [2 parity][2 halves][128 rows]
constexpr int kOffXSum = kOffXMax + 2 * 2 * 128 * 4; // f32 [2 halves][128 rows]
constexpr int kOffBars = kOffXSum + 2 * 128 * 4;
constexpr int kSBufs = 3;
// barriers
constexpr int kBarQFull = 0;    // [Q buffer]
constexpr int kBarQEmpty = 2;   // [Q buffer]
constexpr int kBarKFull = 4;    // [stage]
constexpr int kBarKEmpty = 6;   // [stage]
constexpr int kBarVFull = 8;    // [stage]
constexpr int kBarVEmpty = 10;  // [stage]
constexpr int kBarSFull = 12;   // [S buffer] x3
constexpr int kBarPFull = 15;   // [S buffer] x3, 8 softmax warps
constexpr int kBarPVDone = 18;  // [S buffer] x3: the PV that read P from it has completed
constexpr int kBarOFull = 21;   // the last PV of an item has completed
constexpr int kBarXMax = 22;    // [row quarter][parity]: 2 warps
constexpr int kBarXSum = 30;    // [row quarter]: 2 warps
constexpr int kBarDrainS = 34;
constexpr int kBarDrainPV = 35;
constexpr int kNumBars = 36;
constexpr int kOffTmem = kOffBars + kNumBars * 8;
constexpr int kOffFlags = kOffTmem + 8;
constexpr int kSmemBytes = kOffFlags + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // + 128 * buffer
constexpr uint32_t kColO = 384;
constexpr float kLazyRescale = 8.f;    // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint32_t kFull = 0xffffffffu;

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

template <bool kPrefix>
__device__ __forceinline__ Item get_item(const PrefillParams& p, int idx, bool report) {
  Item it;
  const int g = p.Hq / p.Hkv;
  it.n = 0;
  it.h = 0;
  it.q_begin = 0;
  it.z = 0;
  if constexpr (kPrefix) {
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

// Wait with every lane of the warp; the result is the same for all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(kFull, mbar_wait(bar, parity));
}

// Running position in the three-way S ring: buffer and phase parity.
struct Ring3 {
  int buf = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++buf == kSBufs) {
      buf = 0;
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

// kPrefix = false: causal (chunked) prefill over (row tile, sequence, query head) items.
// kPrefix = true: the shared-prefix pass of a decode batch.  For kv head kvh the
// query rows are the B*g (sequence, query head) pairs of its group (row r =
// sequence r/g, head kvh*g + r%g); every row sees all prefix_tokens keys of the
// blocks that open table row 0, split into key ranges; the output is a
// normalised fp32 partial and its log2-sum-exp per range, merged into the
// decode result afterwards.
template <bool kPrefix>
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
  float* xmax = reinterpret_cast<float*>(smem + kOffXMax);
  float* xsum = reinterpret_cast<float*>(smem + kOffXSum);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = p.Hq / p.Hkv;
  const int n_rounds = (p.n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  const int table_limit = kPrefix ? p.prefix_tokens / kBlockSize : p.maxblk;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i >= kBarPFull && i < kBarPFull + kSBufs) count = kSoftmaxWarps;
      if (i >= kBarXMax && i < kBarDrainS) count = 2;   // the two warps of a row quarter
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
    // The Q of an item is loaded while the previous item streams its keys:
    // right after that item's second K tile (or at the very start).
    bool ok = true;
    int gi = 0, gk = 0;
    BlockIds ids;
    auto load_q = [&](const Item& it, int qi) -> bool {
      const int qb = qi & 1;
      const uint32_t qdst = sbase + kOffQ + qb * kTile;
      if (qi >= 2 && !warp_wait(bar(kBarQEmpty + qb), ((qi - 2) >> 1) & 1)) return false;
      if (!kPrefix && it.rows < kM) {
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
        if (lane == 0) mbar_arrive(bar(kBarQFull + qb));
      } else if (lane == 0) {
        if constexpr (kPrefix) {
          // (sequence, head) rows of the group: box {64 dims, g heads, tokens}
          mbar_arrive_expect_tx(bar(kBarQFull + qb), p.rows_per_tile * 256);
          const int tok0 = it.q0 / g;
          tma_load_3d(qdst, &qmap, bar(kBarQFull + qb), 0, it.kvh * g, tok0);
          tma_load_3d(qdst + kHalf, &qmap, bar(kBarQFull + qb), 64, it.kvh * g, tok0);
        } else {
          mbar_arrive_expect_tx(bar(kBarQFull + qb), kTile);
          const int row0 = it.q_begin + it.q0;
          tma_load_3d(qdst, &qmap, bar(kBarQFull + qb), 0, it.h, row0);
          tma_load_3d(qdst + kHalf, &qmap, bar(kBarQFull + qb), 64, it.h, row0);
        }
      }
      if (lane == 0) flags[3] = qi + 1;
      __syncwarp();
      return true;
    };
    // first non-empty item at or after round k
    auto next_item = [&](int& k, Item& it) -> bool {
      for (; k < n_rounds; ++k) {
        const int idx = item_index(k);
        if (idx >= p.n_items) continue;
        it = get_item<kPrefix>(p, idx, false);
        if (it.n > 0) return true;
      }
      return false;
    };
    int k = 0;
    Item it;
    bool have = next_item(k, it);
    if (have && !load_q(it, 0)) {
      ok = false;
      if (lane == 0) record_error(p.err, kErrTimeout);
    }
    while (have && ok) {
      int k2 = k + 1;
      Item nx;
      const bool have_next = next_item(k2, nx);
      const int q_at = min(1, it.n - 1);   // load the next Q after this K tile
      ids.chunk = -1;
      for (int kt = 0; kt < it.n; ++kt, ++gk) {
        if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
        const int st = gk & 1;
        const int gkt = it.kt0 + kt;
        const int id = ids.get(it.table, table_limit, gkt >> 1, lane, p.num_blocks, p.err);
        const int slot = id * kBlockSize + (gkt & 1) * kN;
        if (gk >= 2 && !warp_wait(bar(kBarKEmpty + st), ((gk - 2) >> 1) & 1)) {
          ok = false;
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
        if (lane == 0) {
          const uint32_t kdst = sbase + kOffK + st * kTile;
          mbar_arrive_expect_tx(bar(kBarKFull + st), kTile);
          tma_load_3d(kdst, &kmap, bar(kBarKFull + st), 0, it.kvh, slot);
          tma_load_3d(kdst + kHalf, &kmap, bar(kBarKFull + st), 64, it.kvh, slot);
          flags[1] = gk + 1;
        }
        __syncwarp();
        if (kt == q_at && have_next && !load_q(nx, gi + 1)) {
          ok = false;
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
      }
      if (!ok) break;
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
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int idx = item_index(k);
      if (idx >= p.n_items) continue;
      const Item it = get_item<kPrefix>(p, idx, false);
      if (it.n == 0) continue;
      ids.chunk = -1;
      for (int kt = 0; kt < it.n; ++kt, ++gk) {
        if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
        const int st = gk & 1;
        const int gkt = it.kt0 + kt;
        const int id = ids.get(it.table, table_limit, gkt >> 1, lane, p.num_blocks, p.err);
        const int slot = id * kBlockSize + (gkt & 1) * kN;
        if (gk >= 2 && !warp_wait(bar(kBarVEmpty + st), ((gk - 2) >> 1) & 1)) {
          ok = false;
          if (lane == 0) record_error(p.err, kErrTimeout);
          break;
        }
        if (lane == 0) {
          const uint32_t vdst = sbase + kOffV + st * kTile;
          mbar_arrive_expect_tx(bar(kBarVFull + st), kTile);
          tma_load_3d(vdst, &vmap, bar(kBarVFull + st), 0, it.kvh, slot);
          tma_load_3d(vdst + kHalf, &vmap, bar(kBarVFull + st), 64, it.kvh, slot);
          flags[2] = gk + 1;
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) flags[0] = 1;
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ MMA: S = Q K^T
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kN, 0);   // B = K, K-major
      bool ok = true, timeout = false;
      int gi = 0, gk = 0;
      Ring3 sb;
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int idx = item_index(k);
        if (idx >= p.n_items) continue;
        const Item it = get_item<kPrefix>(p, idx, false);
        if (it.n == 0) continue;
        const int qb = gi & 1;
        if (!mbar_wait(bar(kBarQFull + qb), (gi >> 1) & 1)) { ok = false; timeout = true; break; }
        const uint32_t q_s = sbase + kOffQ + qb * kTile;
        for (int kt = 0; kt < it.n; ++kt, ++gk, sb.next()) {
          if (flags[0]) { ok = false; break; }
          const int st = gk & 1;
          if (!mbar_wait(bar(kBarKFull + st), (gk >> 1) & 1)) { ok = false; timeout = true; break; }
          // S buffer free: the PV that read P from it (three tiles back) is done
          if (gk >= kSBufs && !mbar_wait(bar(kBarPVDone + sb.buf), sb.ph ^ 1u)) {
            ok = false;
            timeout = true;
            break;
          }
          tc_fence_after();
          const uint32_t k_s = sbase + kOffK + st * kTile;
          const uint32_t d_s = tmem + kColS + sb.buf * kN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
            umma_bf16(d_s, smem_desc_sw128(q_s + off, 16, 1024),
                      smem_desc_sw128(k_s + off, 16, 1024), idesc_s, ks > 0);
          }
          umma_commit(bar(kBarSFull + sb.buf));
          umma_commit(bar(kBarKEmpty + st));
        }
        if (!ok) break;
        umma_commit(bar(kBarQEmpty + qb));
        ++gi;
      }
      if (timeout) record_error(p.err, kErrTimeout);
      if (!ok) flags[0] = 1;
      // every MMA this thread issued has completed once this arrives
      umma_commit(bar(kBarDrainS));
      (void)mbar_wait(bar(kBarDrainS), 0);
    }
  } else if (warp == kPVWarp) {
    // ------------------------------------------------------------ MMA: O += P V
    if (lane == 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(kM, kHeadDim, 1);  // B = V, MN-major
      bool ok = true, timeout = false;
      int gk = 0;
      Ring3 sb;
      const uint32_t d_o = tmem + kColO;
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int idx = item_index(k);
        if (idx >= p.n_items) continue;
        const Item it = get_item<kPrefix>(p, idx, false);
        if (it.n == 0) continue;
        for (int kt = 0; kt < it.n; ++kt, ++gk, sb.next()) {
          if (flags[0]) { ok = false; break; }
          const int st = gk & 1;
          if (!mbar_wait(bar(kBarVFull + st), (gk >> 1) & 1) ||
              !mbar_wait(bar(kBarPFull + sb.buf), sb.ph)) {
            ok = false;
            timeout = true;
            break;
          }
          tc_fence_after();
          const uint32_t v_s = sbase + kOffV + st * kTile;
          const uint32_t p_t = tmem + kColS + sb.buf * kN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // A = P: 16 keys = 8 packed columns per step.  B = V: 64-dim boxes
            // kHalf apart (LBO), 8-key swizzle atoms 1024 bytes apart (SBO).
            umma_bf16_tmem_a(d_o, p_t + ks * 8, smem_desc_sw128(v_s + ks * 2048, kHalf, 1024),
                             idesc_o, (kt > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(bar(kBarVEmpty + st));
          umma_commit(bar(kBarPVDone + sb.buf));
        }
        if (!ok) break;
        umma_commit(bar(kBarOFull));
      }
      if (timeout) record_error(p.err, kErrTimeout);
      if (!ok) flags[0] = 1;
      umma_commit(bar(kBarDrainPV));
      (void)mbar_wait(bar(kBarDrainPV), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;               // row quarter = TMEM lane quarter
    const int c = warp >> 2;               // key-column half of every tile
    const int i = qd * 32 + lane;          // query row within the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    const uint32_t o_col = lane_base + kColO + c * 64;
    const f32x2 sc2 = pack2(p.scale_log2, p.scale_log2);
    bool ok = true, timeout = false;
    int gi = 0, gk = 0;
    Ring3 sb;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int idx = item_index(k);
      if (idx >= p.n_items) continue;
      const Item it = get_item<kPrefix>(p, idx, warp == 0 && lane == 0);
      if (it.n == 0) continue;
      const int vis = it.diag + i;         // last visible key of this row
      float m = -INFINITY;
      f32x2 l2 = pack2(0.f, 0.f);          // this half's running sum, as a pair
      for (int kt = 0; kt < it.n; ++kt, ++gk, sb.next()) {
        if (__any_sync(kFull, flags[0] != 0)) { ok = false; break; }
        const uint32_t s_col = lane_base + kColS + sb.buf * kN;
        if (!(ok = warp_wait(bar(kBarSFull + sb.buf), sb.ph))) { timeout = true; break; }
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64_wait(s_col + c * 64, r);
        const int j0 = (it.kt0 + kt) * kN + c * 64;   // key of column 0 of this half
        if (!kPrefix && j0 + 63 > it.diag) {          // causal edge: hide later keys
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (j0 + cc > vis) r[cc] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = __uint_as_float(r[t]);
#pragma unroll
        for (int cc = 8; cc < 64; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], __uint_as_float(r[cc]));
        const float pm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        // exchange the partial maxima of the two halves of these rows
        float* xm = xmax + (gk & 1) * 256;
        xm[c * 128 + i] = pm;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarXMax + qd * 2 + (gk & 1)));
        if (!(ok = warp_wait(bar(kBarXMax + qd * 2 + (gk & 1)), (gk >> 1) & 1))) {
          timeout = true;
          break;
        }
        // both halves have read their S columns: P may now overwrite them
        const float mt = fmaxf(pm, xm[(c ^ 1) * 128 + i]) * p.scale_log2;
        if (kt == 0) {
          m = mt;
        } else {
          const bool need = mt > m + kLazyRescale;
          if (__any_sync(kFull, need)) {
            // the previous PV must have finished accumulating into O
            const int pb = sb.buf == 0 ? kSBufs - 1 : sb.buf - 1;
            const uint32_t pph = sb.buf == 0 ? sb.ph ^ 1u : sb.ph;
            if (!(ok = warp_wait(bar(kBarPVDone + pb), pph))) { timeout = true; break; }
            tc_fence_after();
            const float alpha = need ? ex2(m - mt) : 1.f;
            if (need) {
              l2 = mul2(l2, pack2(alpha, alpha));
              m = mt;
            }
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t o[32];
              tmem_ld32_wait(o_col + hh * 32, o);
#pragma unroll
              for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
              tmem_st32(o_col + hh * 32, o);
            }
          }
        }
        // P = 2^(scale*s - m) as bf16 pairs: columns [32c, 32c+32) of the S buffer.
        // Hidden keys hold -inf, so their weight is exactly 0.
        const f32x2 nm2 = pack2(-m, -m);
        uint32_t pk[32];
        f32x2 acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const f32x2 x =
              fma2(pack2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1])), sc2, nm2);
          const float e0 = ex2(lo2(x)), e1 = ex2(hi2(x));
          pk[t] = pack_bf16x2(e0, e1);
          if (t & 1)
            acc1 = add2(acc1, pack2(e0, e1));
          else
            acc0 = add2(acc0, pack2(e0, e1));
        }
        l2 = add2(l2, add2(acc0, acc1));
        tmem_st32(s_col + c * 32, pk);
        // keys past the end of the sequence in its last tile: zero their V rows
        // so that 0 * (stale data) cannot put a NaN into O
        if (!kPrefix && kt == it.n - 1 && (it.kt0 + kt) * kN + kN > it.Lk) {
          const int st = gk & 1;
          if (!(ok = warp_wait(bar(kBarVFull + st), (gk >> 1) & 1))) { timeout = true; break; }
          if ((it.kt0 + kt) * kN + i >= it.Lk) {
            const uint4 zero = make_uint4(0, 0, 0, 0);
            const uint32_t vrow = sbase + kOffV + st * kTile + c * kHalf + i * 128;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) sts128(vrow + cc * 16, zero);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + sb.buf));
      }
      if (!ok) break;
      // ---- epilogue: row sum of both halves, O / l, out and lse
      float lsum = lo2(l2) + hi2(l2);
      xsum[c * 128 + i] = lsum;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarXSum + qd));
      if (!(ok = warp_wait(bar(kBarXSum + qd), gi & 1))) { timeout = true; break; }
      lsum += xsum[(c ^ 1) * 128 + i];
      if (!(ok = warp_wait(bar(kBarOFull), gi & 1))) { timeout = true; break; }
      tc_fence_after();
      const float inv = 1.f / lsum;
      const bool valid = i < it.rows;
      int64_t row = 0;
      if constexpr (kPrefix) {
        const int gr = it.q0 + i;
        row = static_cast<int64_t>(gr / g) * p.Hq + it.kvh * g + gr % g;
        row = row * p.splits + it.z;
      } else {
        row = static_cast<int64_t>(it.q_begin + it.q0 + i) * p.Hq + it.h;
      }
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[32];
        tmem_ld32_wait(o_col + hh * 32, o);
        if (!valid) continue;
        if constexpr (kPrefix) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + row * kHeadDim + c * 64 + hh * 32);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            dst[t] = make_float4(__uint_as_float(o[4 * t]) * inv, __uint_as_float(o[4 * t + 1]) * inv,
                                 __uint_as_float(o[4 * t + 2]) * inv,
                                 __uint_as_float(o[4 * t + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * kHeadDim + c * 64 + hh * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * t + 0]) * inv, __uint_as_float(o[8 * t + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * t + 2]) * inv, __uint_as_float(o[8 * t + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * t + 4]) * inv, __uint_as_float(o[8 * t + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * t + 6]) * inv, __uint_as_float(o[8 * t + 7]) * inv);
            dst[t] = v;
          }
        }
      }
      if (valid && c == 0) {
        if constexpr (kPrefix) {
          p.part_lse[row] = m + __log2f(lsum);
        } else {
          if (p.lse) p.lse[row] = (m + __log2f(lsum)) * kLn2;
        }
      }
      ++gi;
    }
    if (timeout && lane == 0) record_error(p.err, kErrTimeout);
    if (!ok && lane == 0) flags[0] = 1;
  }

  tc_fence_before();
  __syncthreads();
  // After an abort, wait (bounded) for TMA copies that may still be landing:
  // the last two issued tiles of each ring.
  if (flags[0] && tid == kQKWarp * 32) {
    const int kin = flags[1], qin = flags[3];
    for (int x = max(0, kin - 2); x < kin; ++x)
      (void)mbar_wait(bar(kBarKFull + (x & 1)), (x >> 1) & 1);
    for (int x = max(0, qin - 2); x < qin; ++x)
      (void)mbar_wait(bar(kBarQFull + (x & 1)), (x >> 1) & 1);
  }
  if (flags[0] && tid == kVWarp * 32) {
    const int vin = flags[2];
    for (int x = max(0, vin - 2); x < vin; ++x)
      (void)mbar_wait(bar(kBarVFull + (x & 1)), (x >> 1) & 1);
  }
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kPrefix>
bool set_smem_attr() {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(paged_prefill_kernel<kPrefix>,
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
  const int64_t items = static_cast<int64_t>(prm.n_qt) * a.B * a.Hq;
  if (items > INT32_MAX) return PKV_ERR_SHAPE;
  prm.n_items = static_cast<int>(items);
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  if (!set_smem_attr<false>()) return PKV_ERR_LAUNCH;
  paged_prefill_kernel<false><<<grid_for(prm.n_items), kThreads, kSmemBytes, stream>>>(qm, km, vm,
                                                                                       prm);
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
  if (!set_smem_attr<true>()) return PKV_ERR_LAUNCH;
  paged_prefill_kernel<true><<<grid_for(prm.n_items), kThreads, kSmemBytes, stream>>>(qm, km, vm,
                                                                                      prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv
