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
//
// One thread block owns two 128-row query tiles that read the same K/V: two
// query heads of one kv head's group (when Hq/Hkv is even), otherwise two
// consecutive row tiles of one head.  Every K/V tile brought in serves both.
//   warp 8 (TMA)      streams 128-key K and V tiles of the kv head from the
//                     paged pool, two stages each (two 64-dim boxes per tile,
//                     128-byte swizzle).  A 128-key tile never straddles a
//                     256-token block.
//   warp 9 (MMA)      one lane issues, per tile X and key tile t,
//                       S_X = Q_X K_t^T   (A, B from shared memory)
//                       O_X += P_X V_t    (A = P_X from tensor memory, B = V_t
//                                          MN-major straight from its TMA tile)
//                     with tcgen05.mma kind::f16 (bf16 in, fp32 accumulate in
//                     TMEM) and tcgen05.commit -> mbarrier completion.  The two
//                     tiles alternate, so the tensor core computes one tile's
//                     PV and next S while the other tile's softmax runs.
//   warps 0-3 / 4-7   softmax of tile 0 / tile 1: thread i owns query row i.
//                     It reads its score row from TMEM, applies the causal
//                     mask, keeps the running max / sum in base 2, rescales
//                     O in TMEM only when the max grew by more than 2^8
//                     (otherwise the stale max is kept: weights <= 256 are
//                     exact enough in fp32 / bf16), writes P as bf16 pairs
//                     over the first 64 columns of its own score buffer, and
//                     at the end normalises O and writes out / lse.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, P_X aliased on S_X.  The MMA that
// overwrites S_X with the next scores is issued after the PV that reads P_X;
// tcgen05.mma operations of one thread execute in issue order.
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
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kHalf = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte swizzled box)
constexpr int kTile = 2 * kHalf;       // 128 rows x 128 bf16
constexpr int kOffQ = 0;               // 2 tiles
constexpr int kOffK = kOffQ + 2 * kTile;   // 2 stages
constexpr int kOffV = kOffK + 2 * kTile;   // 2 stages
constexpr int kOffBars = kOffV + 2 * kTile;
// barriers
constexpr int kBarKFull = 0;   // [2]
constexpr int kBarKEmpty = 2;  // [2]
constexpr int kBarVFull = 4;   // [2]
constexpr int kBarVEmpty = 6;  // [2]
constexpr int kBarSFull = 8;   // [2] per query tile
constexpr int kBarPFull = 10;  // [2] per query tile
constexpr int kBarODone = 12;  // [2] per query tile
constexpr int kBarDrain = 14;
constexpr int kNumBars = 15;
constexpr int kOffTmem = kOffBars + kNumBars * 8;
constexpr int kOffFlags = kOffTmem + 8;
constexpr int kSmemBytes = kOffFlags + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // + 128 * X
constexpr uint32_t kColO = 256;    // + 128 * X
constexpr float kLazyRescale = 8.f;    // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

struct PrefillParams {
  __nv_bfloat16* out;
  float* lse;
  float* part_o;     // shared-prefix mode: [B*Hq, 128] normalised partial
  float* part_lse;   // shared-prefix mode: [B*Hq] log2-sum-exp
  int prefix_tokens; // shared-prefix mode: keys = the first prefix_tokens of table row 0
  int prefix_kt_per; // shared-prefix mode: key tiles per block (blockIdx.z = key range)
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* cu_q;
  const int32_t* cu_k;
  unsigned* err;
  int B, Hq, Hkv, maxblk, max_q, max_k;
  int n_qt;          // ceil(max_q / 128)
  int pair_heads;    // 1: the two tiles are heads 2y, 2y+1; 0: row tiles 2x, 2x+1
  int64_t num_blocks;
  float scale_log2;
};

// Wait with every lane of the warp; the result is the same for all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// kPrefix = false: causal (chunked) prefill, grid over (row-tile pairs, heads, sequences).
// kPrefix = true: the shared-prefix pass of a decode batch.  For kv head
// blockIdx.y the query rows are the B*g (sequence, query head) pairs of its
// group (row r = sequence r/g, head r%g); every row sees all prefix_tokens keys
// of the blocks that open table row 0; the output is a normalised fp32
// partial and its log2-sum-exp, merged into the decode result afterwards.
template <bool kPrefix>
__global__ void __launch_bounds__(kThreads, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
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
  const int b = blockIdx.z;
  const int g = p.Hq / p.Hkv;

  int q_begin = 0, Lk = 0;
  int qt[2], hd[2], rows[2], diag[2], nkt[2];
  int kvh;
  const int32_t* table;
  int kt0 = 0;   // first key tile of this block (shared-prefix mode splits the keys)
  if constexpr (kPrefix) {
    kvh = blockIdx.y;
    table = p.block_tables;
    const int R = p.B * g;
    Lk = p.prefix_tokens;
    kt0 = blockIdx.z * p.prefix_kt_per;
    const int n_here = min(p.prefix_kt_per, p.prefix_tokens / kN - kt0);
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      qt[x] = 2 * blockIdx.x + x;           // row tile of the group's B*g rows
      hd[x] = 0;
      rows[x] = max(0, min(kM, R - qt[x] * kM));
      diag[x] = INT32_MAX / 2;              // no mask
      nkt[x] = rows[x] > 0 ? max(n_here, 0) : 0;
    }
  } else {
    q_begin = p.cu_q[b];
    const int Lq = p.cu_q[b + 1] - q_begin;
    Lk = p.cu_k[b + 1] - p.cu_k[b];
    if (Lq < 0 || Lk < Lq || Lq > p.max_q || Lk > p.max_k ||
        static_cast<int64_t>(Lk) > static_cast<int64_t>(p.maxblk) * kBlockSize) {
      if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_error(p.err, kErrIndex);
      return;
    }
    // The two query tiles of this block; heavier (later) row tiles first.
    if (p.pair_heads) {
      qt[0] = qt[1] = p.n_qt - 1 - static_cast<int>(blockIdx.x);
      hd[0] = 2 * blockIdx.y;
      hd[1] = 2 * blockIdx.y + 1;
    } else {
      const int n_pairs = (p.n_qt + 1) / 2;
      qt[0] = 2 * (n_pairs - 1 - static_cast<int>(blockIdx.x));
      qt[1] = qt[0] + 1;
      hd[0] = hd[1] = blockIdx.y;
    }
    kvh = hd[0] / g;
    table = p.block_tables + static_cast<int64_t>(b) * p.maxblk;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int q0 = qt[x] * kM;
      rows[x] = q0 < Lq ? min(kM, Lq - q0) : 0;
      diag[x] = Lk - Lq + q0;                       // row i sees keys j <= diag + i
      nkt[x] = rows[x] > 0 ? (diag[x] + rows[x] - 1) / kN + 1 : 0;
    }
  }
  const int n_max = max(nkt[0], nkt[1]);
  if (n_max == 0) return;
  // (sequence, query head) of row i of tile x
  auto row_of = [&](int x, int i, int& rb, int& rh) {
    if constexpr (kPrefix) {
      const int gr = (x ? qt[1] : qt[0]) * kM + i;
      rb = gr / g;
      rh = kvh * g + gr % g;
    } else {
      rb = q_begin + (x ? qt[1] : qt[0]) * kM + i;   // row of q / out
      rh = x ? hd[1] : hd[0];
    }
  };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), (i == kBarPFull || i == kBarPFull + 1) ? 4 : 1);
    flags[0] = 0;  // abort
    flags[1] = 0;  // K tiles issued
    flags[2] = 0;  // V tiles issued
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + kOffTmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_map(&kmap);
    tma_prefetch_map(&vmap);
  }
  // Q tiles -> shared memory (K-major, 128-byte swizzle); rows past Lq are zero.
  if (warp < kSoftmaxWarps) {
    const int x = warp >> 2;
    const int i = tid & 127;
    const bool valid = i < (x ? rows[1] : rows[0]);
    int rb = 0, rh = 0;
    if (valid) row_of(x, i, rb, rh);
    const __nv_bfloat16* src = p.q + (static_cast<int64_t>(rb) * p.Hq + rh) * kHeadDim;
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (valid) v = __ldg(reinterpret_cast<const uint4*>(src) + cc);
      sts128(sbase + kOffQ + x * kTile + (cc >> 3) * kHalf + i * 128 +
                 (((cc & 7) ^ (i & 7)) << 4),
             v);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kt = 0;
      for (; kt < n_max && !flags[0]; ++kt) {
        const int st = kt & 1;
        const uint32_t ph = ((kt >> 1) - 1) & 1;
        const int gkt = kt0 + kt;   // key tile within the sequence
        int id = __ldg(table + (gkt >> 1));
        if (id < 0 || id >= p.num_blocks) {
          record_error(p.err, kErrIndex);
          id = 0;
        }
        const int slot = id * kBlockSize + (gkt & 1) * kN;
        if (kt >= 2 && !mbar_wait(bar(kBarKEmpty + st), ph)) break;
        const uint32_t kdst = sbase + kOffK + st * kTile;
        mbar_arrive_expect_tx(bar(kBarKFull + st), kTile);
        tma_load_3d(kdst, &kmap, bar(kBarKFull + st), 0, kvh, slot);
        tma_load_3d(kdst + kHalf, &kmap, bar(kBarKFull + st), 64, kvh, slot);
        flags[1] = kt + 1;
        if (kt >= 2 && !mbar_wait(bar(kBarVEmpty + st), ph)) break;
        const uint32_t vdst = sbase + kOffV + st * kTile;
        mbar_arrive_expect_tx(bar(kBarVFull + st), kTile);
        tma_load_3d(vdst, &vmap, bar(kBarVFull + st), 0, kvh, slot);
        tma_load_3d(vdst + kHalf, &vmap, bar(kBarVFull + st), 64, kvh, slot);
        flags[2] = kt + 1;
      }
      if (kt < n_max && !flags[0]) {
        record_error(p.err, kErrTimeout);
        flags[0] = 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kN, 0);        // B = K, K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(kM, kHeadDim, 1);  // B = V, MN-major
      auto issue_s = [&](int x, int kt) {
        const uint32_t q_s = sbase + kOffQ + x * kTile;
        const uint32_t k_s = sbase + kOffK + (kt & 1) * kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
          umma_bf16(tmem + kColS + x * kN, smem_desc_sw128(q_s + off, 16, 1024),
                    smem_desc_sw128(k_s + off, 16, 1024), idesc_s, ks > 0);
        }
      };
      auto issue_pv = [&](int x, int kt) {
        const uint32_t v_s = sbase + kOffV + (kt & 1) * kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          // A = P_x: 16 keys = 8 packed columns per step.  B = V: 64-dim boxes
          // kHalf apart (LBO), 8-key swizzle atoms 1024 bytes apart (SBO).
          umma_bf16_tmem_a(tmem + kColO + x * kHeadDim, tmem + kColS + x * kN + ks * 8,
                           smem_desc_sw128(v_s + ks * 2048, kHalf, 1024), idesc_o,
                           (kt > 0 || ks > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(kBarKFull + 0), 0);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if ((x ? nkt[1] : nkt[0]) > 0) {
            issue_s(x, 0);
            umma_commit(bar(kBarSFull + x));
          }
        umma_commit(bar(kBarKEmpty + 0));
      }
      for (int kt = 0; kt < n_max && ok && !flags[0]; ++kt) {
        const int st = kt & 1;
        const bool more = kt + 1 < nkt[0] || kt + 1 < nkt[1];
        bool k_next = false;
        if (!(ok = mbar_wait(bar(kBarVFull + st), (kt >> 1) & 1))) break;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int nx = x ? nkt[1] : nkt[0];
          if (!ok || kt >= nx) continue;
          if (!(ok = mbar_wait(bar(kBarPFull + x), kt & 1))) continue;
          tc_fence_after();
          issue_pv(x, kt);
          if (kt + 1 < nx) {
            if (!k_next) {
              if (!(ok = mbar_wait(bar(kBarKFull + ((kt + 1) & 1)), ((kt + 1) >> 1) & 1))) continue;
              tc_fence_after();
              k_next = true;
            }
            issue_s(x, kt + 1);
            umma_commit(bar(kBarSFull + x));
          } else {
            umma_commit(bar(kBarODone + x));
          }
        }
        if (!ok) break;
        umma_commit(bar(kBarVEmpty + st));
        if (more) umma_commit(bar(kBarKEmpty + ((kt + 1) & 1)));
      }
      if (!ok) {
        record_error(p.err, kErrTimeout);
        flags[0] = 1;
      }
      // every MMA issued so far has completed once this arrives
      umma_commit(bar(kBarDrain));
      (void)mbar_wait(bar(kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;               // query tile of this warpgroup
    const int i = tid & 127;               // query row within the tile = TMEM lane
    const int my_diag = x ? diag[1] : diag[0];
    const int my_rows = x ? rows[1] : rows[0];
    const int vis = my_diag + i;           // last visible key
    const int n = x ? nkt[1] : nkt[0];
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + kColS + x * kN;
    const uint32_t o_col = lane_base + kColO + x * kHeadDim;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int kt = 0; kt < n; ++kt) {
      if (flags[0]) { ok = false; break; }
      // S_x(kt) is complete, and so is every earlier MMA (PV_x(kt-1) included)
      if (!(ok = warp_wait(bar(kBarSFull + x), kt & 1))) break;
      tc_fence_after();
      // Pass 1: row max of the raw scores, 64 columns per TMEM round trip (the
      // scale is positive, so it is applied to the max afterwards).
      const int j0 = kt * kN;
      const bool edge = !kPrefix && j0 + kN - 1 > my_diag;   // causal edge inside this tile
      float smax = -INFINITY;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t r[64];
        tmem_ld64_wait(s_col + hh * 64, r);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float v = __uint_as_float(r[c]);
          smax = fmaxf(smax, (!edge || j0 + hh * 64 + c <= vis) ? v : -INFINITY);
        }
      }
      const float mt = smax * p.scale_log2;
      if (kt == 0) {
        m = mt;  // key 0 is visible to every row
      } else {
        const bool need = mt > m + kLazyRescale;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m - mt) : 1.f;
          if (need) {
            l *= alpha;
            m = mt;
          }
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t o[32];
            tmem_ld32_wait(o_col + c4 * 32, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(o_col + c4 * 32, o);
          }
        }
      }
      // Pass 2: P = 2^(scale*s - m) as bf16 pairs over the first 64 columns of
      // S_x: score columns [64hh, 64hh+64) become P columns [32hh, 32hh+32),
      // all of which have been read already.
      const float neg_m = -m;
      float rs = 0.f;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t r[64];
        tmem_ld64_wait(s_col + hh * 64, r);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k0 = j0 + hh * 64 + 2 * c;
          float e0 = ex2(fmaf(__uint_as_float(r[2 * c]), p.scale_log2, neg_m));
          float e1 = ex2(fmaf(__uint_as_float(r[2 * c + 1]), p.scale_log2, neg_m));
          if (edge) {
            e0 = k0 <= vis ? e0 : 0.f;
            e1 = k0 + 1 <= vis ? e1 : 0.f;
          }
          rs += e0 + e1;
          pk[c] = pack_bf16x2(e0, e1);
        }
        tmem_st32(s_col + hh * 32, pk);
      }
      l += rs;
      tmem_wait_st();
      // keys past the end of the sequence inside the last tile: zero their V
      // rows so that 0 * (stale data) cannot produce a NaN in O
      if (!kPrefix && kt == n - 1 && j0 + kN > Lk) {
        if (!(ok = warp_wait(bar(kBarVFull + (kt & 1)), (kt >> 1) & 1))) break;
        if (j0 + i >= Lk) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          const uint32_t vrow = sbase + kOffV + (kt & 1) * kTile + i * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            sts128(vrow + cc * 16, z);
            sts128(vrow + kHalf + cc * 16, z);
          }
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + x));
    }
    if (n > 0) {
      if (ok) ok = warp_wait(bar(kBarODone + x), 0);
      if (!ok) {
        if (lane == 0) {
          record_error(p.err, kErrTimeout);
          flags[0] = 1;
        }
      } else {
        tc_fence_after();
        const float inv = 1.f / l;
        const bool valid = i < my_rows;
        int rb = 0, rh = 0;
        if (valid) row_of(x, i, rb, rh);
        const int64_t row = static_cast<int64_t>(rb) * p.Hq + rh;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t r[32];
          tmem_ld32_wait(o_col + c4 * 32, r);
          if (!valid) continue;
          if constexpr (kPrefix) {
            const int64_t prow = row * gridDim.z + blockIdx.z;
            float4* dst = reinterpret_cast<float4*>(p.part_o + prow * kHeadDim) + c4 * 8;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                   __uint_as_float(r[4 * k + 2]) * inv,
                                   __uint_as_float(r[4 * k + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(p.out + row * kHeadDim) + c4 * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv,
                                __uint_as_float(r[8 * k + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv,
                                __uint_as_float(r[8 * k + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv,
                                __uint_as_float(r[8 * k + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv,
                                __uint_as_float(r[8 * k + 7]) * inv);
              dst[k] = v;
            }
          }
        }
        if (valid) {
          if constexpr (kPrefix) {
            p.part_lse[row * gridDim.z + blockIdx.z] = m + __log2f(l);
          } else {
            if (p.lse) p.lse[row] = (m + __log2f(l)) * kLn2;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // After an abort, wait (bounded) for any TMA copy that may still be landing.
  if (flags[0] && tid == kTmaWarp * 32) {
    const int kin = flags[1], vin = flags[2];
    for (int st = 0; st < 2; ++st) {
      for (int kt = kin - 1; kt >= 0; --kt)
        if ((kt & 1) == st) { (void)mbar_wait(bar(kBarKFull + st), (kt >> 1) & 1); break; }
      for (int kt = vin - 1; kt >= 0; --kt)
        if ((kt & 1) == st) { (void)mbar_wait(bar(kBarVFull + st), (kt >> 1) & 1); break; }
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
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

}  // namespace

int launch_prefill(const PrefillArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.B == 0 || a.max_seqlen_q == 0) return PKV_OK;
  CUtensorMap km, vm;
  const int64_t slots = a.num_blocks * kBlockSize;
  if (!encode_pool_map(&km, a.k_cache, slots, a.Hkv, kN) ||
      !encode_pool_map(&vm, a.v_cache, slots, a.Hkv, kN))
    return PKV_ERR_ARG;
  PrefillParams prm;
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
  prm.pair_heads = ((a.Hq / a.Hkv) % 2 == 0) ? 1 : 0;
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.part_o = nullptr;
  prm.part_lse = nullptr;
  prm.prefix_tokens = 0;
  if (!set_smem_attr<false>()) return PKV_ERR_LAUNCH;
  dim3 grid;
  if (prm.pair_heads)
    grid = dim3(prm.n_qt, a.Hq / 2, a.B);
  else
    grid = dim3((prm.n_qt + 1) / 2, a.Hq, a.B);
  paged_prefill_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int launch_prefix_attention(const PrefixArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.B == 0 || a.prefix_tokens == 0) return PKV_OK;
  CUtensorMap km, vm;
  const int64_t slots = a.num_blocks * kBlockSize;
  if (!encode_pool_map(&km, a.k_cache, slots, a.Hkv, kN) ||
      !encode_pool_map(&vm, a.v_cache, slots, a.Hkv, kN))
    return PKV_ERR_ARG;
  PrefillParams prm = {};
  prm.part_o = a.part_o;
  prm.part_lse = a.part_lse;
  prm.prefix_tokens = a.prefix_tokens;
  prm.prefix_kt_per = a.kt_per;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_tables = a.block_tables;
  prm.err = err;
  prm.B = a.B;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  if (!set_smem_attr<true>()) return PKV_ERR_LAUNCH;
  const int rows = a.B * (a.Hq / a.Hkv);
  const int tiles = (rows + kM - 1) / kM;
  dim3 grid((tiles + 1) / 2, a.Hkv, a.splits);
  paged_prefill_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv
