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
// One thread block computes a 128-row query tile of one (sequence, query head):
//   warp 4 (TMA)     streams 128-key K and V tiles of the kv head from the
//                    paged pool into two stages each (two 64-dim boxes per tile,
//                    128-byte swizzle).  A 128-key tile never straddles a
//                    256-token block.
//   warp 5 (MMA)     one lane issues S = Q K^T (M=N=128, K=128; tcgen05.mma
//                    kind::f16, bf16 in, fp32 out) into one of two TMEM score
//                    buffers, and O += P V into the TMEM output accumulator,
//                    signalling completion through tcgen05.commit -> mbarrier.
//                    S of tile t+1 is issued before PV of tile t, so the tensor
//                    core works on the next scores while softmax runs.
//   warps 0-3        thread i owns query row i: reads its score row from TMEM,
//                    applies the causal mask, keeps the running max / sum in
//                    base 2, rescales O in TMEM only when the max grew by more
//                    than 2^8 (otherwise the stale max is kept: p <= 256 stays
//                    exact enough in fp32 / bf16), writes P as bf16 into the
//                    swizzled K-major layout the PV product reads, and at the
//                    end normalises O and writes out / lse.
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
constexpr int kThreads = 6 * 32;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kHalf = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte swizzled box)
constexpr int kTile = 2 * kHalf;       // 128 rows x 128 bf16
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;   // 2 stages
constexpr int kOffV = kOffK + 2 * kTile;
constexpr int kOffP = kOffV + 2 * kTile;
constexpr int kOffBars = kOffP + kTile;
// barriers
constexpr int kBarKFull = 0;   // [2]
constexpr int kBarKEmpty = 2;  // [2]
constexpr int kBarVFull = 4;   // [2]
constexpr int kBarVEmpty = 6;  // [2]
constexpr int kBarSFull = 8;   // [2]
constexpr int kBarPFull = 10;
constexpr int kBarODone = 11;
constexpr int kBarDrain = 12;
constexpr int kNumBars = 13;
constexpr int kOffTmem = kOffBars + kNumBars * 8;
constexpr int kOffFlags = kOffTmem + 8;
constexpr int kSmemBytes = kOffFlags + 16 + 1024;
constexpr uint32_t kTmemCols = 512;    // S0 | S1 | O | unused
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr float kLazyRescale = 8.f;    // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

struct PrefillParams {
  __nv_bfloat16* out;
  float* lse;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* cu_q;
  const int32_t* cu_k;
  unsigned* err;
  int B, Hq, Hkv, maxblk, max_q, max_k;
  int64_t num_blocks;
  float scale_log2;
};

// Wait with every lane of the warp; the result is the same for all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

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
  const int qt = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / (p.Hq / p.Hkv);

  const int q_begin = p.cu_q[b];
  const int Lq = p.cu_q[b + 1] - q_begin;
  const int Lk = p.cu_k[b + 1] - p.cu_k[b];
  if (Lq < 0 || Lk < Lq || Lq > p.max_q || Lk > p.max_k ||
      static_cast<int64_t>(Lk) > static_cast<int64_t>(p.maxblk) * kBlockSize) {
    if (tid == 0 && qt == 0 && h == 0) record_error(p.err, kErrIndex);
    return;
  }
  const int tile_q0 = qt * kM;
  if (tile_q0 >= Lq) return;
  const int rows = min(kM, Lq - tile_q0);
  const int diag = Lk - Lq + tile_q0;   // row i sees keys j <= diag + i
  const int n_kt = (diag + rows - 1) / kN + 1;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), i == kBarPFull ? 4 : 1);
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
  // Q tile -> shared memory (K-major, 128-byte swizzle); rows past Lq are zero.
  if (warp < 4) {
    const int i = tid;
    const bool valid = i < rows;
    const __nv_bfloat16* src =
        p.q + (static_cast<int64_t>(q_begin + tile_q0 + i) * p.Hq + h) * kHeadDim;
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (valid) v = __ldg(reinterpret_cast<const uint4*>(src) + cc);
      const uint32_t dst = sbase + kOffQ + (cc >> 3) * kHalf + i * 128 +
                           ((((cc & 7) ^ (i & 7))) << 4);
      sts128(dst, v);
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
      const int32_t* table = p.block_tables + static_cast<int64_t>(b) * p.maxblk;
      int kt = 0;
      for (; kt < n_kt && !flags[0]; ++kt) {
        const int st = kt & 1;
        const uint32_t ph = ((kt >> 1) - 1) & 1;
        int id = __ldg(table + (kt >> 1));
        if (id < 0 || id >= p.num_blocks) {
          record_error(p.err, kErrIndex);
          id = 0;
        }
        const int slot = id * kBlockSize + (kt & 1) * kN;
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
      if (kt < n_kt && !flags[0]) {
        record_error(p.err, kErrTimeout);
        flags[0] = 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kN, 0);        // B = K, K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(kM, kHeadDim, 1);  // B = V, MN-major
      const uint32_t q_s = sbase + kOffQ;
      const uint32_t p_s = sbase + kOffP;
      bool ok = true;
      for (int kt = 0; kt <= n_kt && ok && !flags[0]; ++kt) {
        if (kt < n_kt) {
          const int st = kt & 1;
          if (!(ok = mbar_wait(bar(kBarKFull + st), (kt >> 1) & 1))) break;
          tc_fence_after();
          const uint32_t k_s = sbase + kOffK + st * kTile;
          const uint32_t d = tmem + kColS + st * kN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
            umma_bf16(d, smem_desc_sw128(q_s + off, 16, 1024),
                      smem_desc_sw128(k_s + off, 16, 1024), idesc_s, ks > 0);
          }
          umma_commit(bar(kBarSFull + st));
          umma_commit(bar(kBarKEmpty + st));
        }
        if (kt >= 1) {
          const int j = kt - 1;
          const int st = j & 1;
          if (!(ok = mbar_wait(bar(kBarPFull), j & 1))) break;
          if (!(ok = mbar_wait(bar(kBarVFull + st), (j >> 1) & 1))) break;
          tc_fence_after();
          const uint32_t v_s = sbase + kOffV + st * kTile;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // A = P (K-major over keys), B = V (MN-major: 64-dim boxes kHalf
            // apart, 8-key swizzle atoms 1024 bytes apart; 16 keys per step).
            umma_bf16(tmem + kColO, smem_desc_sw128(p_s + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024),
                      smem_desc_sw128(v_s + ks * 2048, kHalf, 1024), idesc_o,
                      (j > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(bar(kBarODone));
          umma_commit(bar(kBarVEmpty + st));
        }
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
    const int i = tid;                 // query row within the tile = TMEM lane
    const int vis = diag + i;          // last visible key
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int kt = 0; kt < n_kt; ++kt) {
      if (flags[0]) { ok = false; break; }
      const int sb = kt & 1;
      if (!(ok = warp_wait(bar(kBarSFull + sb), (kt >> 1) & 1))) break;
      tc_fence_after();
      float s[kN];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t r[32];
        tmem_ld32(lane_base + kColS + sb * kN + c4 * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c4 * 32 + c] = __uint_as_float(r[c]) * p.scale_log2;
      }
      const int j0 = kt * kN;
      float mt = -INFINITY;
      if (j0 + kN - 1 > diag) {  // causal edge inside this tile
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          s[c] = (j0 + c <= vis) ? s[c] : -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kN; ++c) mt = fmaxf(mt, s[c]);
      }
      if (kt == 0) {
        m = mt;  // key 0 is visible to every row
      } else {
        // PV of the previous tile must be done before O is rescaled or P reused
        if (!(ok = warp_wait(bar(kBarODone), (kt - 1) & 1))) break;
        tc_fence_after();
        const bool need = mt > m + kLazyRescale;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m - mt) : 1.f;
          if (need) {
            l *= alpha;
            m = mt;
          }
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t r[32];
            tmem_ld32(lane_base + kColO + c4 * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tmem_st32(lane_base + kColO + c4 * 32, r);
          }
          tmem_wait_st();
        }
      }
      // P = 2^(s - m) as bf16 into the swizzled K-major layout
      float rs = 0.f;
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          e[k] = ex2(s[cc * 8 + k] - m);
          rs += e[k];
        }
        uint4 v;
        v.x = pack_bf16x2(e[0], e[1]);
        v.y = pack_bf16x2(e[2], e[3]);
        v.z = pack_bf16x2(e[4], e[5]);
        v.w = pack_bf16x2(e[6], e[7]);
        sts128(sbase + kOffP + (cc >> 3) * kHalf + i * 128 + (((cc & 7) ^ (i & 7)) << 4), v);
      }
      l += rs;
      // keys past the end of the sequence inside the last tile: zero their V
      // rows so that 0 * (stale data) cannot produce a NaN in O
      if (kt == n_kt - 1 && j0 + kN > Lk) {
        if (!(ok = warp_wait(bar(kBarVFull + sb), (kt >> 1) & 1))) break;
        if (j0 + i >= Lk) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            sts128(sbase + kOffV + sb * kTile + i * 128 + cc * 16, z);
            sts128(sbase + kOffV + sb * kTile + kHalf + i * 128 + cc * 16, z);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
    }
    if (ok) ok = warp_wait(bar(kBarODone), (n_kt - 1) & 1);
    if (!ok) {
      if (lane == 0) {
        record_error(p.err, kErrTimeout);
        flags[0] = 1;
      }
    } else {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool valid = i < rows;
      __nv_bfloat16* dst =
          p.out + (static_cast<int64_t>(q_begin + tile_q0 + i) * p.Hq + h) * kHeadDim;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t r[32];
        tmem_ld32(lane_base + kColO + c4 * 32, r);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv);
            reinterpret_cast<uint4*>(dst)[c4 * 4 + k] = v;
          }
        }
      }
      if (valid && p.lse)
        p.lse[static_cast<int64_t>(q_begin + tile_q0 + i) * p.Hq + h] = (m + __log2f(l)) * kLn2;
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
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return PKV_ERR_LAUNCH;
    attr_set[dev] = true;
  }
  dim3 grid((a.max_seqlen_q + kM - 1) / kM, a.Hq, a.B);
  paged_prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv
