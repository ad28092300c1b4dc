// decode.cu — paged decode attention (split-K flash-decoding) for sm_103a.
//
// Operation: "During decode, gathers all cached K/V from paged blocks before
// calling scaled_dot_product_attention" (Nano-vLLM System Architecture
// Analysis, §2 Core Components, "Attention with Paged Cache"), GQA per §6.
// Decode is the memory-bound phase (same page, "Differences", §3 "Prefill vs.
// Decode Separation"), so this kernel never materialises the gathered K/V: it
// streams each sequence's blocks straight from the pool once.
//
// Work decomposition
//   grid = (S splits, Hkv * head_groups, B).  One thread block owns one
//   (sequence, kv head, range of whole KV blocks) and serves the G query heads
//   of that kv head's group that it is assigned, so each K/V byte is read from
//   HBM once per G heads.
//   The range's K and V stream through a ring of shared-memory stages with
//   TMA (64 tokens x 128 dims per stage, 128-byte swizzle) and mbarrier
//   completion: bf16 pools 3 stages, each operand two 64-dim boxes; E4M3
//   pools (one byte per element) one 128-byte box per operand, 4 stages (or
//   6 with a producer warp, below).
//   Copies: a fifth warp (the producer) copies whole stages and refills each
//   one as soon as every consumer warp has released it (bf16 pools, and E4M3
//   pools with splits of 8 blocks or more); otherwise (E4M3, shorter splits,
//   three blocks per SM) lane 0 of the issuing consumer warps copies one box
//   each and refills the stage released one tile earlier.
//   Four warps consume, warp w taking tokens [16w, 16w+16) of every stage.
//   Both contractions run on the warp-level tensor-core MMA (m16n8k16,
//   16-bit operands, fp32 accumulation) with the G query heads as MMA rows:
//   scores = q K^T straight from the stage (bf16 words as they are; E4M3
//   pairs converted to f16 pairs, exactly), an online softmax per row, then
//   o += P V with V pairs formed by byte permutes.  The MMA rows past the
//   heads carry the rounded remainder of the weights, so P enters with about
//   16 (bf16) or 22 (f16) significant bits.
//   End of the range: the four warps' streams are merged by log-sum-exp
//   through shared memory.  With one split the block writes out/lse
//   directly.  Otherwise it writes a normalised partial (o, log2-sum-exp) to
//   the workspace and takes a ticket from the (sequence, head group)
//   counter; the last block to arrive merges all partials with a
//   warp-shuffle log-sum-exp reduction, writes out/lse and resets the
//   counter, so nothing ever spins.
// Scores are kept in base-2 units (the score multiplier includes log2(e))
// and converted to a natural-log LSE on output.

#include <cuda_bf16.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kTile = 64;                       // tokens per pipeline stage
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = kConsumerWarps * 32;
static_assert(kConsumerWarps == 4, "each warp loads one quarter (K or V, one 64-dim half) of a stage");
constexpr int kHalfBytes = kTile * 128;         // 64 rows x 64 dims x 2 B
constexpr int kOperandBytes = 2 * kHalfBytes;   // one of K or V for a tile
constexpr int kStageBytes = 2 * kOperandBytes;  // K and V
constexpr int kMaxSplitBlocks = 32;             // block ids prefetched per split
constexpr int kMaxSplits = 1024;
// Arrival counters live in a fixed region at the start of the workspace, the
// same for every call shape, so partial results of one call can never land
// where another call keeps its counters.
constexpr size_t kCounterRegion = size_t(1) << 20;
constexpr int64_t kMaxCounters = kCounterRegion / sizeof(unsigned);
constexpr float kLn2 = 0.69314718055994530942f;

struct DecodeParams {
  __nv_bfloat16* out;
  float* lse;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_o;        // [B*Hq, S, 128] normalised partial outputs
  float* ws_lse;      // [B*Hq, S] partial log2-sum-exp
  unsigned* ws_count; // [B * Hkv * head_groups] arrival counters
  unsigned* err;
  // Hq counts "virtual" heads: q_len query positions x the physical heads;
  // virtual head v of kv head kv is position (v%g)/(g/q_len), head
  // kv*(g/q_len) + (v%g)%(g/q_len), with g = Hq/Hkv.  q_len = 1 is plain decode.
  int B, Hq, Hkv, maxblk, num_splits, split_tokens, head_groups;
  int q_len, Hq_phys;
  float k_scale, v_scale;   // FP8 pools: element value = code value * scale
  int64_t num_blocks;
  float scale_log2;
  // Shared prefix (0 = none): every sequence's first prefix_tokens tokens are
  // the same physical blocks, already reduced to one normalised partial per
  // (sequence, query head); this kernel then covers [prefix_tokens, ctx) only
  // and folds that partial into its merge.
  int prefix_tokens;
  int metadata_ready;       // tables and lengths may be read before the dependency wait
  int prefix_splits;        // partials per row of the shared-prefix pass
  const float* prefix_o;    // [B*Hq, prefix_splits, 128]
  const float* prefix_lse;  // [B*Hq, prefix_splits] log2-sum-exp
  // Fused store (new_slots == nullptr: none): the new token of sequence b,
  // bf16 rows k_new / v_new + b * stride, goes to slot new_slots[b].
  const int32_t* new_slots;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t k_new_stride, v_new_stride;  // elements
  uint4* k_pool;                       // the pools, writable
  uint4* v_pool;
  float k_inv, v_inv;                  // E4M3 pools: binary32 1/k_scale, 1/v_scale
};

// Log-sum-exp merge of one output row by one warp: nsplit partials
// (lse2[s], o[s][128]) of the row's own tokens plus np partials of a shared
// prefix, all normalised.  Lanes run over partials for the max and the sum
// (warp shuffles), then over dims (4 each) for the weighted sum, eight
// partials at a time so that their loads are in flight together.
__device__ __forceinline__ void merge_row(const float* lrow, const float* orow, int nsplit,
                                          const float* plrow, const float* porow, int np,
                                          __nv_bfloat16* out, float* lse, int lane) {
  float mx = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) mx = fmaxf(mx, __ldcg(lrow + s));
  for (int s = lane; s < np; s += 32) mx = fmaxf(mx, __ldcg(plrow + s));
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
  float sum = 0.f;
  for (int s = lane; s < nsplit; s += 32) sum += ex2(__ldcg(lrow + s) - mx);
  for (int s = lane; s < np; s += 32) sum += ex2(__ldcg(plrow + s) - mx);
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
  const float inv = 1.f / sum;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](const float* lr, const float* orr, int n) {
    for (int s0 = 0; s0 < n; s0 += 8) {
      float l8[8];
      float4 v8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (s0 + k < n) {
          l8[k] = __ldcg(lr + s0 + k);
          v8[k] = __ldcg(reinterpret_cast<const float4*>(orr + (s0 + k) * kHeadDim) + lane);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (s0 + k < n) {
          const float w = ex2(l8[k] - mx) * inv;
          acc.x = fmaf(w, v8[k].x, acc.x);
          acc.y = fmaf(w, v8[k].y, acc.y);
          acc.z = fmaf(w, v8[k].z, acc.z);
          acc.w = fmaf(w, v8[k].w, acc.w);
        }
      }
    }
  };
  add(plrow, porow, np);
  add(lrow, orow, nsplit);
  __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo2);
  packed.y = *reinterpret_cast<uint32_t*>(&hi2);
  *reinterpret_cast<uint2*>(out + 4 * lane) = packed;
  if (lse && lane == 0) *lse = (mx + __log2f(sum)) * 0.69314718055994530942f;
}

// Pipeline geometry per element type.  bf16: 3 stages of 64 tokens, each
// operand two 64-dim boxes (four copies per stage).  FP8 (E4M3, one byte per
// element): a row of 128 dims is one 128-byte box, so a stage of 64 tokens
// holds 16 KB; without a producer warp, 4 stages (64 KB) let three blocks
// share an SM and warps 0 and 1 issue the K and the V copy of each stage;
// with one (kProd), 6 stages at two blocks per SM (the fifth warp's registers
// leave no room for a third block).  bf16 without a producer warp (batches
// split into 64-token tiles, one or a few per block): 2 stages, three blocks
// per SM, so that all of such a batch's blocks are resident at once.  bf16
// with two consumer groups (kGroups = 2: one block per SM, batches whose
// one-split grid fits one wave): 6 stages; an even count keeps each stage's
// tiles in one group (see the consumer notes in the kernel).
template <bool kFp8, bool kProd = false, int kGroups = 1>
struct Geo {
  static_assert(kGroups == 1 || (kGroups == 2 && kProd && !kFp8), "two groups: bf16, producer warp");
  static constexpr int kStagesN = kGroups == 2 ? 6 : kFp8 ? (kProd ? 6 : 4) : (kProd ? 3 : 2);
  static_assert(kGroups == 1 || kStagesN % 2 == 0, "two groups need an even stage count");
  static constexpr int kOpBytes = kTile * (kFp8 ? 128 : 256);  // one of K or V for a stage
  static constexpr int kStageB = 2 * kOpBytes;
  static constexpr int kIssuers = kFp8 ? 2 : 4;
};
static_assert(Geo<false, true>::kStagesN == kStages && Geo<false, true>::kStageB == kStageBytes,
              "geometry");

template <int G, bool kFp8 = false, bool kProd = false, int kGroups = 1>
struct SmemLayout {
  static constexpr int kStages = Geo<kFp8, kProd, kGroups>::kStagesN;
  static constexpr int kStageBytes = Geo<kFp8, kProd, kGroups>::kStageB;
  static constexpr int kCW = kConsumerWarps * kGroups;   // consumer warps
  // [kCW][G][128] f32, over the stage ring: written only once every warp is
  // done with the stages and no copy is in flight
  static constexpr int kMergeO = 0;
  static_assert(kCW * G * 128 * 4 <= kStages * kStageBytes, "merge buffer");
  static constexpr int kMergeM = kStages * kStageBytes;                      // [kCW][G]
  static constexpr int kMergeL = kMergeM + kCW * G * 4;                      // [kCW][G]
  static constexpr int kBlk = kMergeL + kCW * G * 4;                         // [32] int
  static constexpr int kBars = kBlk + kMaxSplitBlocks * 4;                   // full[], empty[]
  static constexpr int kFlags = kBars + (2 * kStages + 1) * 8;  // + stored; abort, last, issued
  static constexpr int kEnd = kFlags + 16;
  static constexpr int kBytes = kEnd + 1024;                                 // + alignment slack
};

// Weight of a stream with log2-max m against the common max mn (0 for an
// empty stream).
__device__ __forceinline__ float rescale(float m, float mn) {
  return m == -INFINITY ? 0.f : ex2(m - mn);
}

// A operand of the score MMA for the lane's row gq from its 16 words of q
// (bf16 pairs of dims [32c, 32c+32)), and the multiplier that turns a raw
// score into the log2 domain.  bf16 pools: the words as they are.  E4M3
// pools: q goes to f16 scaled by the power of two that brings its row maximum
// into [2^14, 2^15), where every bf16 element down to 2^-32 of that maximum
// converts exactly; the multiplier undoes that power and applies k_scale.
// Every lane of the warp takes part (row maxima by shuffles).
template <bool kFp8>
__device__ __forceinline__ void q_fragments(const uint32_t (&qw)[16], float scale_log2,
                                            float k_scale, uint32_t (&qa)[8][2], float& qmul) {
  if constexpr (kFp8) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(bf16lo(qw[i])), fabsf(bf16hi(qw[i]))));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // amax = f * 2^e, f in [0.5, 1) (e = -126 for zero and subnormals)
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 126;
    const int sh = min(15 - e, 100);
    const float up = __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
    qmul = scale_log2 * k_scale * __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      qa[m][0] = pack_f16x2(bf16lo(qw[2 * m]) * up, bf16hi(qw[2 * m]) * up);
      qa[m][1] = pack_f16x2(bf16lo(qw[2 * m + 1]) * up, bf16hi(qw[2 * m + 1]) * up);
    }
  } else {
    qmul = scale_log2;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      qa[m][0] = qw[2 * m];
      qa[m][1] = qw[2 * m + 1];
    }
  }
}

// One 64-token stage consumed by one warp (see the consumer notes in the
// kernels below): the scores of the warp's 16 tokens [16 warp, 16 warp + 16)
// against the G query rows, the online-softmax update of (m_run, l_run, o) and
// o += P V.  kb / vb: shared addresses of the stage's K and V.  n_valid: tokens
// of the stage inside the key range.  lim (several query positions only): keys
// that row gq may see, counted from the stage's first token.
template <int G, bool kMQ, bool kFp8>
__device__ __forceinline__ void consume_stage(uint32_t kb, uint32_t vb, int warp, int gq, int c,
                                              const uint32_t (&qa)[8][2], float qmul,
                                              int n_valid, int lim, float (&o)[16][4],
                                              float& m_run, float& l_run) {
  const int t0 = 16 * warp;

  // scores of token groups n = 0, 1: row (token) t0 + 8n + gq; a
  // 128-byte row's 16-byte chunk j sits at chunk j ^ (row & 7) = j ^ gq
  float sc[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    uint32_t kw[16];
    if constexpr (kFp8) {
      const uint32_t row = kb + (t0 + 8 * n + gq) * 128;
      const uint4 k0 = lds128(row + (((2 * c) ^ gq) << 4));
      const uint4 k1 = lds128(row + (((2 * c + 1) ^ gq) << 4));
      const uint32_t w[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        kw[2 * i] = e4m3x2_lo_to_f16x2(w[i]);
        kw[2 * i + 1] = e4m3x2_hi_to_f16x2(w[i]);
      }
    } else {
      // dims [32c, 32c+32): half c >> 1, chunks 4 (c & 1) .. + 3
      const uint32_t row = kb + (c >> 1) * kHalfBytes + (t0 + 8 * n + gq) * 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = lds128(row + (((4 * (c & 1) + i) ^ gq) << 4));
        kw[4 * i] = u.x;
        kw[4 * i + 1] = u.y;
        kw[4 * i + 2] = u.z;
        kw[4 * i + 3] = u.w;
      }
    }
    sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int mm = 0; mm < 8; ++mm)
      mma_16x8x16<kFp8>(sc[n], qa[mm][0], 0u, qa[mm][1], 0u, kw[2 * mm], kw[2 * mm + 1]);
  }
  // online softmax of row gq over the warp's 16 tokens; this lane has
  // tokens t0 + 8 (i >> 1) + 2c + (i & 1), i = 0..3
  bool ok[4];
  float sv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 8 * (i >> 1) + 2 * c + (i & 1);
    ok[i] = t < n_valid && (!kMQ || t < lim);
    sv[i] = ok[i] ? sc[i >> 1][i & 1] * qmul : -INFINITY;
  }
  float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
  mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
  // the running max moves only when the tile's exceeds it by 2^8; below
  // that the weights stay within 256 and o is not rescaled
  if (mt > m_run + 8.f) {
    const float alpha = rescale(m_run, mt);
    l_run *= alpha;
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) {
      o[jn][0] *= alpha;
      o[jn][1] *= alpha;
      o[jn][2] *= alpha;
      o[jn][3] *= alpha;
    }
    m_run = mt;
  }
  float pw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    pw[i] = ok[i] ? ex2(sv[i] - m_run) : 0.f;
    l_run += pw[i];
  }
  // A operand of P V: k positions 2c, 2c+1 are tokens t0 + 2c, +1 (a0 / a1)
  // and 2c+8, 2c+9 tokens t0 + 8 + 2c, +1 (a2 / a3)
  uint32_t ph0, pl0, ph2, pl2;
  split_pair<kFp8>(pw[0], pw[1], ph0, pl0);
  split_pair<kFp8>(pw[2], pw[3], ph2, pl2);

  // values: this lane gives B column gq at k positions 2c, 2c+1 (tokens
  // A, B) and 2c+8, 2c+9 (tokens C, D).  Tokens past the context are
  // zeroed: stale slots may hold NaN patterns.
  if constexpr (kFp8) {
    // column gq of n-tile jn is dim 16 gq + jn: byte jn of the chunk
    uint32_t vw[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = t0 + 8 * (k >> 1) + 2 * c + (k & 1);
      uint4 v = lds128(vb + t * 128 + ((gq ^ (t & 7)) << 4));
      if (t >= n_valid) v = make_uint4(0u, 0u, 0u, 0u);
      vw[k][0] = v.x;
      vw[k][1] = v.y;
      vw[k][2] = v.z;
      vw[k][3] = v.w;
    }
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      // bytes 4wi..4wi+3 of two tokens interleaved: n-tiles 4wi..4wi+3
      const uint32_t ab01 = __byte_perm(vw[0][wi], vw[1][wi], 0x5140);
      const uint32_t ab23 = __byte_perm(vw[0][wi], vw[1][wi], 0x7362);
      const uint32_t cd01 = __byte_perm(vw[2][wi], vw[3][wi], 0x5140);
      const uint32_t cd23 = __byte_perm(vw[2][wi], vw[3][wi], 0x7362);
      mma_16x8x16<true>(o[4 * wi], ph0, pl0, ph2, pl2, e4m3x2_lo_to_f16x2(ab01),
                        e4m3x2_lo_to_f16x2(cd01));
      mma_16x8x16<true>(o[4 * wi + 1], ph0, pl0, ph2, pl2, e4m3x2_hi_to_f16x2(ab01),
                        e4m3x2_hi_to_f16x2(cd01));
      mma_16x8x16<true>(o[4 * wi + 2], ph0, pl0, ph2, pl2, e4m3x2_lo_to_f16x2(ab23),
                        e4m3x2_lo_to_f16x2(cd23));
      mma_16x8x16<true>(o[4 * wi + 3], ph0, pl0, ph2, pl2, e4m3x2_hi_to_f16x2(ab23),
                        e4m3x2_hi_to_f16x2(cd23));
    }
  } else {
    // dims [16 gq, 16 gq + 16): half gq >> 2, chunks 2 (gq & 3) + {0, 1},
    // the two loaded in the order (gq & 1, 1 - (gq & 1)) so that each load
    // instruction touches all eight chunk positions; load i then holds
    // dims 16 gq + 8 (i ^ (gq & 1)) + 0..7, and column gq of n-tile jn is
    // dim 16 gq + (jn ^ 8 (gq & 1))
    uint32_t vw[4][8];
    const uint32_t vhalf = vb + (gq >> 2) * kHalfBytes;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = t0 + 8 * (k >> 1) + 2 * c + (k & 1);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int chunk = 2 * (gq & 3) + (i ^ (gq & 1));
        uint4 v = lds128(vhalf + t * 128 + ((chunk ^ (t & 7)) << 4));
        if (t >= n_valid) v = make_uint4(0u, 0u, 0u, 0u);
        vw[k][4 * i] = v.x;
        vw[k][4 * i + 1] = v.y;
        vw[k][4 * i + 2] = v.z;
        vw[k][4 * i + 3] = v.w;
      }
    }
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) {
      // word jn >> 1 holds the dims 2 (jn >> 1), +1 of load jn >> 3
      const uint32_t sel = (jn & 1) ? 0x7632u : 0x5410u;
      const uint32_t b0 = __byte_perm(vw[0][jn >> 1], vw[1][jn >> 1], sel);
      const uint32_t b1 = __byte_perm(vw[2][jn >> 1], vw[3][jn >> 1], sel);
      mma_16x8x16<false>(o[jn], ph0, pl0, ph2, pl2, b0, b1);
    }
  }
}

// Fused store, by one whole warp: the new token's row of kv head kvh0 goes to
// slot sl, which must be the slot of position pos = ctx - 1 (block blk of the
// sequence's table): no other range reads it, and blocks of other head
// groups write the same bytes.  Any other slot is reported and not written.
// bf16: lanes 0-15 copy the K row, 16-31 the V row, 16 bytes each.  E4M3:
// lanes 0-7 quantize 16 elements of the K row, 8-15 of the V row, exactly as
// kv_cache_store_fp8 does (fp32 product with the binary32 reciprocal scale,
// nearest code, ties to even, saturating).  Each writing lane then orders its
// write before later tensor copies (async proxy) of the same bytes.
template <bool kFp8>
__device__ __forceinline__ void store_new_row(const DecodeParams& p, int b, int kvh0, int sl,
                                              int blk, int pos, int lane) {
  if (sl != blk * kBlockSize + pos % kBlockSize) {
    if (lane == 0) record_error(p.err, kErrIndex);
    return;
  }
  const int64_t row_idx = static_cast<int64_t>(sl) * p.Hkv + kvh0;
  if constexpr (kFp8) {
    if (lane < 16) {
      const bool is_k = lane < 8;
      const __nv_bfloat16* row = is_k ? p.k_new + b * p.k_new_stride
                                      : p.v_new + b * p.v_new_stride;
      const uint4* src = reinterpret_cast<const uint4*>(row + kvh0 * kHeadDim) + 2 * (lane & 7);
      const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
      const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const float inv = is_k ? p.k_inv : p.v_inv;
      uint32_t cw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c0 = e4m3x2_from_f32(bf16lo(w[2 * j]) * inv, bf16hi(w[2 * j]) * inv);
        const uint32_t c1 =
            e4m3x2_from_f32(bf16lo(w[2 * j + 1]) * inv, bf16hi(w[2 * j + 1]) * inv);
        cw[j] = c0 | (c1 << 16);
      }
      uint4* pool = is_k ? p.k_pool : p.v_pool;
      pool[row_idx * (kHeadDim / 16) + (lane & 7)] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      fence_proxy_async_global();
    }
  } else {
    const __nv_bfloat16* row = lane < 16 ? p.k_new + b * p.k_new_stride
                                         : p.v_new + b * p.v_new_stride;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + kvh0 * kHeadDim) + (lane & 15));
    uint4* pool = lane < 16 ? p.k_pool : p.v_pool;
    pool[row_idx * (kHeadDim / 8) + (lane & 15)] = v;
    fence_proxy_async_global();
  }
}

// kMQ: several query positions per sequence (q_len > 1); plain decode
// compiles without the per-row key limits.  kFp8: E4M3 pools.  kProd: a fifth
// warp issues every copy, so that no consumer warp waits for the others to
// release a stage before its next tile.  One kv head per block; G of its
// query heads.
template <int G, bool kMQ, bool kFp8, bool kProd, int kGroups = 1>
__global__ void __launch_bounds__(kProd ? kThreads * kGroups + 32 : kThreads,
                                  kGroups == 2 ? 1 : (kProd ? 2 : 3))
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using L = SmemLayout<G, kFp8, kProd, kGroups>;
  constexpr int kStagesN = Geo<kFp8, kProd, kGroups>::kStagesN;
  constexpr int kStageB = Geo<kFp8, kProd, kGroups>::kStageB;
  constexpr int kOpBytes = Geo<kFp8, kProd, kGroups>::kOpBytes;
  constexpr int kIssuers = Geo<kFp8, kProd, kGroups>::kIssuers;
  constexpr int kCW = L::kCW;   // consumer warps
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* merge_o = reinterpret_cast<float*>(smem + L::kMergeO);
  float* merge_m = reinterpret_cast<float*>(smem + L::kMergeM);
  float* merge_l = reinterpret_cast<float*>(smem + L::kMergeL);
  int* sblk = reinterpret_cast<int*>(smem + L::kBlk);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L::kFlags);
  const uint32_t bars = smem_addr(smem + L::kBars);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStagesN + s); };
  const uint32_t stored_bar = bars + 8u * (2 * kStagesN);  // fused store: the new row written

  // The tensor maps are launch parameters, which no earlier kernel writes:
  // fetch them into the SM's descriptor cache before waiting, so that the
  // block's first copy does not wait for them.
  if (threadIdx.x == 0) {
    tma_prefetch_map(&kmap);
    tma_prefetch_map(&vmap);
  }
  // Programmatic dependent launch: the next kernel of the stream may be
  // scheduled once every block of this one has started, and this kernel
  // reads no global memory before the grids it depends on have completed
  // (with metadata_ready: none but block_tables and context_lens, which the
  // caller wrote before those grids; the wait then follows the block's
  // early exit below, before anything else is read or written).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!p.metadata_ready) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int split = blockIdx.x;
  const int hg = blockIdx.y;  // kv head * head_groups + query head group
  const int b = blockIdx.z;
  const int g = p.Hq / p.Hkv;
  const int kvh0 = hg / p.head_groups;           // the block's kv head
  const int hoff = (hg % p.head_groups) * G;     // first query head within its group
  auto qhead = [&](int h) { return kvh0 * g + hoff + h; };
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Block ids of this split's whole range, loaded speculatively (they do not
  // depend on the context length, so both loads are in flight together).  A
  // range is whole blocks, or (small batches) whole 64-token tiles, which may
  // start inside a block and so touch one block more.
  const int split_tokens = p.split_tokens;
  const int blk_begin = (p.prefix_tokens + split * split_tokens) / kBlockSize;
  const int range_blocks = split_tokens % kBlockSize == 0 ? split_tokens / kBlockSize
                                                          : split_tokens / kBlockSize + 2;
  int spec_id = 0;
  if (warp == 0 && lane < range_blocks && blk_begin + lane < p.maxblk)
    spec_id = __ldg(p.block_tables + static_cast<int64_t>(b) * p.maxblk + blk_begin + lane);
  // Context of this sequence (clamped to what its block table can address).
  int ctx = p.context_lens[b];
  const int cap = p.maxblk * kBlockSize;
  const int P = p.prefix_tokens;
  if (ctx < 0 || ctx > cap || ctx < P) {
    if (tid == 0 && split == 0 && hg == 0) record_error(p.err, kErrIndex);
    ctx = ctx < P ? P : cap;
  }
  // several query positions: every one of the q_len new tokens is in the cache
  if (kMQ && ctx < p.q_len && tid == 0 && split == 0 && hg == 0) record_error(p.err, kErrIndex);
  // row of q / out / lse for virtual head v, and the number of keys it sees
  // (position i of q_len sees keys j < ctx - q_len + 1 + i)
  const int gp = g / p.q_len;
  auto phys_row = [&](int v) -> int64_t {
    if (!kMQ) return static_cast<int64_t>(b) * p.Hq + v;
    const int kv = v / g, r = v - kv * g;
    return (static_cast<int64_t>(b) * p.q_len + r / gp) * p.Hq_phys + kv * gp + r % gp;
  };
  auto key_limit = [&](int v) -> int {
    if (!kMQ) return ctx;
    return ctx - (p.q_len - 1 - (v % g) / gp);
  };
  const int nsplit = (ctx - P + split_tokens - 1) / split_tokens;
  if (split >= (nsplit > 0 ? nsplit : 1)) return;  // whole block exits: no work
  if (p.metadata_ready) asm volatile("griddepcontrol.wait;" ::: "memory");

  // Fused store: the blocks of a sequence's last range write the step's new
  // token (see below); a sequence with no token to attend takes none.
  const bool store_here = p.new_slots != nullptr && split == (nsplit > 0 ? nsplit : 1) - 1;
  if (store_here && ctx == P && tid == 0 && __ldg(p.new_slots + b) >= 0)
    record_error(p.err, kErrIndex);

  if (P > 0 && split == 0 && hg == 0 && warp == 0) {
    // the shared prefix must be the same physical blocks as sequence 0's
    const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.maxblk;
    bool same = true;
    for (int i = lane; i < P / kBlockSize; i += 32) same &= row[i] == p.block_tables[i];
    if (!__all_sync(0xffffffffu, same) && lane == 0) record_error(p.err, kErrIndex);
  }

  if (ctx == P) {  // nothing past the prefix: out = the prefix's result (or 0, -inf)
    if (P > 0) {
      for (int r = warp; r < G && warp < kConsumerWarps; r += kConsumerWarps) {
        const int64_t row = static_cast<int64_t>(b) * p.Hq + qhead(r);
        const int np = p.prefix_splits;
        const int64_t prow = phys_row(qhead(r));
        merge_row(nullptr, nullptr, 0, p.prefix_lse + row * np, p.prefix_o + row * np * kHeadDim,
                  np, p.out + prow * kHeadDim, p.lse ? p.lse + prow : nullptr, lane);
      }
      return;
    }
    for (int i = tid; i < G * kHeadDim; i += blockDim.x) {
      const int r = i / kHeadDim, d = i % kHeadDim;
      p.out[phys_row(qhead(r)) * kHeadDim + d] = __float2bfloat16_rn(0.f);
    }
    if (p.lse && tid < G) p.lse[phys_row(qhead(tid))] = -INFINITY;
    return;
  }

  const int tok_begin = P + split * split_tokens;
  const int tok_end = min(ctx, tok_begin + split_tokens);
  const int n_tiles = (tok_end - tok_begin + kTile - 1) / kTile;

  // kProd: lane 0 of the producer warp copies whole stages (bf16: K dims
  // [0,64), [64,128), V [0,64), [64,128); E4M3: the K and the V box), filling
  // the ring up front and refilling each stage as soon as every consumer warp
  // has released it.  Otherwise the consumer warps copy: bf16: warp w loads
  // the w-th of those four boxes; E4M3: warps 0 and 1 the K and the V box.
  // Each issuing warp fills its part of the ring up front and refills the
  // stage released one tile earlier.  The whole warp runs the issue code and
  // waits; one elected lane issues each copy (issuing from a lane-0 branch
  // spent about 440 cycles per tile there).
  const uint64_t policy = l2_policy_evict_first();
  const int withhold = withheld_tile();   // test hook: tiles from here on are never copied
  auto issue = [&](int it) {
    if (it >= withhold) return;
    const int s = it % kStagesN;
    const int tok = tok_begin + it * kTile;
    const int slot = sblk[tok / kBlockSize - blk_begin] * kBlockSize + tok % kBlockSize;
    // the tile holding the new token is read only once that token is written
    if (store_here && it == n_tiles - 1 && !__all_sync(0xffffffffu, mbar_wait(stored_bar, 0))) {
      if (lane == 0) {
        record_error(p.err, kErrTimeout);
        flags[0] = 1;
      }
      return;
    }
    if constexpr (kProd) {
      const uint32_t dst = smem_addr(smem + s * kStageB);
      mbar_arrive_expect_tx_warp(full_bar(s), kStageB);
      tma_load_3d_hint_warp(dst, &kmap, full_bar(s), 0, kvh0, slot, policy);
      if constexpr (!kFp8)
        tma_load_3d_hint_warp(dst + kHalfBytes, &kmap, full_bar(s), 64, kvh0, slot, policy);
      tma_load_3d_hint_warp(dst + kOpBytes, &vmap, full_bar(s), 0, kvh0, slot, policy);
      if constexpr (!kFp8)
        tma_load_3d_hint_warp(dst + kOpBytes + kHalfBytes, &vmap, full_bar(s), 64, kvh0, slot,
                              policy);
    } else if constexpr (kFp8) {
      // warp 0: the K tile, warp 1: the V tile (one 128-byte-wide box each)
      const uint32_t dst = smem_addr(smem + s * kStageB) + warp * kOpBytes;
      mbar_arrive_expect_tx_warp(full_bar(s), kOpBytes);
      if (warp == 0)
        tma_load_3d_hint_warp(dst, &kmap, full_bar(s), 0, kvh0, slot, policy);
      else
        tma_load_3d_hint_warp(dst, &vmap, full_bar(s), 0, kvh0, slot, policy);
    } else {
      const uint32_t dst = smem_addr(smem + s * kStageB) + warp * kHalfBytes;
      mbar_arrive_expect_tx_warp(full_bar(s), kHalfBytes);
      if (warp < 2)
        tma_load_3d_hint_warp(dst, &kmap, full_bar(s), (warp & 1) * 64, kvh0, slot, policy);
      else
        tma_load_3d_hint_warp(dst, &vmap, full_bar(s), (warp & 1) * 64, kvh0, slot, policy);
    }
    if (lane == 0) atomicMax(const_cast<int*>(flags + 2), it + 1);
  };
  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < kStagesN; ++s) {
        mbar_init(full_bar(s), kProd ? 1 : kIssuers);  // one arrival per issuing warp
        mbar_init(empty_bar(s), kConsumerWarps);
      }
      mbar_init(stored_bar, 1);
      flags[0] = 0;  // abort
      flags[1] = 0;  // last-arrival flag
      flags[2] = 0;  // tiles issued
      fence_barrier_init();
    }
    // Block ids of the range actually used (validated; a bad id is reported
    // and replaced by block 0 so that no out-of-range address is ever formed).
    const int nblk = (tok_end - 1) / kBlockSize - blk_begin + 1;
    if (lane < nblk) {
      if (spec_id < 0 || spec_id >= p.num_blocks) {
        record_error(p.err, kErrIndex);
        spec_id = 0;
      }
      sblk[lane] = spec_id;
    }
  }
  __syncthreads();
  if (store_here && warp == 1) {
    // Warp 1 writes the new token's row of this kv head at its slot (see
    // store_new_row), then tells the issuing lanes, one of which waits for it
    // before copying the tile that holds the row.
    const int sl = __ldg(p.new_slots + b);
    if (sl >= 0) {
      const int pos = ctx - 1;
      store_new_row<kFp8>(p, b, kvh0, sl, sblk[pos / kBlockSize - blk_begin], pos, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(stored_bar);
  }
  const bool prodw = kProd && warp == kCW;  // the producer warp
  if (kProd ? prodw : warp < kIssuers)
    for (int it = 0; it < kStagesN && it < n_tiles; ++it) issue(it);

  {
    // ------------------------------------------------------------ consumers
    // Both contractions run on the warp-level tensor-core MMA (16-bit
    // operands, fp32 accumulation): scores = q K^T with the block's G query
    // heads as MMA rows, output += P V.  Warp w takes tokens [16w, 16w+16) of
    // each 64-token stage.  Lane l = 4 gq + c holds row gq (a query head when
    // gq < G).  A dot product does not depend on which MMA k position carries
    // which dim, so lane (gq, c) reads dims [32c, 32c+32) of token 8n + gq of
    // token group n, and the m-th MMA gets dims 32c+4m+{0,1} at k positions
    // 2c, 2c+1 and 32c+4m+{2,3} at 2c+8, 2c+9, for q and K alike.
    //   bf16 pools: q and K words are the operands as they are.
    //   E4M3 pools: each code pair converts to an f16 operand pair (exact);
    //   q goes to f16 scaled by the power of two that brings its row maximum
    //   into [2^14, 2^15), where every bf16 element down to 2^-32 of that
    //   maximum converts exactly.
    // P V: rows gq carry the weights rounded to 16 bits and rows gq + 8 the
    // rounded remainders, so the weights enter with about 16 (bf16) or 22
    // (f16) significant bits.
    const int gq = lane >> 2;
    const int c = lane & 3;
    // o[jn][0..1]: rows gq, o[jn][2..3]: rows gq + 8 (the weight remainders);
    // summed when the loop ends.  Output column n of n-tile jn is dim
    // vdim(n, jn) below.
    float o[16][4];
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) o[jn][0] = o[jn][1] = o[jn][2] = o[jn][3] = 0.f;
    float m_run = -INFINITY;  // log2-domain running max of row gq
    float l_run = 0.f;        // sum of the weights of this lane's tokens
    if (prodw) {
      for (int it = kStagesN; it < n_tiles; ++it) {
        if (__any_sync(0xffffffffu, flags[0] != 0)) break;
        const int pv = it - kStagesN;
        if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(pv % kStagesN), (pv / kStagesN) & 1))) {
          if (lane == 0) {
            record_error(p.err, kErrTimeout);
            flags[0] = 1;
          }
          break;
        }
        issue(it);
      }
      __syncwarp();
    } else {
    uint32_t qa[8][2];
    float qmul;
    {
      uint32_t qw[16];
      if (gq < G) {
        const uint4* qp = reinterpret_cast<const uint4*>(
            p.q + phys_row(qhead(gq)) * kHeadDim + 32 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 u = __ldg(qp + i);
          qw[4 * i] = u.x;
          qw[4 * i + 1] = u.y;
          qw[4 * i + 2] = u.z;
          qw[4 * i + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) qw[i] = 0u;
      }
      q_fragments<kFp8>(qw, p.scale_log2, p.k_scale, qa, qmul);
    }
    // keys of this split row gq may see (several query positions only)
    const int lim = kMQ ? key_limit(qhead(gq < G ? gq : 0)) - tok_begin : 0;

    // Two groups (kGroups = 2): warps [4 grp, 4 grp + 4) take tiles grp,
    // grp + 2, ...; with an even stage count a stage only ever holds one
    // group's tiles, so a warp that waits for tile it has itself consumed the
    // stage's previous tile, it - kStagesN (the wait is never two phases
    // ahead), and each tile's empty barrier counts that group's four warps.
    const int grp = warp / kConsumerWarps;
    const int wg = warp % kConsumerWarps;   // the warp's 16-token slice of a tile
    for (int it = grp; it < n_tiles; it += kGroups) {
      const int s = it % kStagesN;
      if (flags[0]) break;
      if (!mbar_wait(full_bar(s), (it / kStagesN) & 1)) {
        record_error(p.err, kErrTimeout);
        flags[0] = 1;
        break;
      }
      const int n_valid = min(kTile, tok_end - (tok_begin + it * kTile));
      const uint32_t kb = smem_addr(smem + s * kStageB);
      consume_stage<G, kMQ, kFp8>(kb, kb + kOpBytes, wg, gq, c, qa, qmul, n_valid,
                                  lim - it * kTile, o, m_run, l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      // refill the stage released one tile ago: by now every warp has usually
      // released it too, so the issuing warps seldom wait
      const int pv = it - 1;
      if (!kProd && warp < kIssuers && pv >= 0 && pv + kStagesN < n_tiles &&
          !__any_sync(0xffffffffu, flags[0] != 0)) {
        if (__all_sync(0xffffffffu, mbar_wait(empty_bar(pv % kStagesN), (pv / kStagesN) & 1))) {
          issue(pv + kStagesN);
        } else if (lane == 0) {
          record_error(p.err, kErrTimeout);
          flags[0] = 1;
        }
      }
      __syncwarp();
    }
    }

    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    __syncthreads();  // every warp is done with the stage ring
    // After a timeout, wait (bounded) for copies still in flight before the
    // ring's memory is written or the block's shared memory released.
    if (flags[0] && tid == 0) {
      const int issued = flags[2];
      for (int s = 0; s < kStagesN; ++s) {
        int last = -1;
        for (int it = s; it < issued; it += kStagesN) last = it;
        if (last >= 0) (void)mbar_wait(full_bar(s), (last / kStagesN) & 1);
      }
    }
    __syncthreads();
    if (gq < G && !prodw) {
      // this lane's output columns: n = 2c at dims 32c + jn and n = 2c + 1 at
      // dims 32c + 16 + jn (bf16: 32c + 16 + (jn ^ 8))
      float* dst = merge_o + (warp * G + gq) * kHeadDim + 32 * c;
#pragma unroll
      for (int jn = 0; jn < 16; ++jn) {
        dst[jn] = o[jn][0] + o[jn][2];
        dst[16 + (kFp8 ? jn : (jn ^ 8))] = o[jn][1] + o[jn][3];
      }
      if (c == 0) {
        merge_m[warp * G + gq] = m_run;
        merge_l[warp * G + gq] = l_run;
      }
    }
  }

  __syncthreads();
  // the producer warp and a second consumer group leave: the epilogue (and
  // its named barrier) runs on threads 0..127
  if (tid >= kConsumerWarps * 32) return;

  // ---------------------------------------------------------------- epilogue
  // thread tid (0..127) owns dim d = tid of every head
  const int d = tid;
  const bool single = nsplit == 1 && P == 0;
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, merge_m[w * G + h]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
      const float c = rescale(merge_m[w * G + h], M);
      Ls += merge_l[w * G + h] * c;
      Os += merge_o[(w * G + h) * kHeadDim + d] * c;
    }
    // a split may hold no key a row can see (later query positions only):
    // its partial is then 0 with log2-sum-exp -inf, which the merge ignores
    float on = Ls > 0.f ? Os / Ls : 0.f;
    if constexpr (kFp8) on *= p.v_scale;
    const float lse2 = M + __log2f(Ls);
    const int64_t row = static_cast<int64_t>(b) * p.Hq + qhead(h);
    if (single) {
      const int64_t orow = phys_row(qhead(h));
      p.out[orow * kHeadDim + d] = __float2bfloat16_rn(on);
      if (p.lse && d == 0) p.lse[orow] = lse2 * kLn2;
    } else {
      const int64_t prow = row * p.num_splits + split;
      __stcg(p.ws_o + prow * kHeadDim + d, on);
      if (d == 0) __stcg(p.ws_lse + prow, lse2);
    }
  }
  if (single) return;

  // ---------------------------------------------------------------- split merge
  // All partial stores of the block precede the barrier; one thread then
  // publishes them at device scope and takes the ticket.
  named_barrier(1, kConsumerWarps * 32);
  unsigned* counter = p.ws_count + static_cast<int64_t>(b) * gridDim.y + hg;
  if (tid == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(counter, 1u);
    const bool last = ticket == static_cast<unsigned>(nsplit - 1);
    if (last) __threadfence();
    flags[1] = last ? 1 : 0;
  }
  named_barrier(1, kConsumerWarps * 32);
  if (!flags[1]) return;
  for (int r = warp; r < G; r += kConsumerWarps) {
    const int64_t row = static_cast<int64_t>(b) * p.Hq + qhead(r);
    const int64_t orow = phys_row(qhead(r));
    const int np = P > 0 ? p.prefix_splits : 0;
    merge_row(p.ws_lse + row * p.num_splits, p.ws_o + row * p.num_splits * kHeadDim, nsplit,
              np ? p.prefix_lse + row * np : nullptr,
              np ? p.prefix_o + row * np * kHeadDim : nullptr, np, p.out + orow * kHeadDim,
              p.lse ? p.lse + orow : nullptr, lane);
  }
  if (tid == 0) *counter = 0u;  // ready for the next call
}

template <int G, bool kMQ, bool kFp8, bool kProd, int kGroups = 1>
int launch_g(const DecodeArgs& a, const DecodePlan& plan, const DecodeParams& prm,
             const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t stream) {
  using L = SmemLayout<G, kFp8, kProd, kGroups>;
  static_assert(L::kBytes <= (kGroups == 2 ? 227 : 113) * 1024,
                "two blocks per SM (one with two consumer groups) must fit");
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(paged_decode_kernel<G, kMQ, kFp8, kProd, kGroups>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kBytes) != cudaSuccess)
      return PKV_ERR_LAUNCH;
    attr_set[dev] = true;
  }
  // launched with programmatic stream serialization: it may start while the
  // previous kernel of the stream finishes, and waits (griddepcontrol.wait)
  // before its first global read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.num_splits, a.Hkv * plan.head_groups, a.B);
  cfg.blockDim = dim3(kProd ? kThreads * kGroups + 32 : kThreads);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, paged_decode_kernel<G, kMQ, kFp8, kProd, kGroups>, km, vm, prm) !=
      cudaSuccess)
    return PKV_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

int set_wait_hook_decode(unsigned long long limit_ns, int withhold_plus1) {
  const WaitHook h{limit_ns, withhold_plus1, 0};
  return cudaMemcpyToSymbol(g_wait_hook, &h, sizeof h) == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int plan_decode(int B, int Hq, int Hkv, int max_blocks_per_seq, int num_splits,
                int sm_count, int prefix_blocks, DecodePlan* plan) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || prefix_blocks < 0 ||
      prefix_blocks > max_blocks_per_seq)
    return PKV_ERR_ARG;
  if (Hq % Hkv) return PKV_ERR_SHAPE;
  const int g = Hq / Hkv;
  const int G = (g % 8 == 0) ? 8 : (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
  plan->heads_per_cta = G;
  plan->head_groups = g / G;
  plan->consumer_groups = 1;
  // One kv head per block.  (Reading two kv heads per block as 512-byte
  // chunks per token measured 2% slower on GB300 on the batch-64 decode and
  // slower on short contexts.)
  const int kv_groups = Hkv;
  const int rest = max_blocks_per_seq - prefix_blocks;
  const int maxblk = rest > 0 ? rest : 1;
  const int sms = sm_count > 0 ? sm_count : 148;
  const int64_t seq_units = static_cast<int64_t>(B) * kv_groups * plan->head_groups;
  int split_blocks;
  bool small = false;
  if (num_splits > 0) {
    split_blocks = (maxblk + num_splits - 1) / num_splits;
  } else {
    // Enough (sequence, head group, split) units for about eight waves of two
    // blocks per SM if every context were full length; whole blocks per split.
    const int64_t units = seq_units * maxblk;
    const int64_t target = static_cast<int64_t>(sms) * 2 * 8;
    split_blocks = static_cast<int>((units + target - 1) / target);
    // A batch whose one-block splits would not even fill one wave of one
    // block per SM splits into 64-token tiles instead (a launch-latency
    // bound step: more blocks, each with a shorter chain of copies).
    small = units < sms;
    if (split_blocks < 2) split_blocks = maxblk < 2 ? maxblk : 2;
  }
  if (split_blocks < 1) split_blocks = 1;
  if (split_blocks > kMaxSplitBlocks) split_blocks = kMaxSplitBlocks;
  int S = (maxblk + split_blocks - 1) / split_blocks;
  if (S > kMaxSplits) return PKV_ERR_SHAPE;
  // re-balance so that the splits are as even as possible
  split_blocks = (maxblk + S - 1) / S;
  plan->split_tokens = split_blocks * kBlockSize;
  if (small && maxblk <= 3) {
    // Contexts of at most three blocks: one split per sequence, no merge.  The
    // merge of split partials (store, ticket, reads) costs about as much as
    // eight or nine 64-token tiles of one block's chain (measured: 4 sequences
    // of up to 513 tokens, 6.74 us per call under graph replay against 7.34
    // us with 64-token splits; 13.3 against 14.3 us per call).
    S = 1;
    plan->split_tokens = maxblk * kBlockSize;
    // The grid (one block per sequence and kv head group) is under one wave,
    // so each block may take a whole SM: two groups of consumer warps take
    // alternate tiles, which halves the chain of tiles of the longest context.
    plan->consumer_groups = 2;
  } else if (small) {
    constexpr int kTilesPerBlock = kBlockSize / kTile;
    const int64_t tiles = static_cast<int64_t>(maxblk) * kTilesPerBlock;
    const int64_t want = static_cast<int64_t>(sms) * 4;   // about one tile per block
    int split_tiles = static_cast<int>((seq_units * tiles + want - 1) / want);
    if (split_tiles < 1) split_tiles = 1;
    if (split_tiles < kTilesPerBlock) {
      S = static_cast<int>((tiles + split_tiles - 1) / split_tiles);
      plan->split_tokens = split_tiles * kTile;
    }
  }
  plan->num_splits = S;
  plan->prefix_offset = 0;
  plan->prefix_splits = 0;
  plan->prefix_kt_per = 0;
  if (prefix_blocks > 0) {
    // Key ranges of the shared-prefix pass: enough blocks for about one wave.
    const int kt = prefix_blocks * (kBlockSize / 128);
    const int rpt = prefix_rows_per_tile(g);
    if (rpt == 0) return PKV_ERR_SHAPE;
    const int base = (B * g + rpt - 1) / rpt * Hkv;   // query tiles of the pass
    const int sms = sm_count > 0 ? sm_count : 148;
    int ps = base >= sms ? 1 : sms / base;
    if (ps > kt) ps = kt;
    if (ps < 1) ps = 1;
    plan->prefix_kt_per = (kt + ps - 1) / ps;
    plan->prefix_splits = (kt + plan->prefix_kt_per - 1) / plan->prefix_kt_per;
  }
  if (S == 1 && prefix_blocks == 0) {
    plan->workspace_bytes = 0;
  } else {
    if (static_cast<int64_t>(B) * kv_groups * plan->head_groups > kMaxCounters)
      return PKV_ERR_SHAPE;
    const size_t rows = static_cast<size_t>(B) * Hq * S;
    size_t bytes = kCounterRegion;
    bytes += align_up(rows * kHeadDim * sizeof(float), 256);
    bytes += align_up(rows * sizeof(float), 256);
    if (prefix_blocks > 0) {
      plan->prefix_offset = bytes;
      const size_t prow = static_cast<size_t>(B) * Hq * plan->prefix_splits;
      bytes += align_up(prow * kHeadDim * sizeof(float), 256);
      bytes += align_up(prow * sizeof(float), 256);
    }
    plan->workspace_bytes = bytes;
  }
  return PKV_OK;
}

int launch_decode(const DecodeArgs& a, const DecodePlan& plan, unsigned* err,
                  cudaStream_t stream) {
  if (a.B == 0) return PKV_OK;
  CUtensorMap km, vm;
  const int64_t slots = a.num_blocks * kBlockSize;
  if (a.fp8) {
    if (!encode_pool_map_u8(&km, a.k_cache, slots, a.Hkv, kTile) ||
        !encode_pool_map_u8(&vm, a.v_cache, slots, a.Hkv, kTile))
      return PKV_ERR_ARG;
  } else if (!encode_pool_map(&km, a.k_cache, slots, a.Hkv, kTile) ||
             !encode_pool_map(&vm, a.v_cache, slots, a.Hkv, kTile)) {
    return PKV_ERR_ARG;
  }
  DecodeParams prm;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.lse = a.lse;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.err = err;
  prm.B = a.B;
  prm.Hq = a.Hq * a.q_len;   // virtual heads (see DecodeParams)
  prm.Hq_phys = a.Hq;
  prm.q_len = a.q_len;
  prm.k_scale = a.k_scale;
  prm.v_scale = a.v_scale;
  prm.Hkv = a.Hkv;
  prm.maxblk = a.max_blocks_per_seq;
  prm.num_splits = plan.num_splits;
  prm.split_tokens = plan.split_tokens;
  prm.head_groups = plan.head_groups;
  prm.num_blocks = a.num_blocks;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.prefix_tokens = a.prefix_tokens;
  prm.metadata_ready = a.metadata_ready;
  prm.prefix_splits = plan.prefix_splits;
  prm.new_slots = a.new_slots;
  prm.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  prm.k_new_stride = a.k_new_stride;
  prm.v_new_stride = a.v_new_stride;
  prm.k_pool = static_cast<uint4*>(const_cast<void*>(a.k_cache));
  prm.v_pool = static_cast<uint4*>(const_cast<void*>(a.v_cache));
  // the store's quantizer multiplies by the binary32 reciprocal of each scale
  prm.k_inv = 1.0f / a.k_scale;
  prm.v_inv = 1.0f / a.v_scale;
  prm.prefix_o = nullptr;
  prm.prefix_lse = nullptr;
  if (a.prefix_tokens > 0) {
    const uint8_t* base = static_cast<const uint8_t*>(a.workspace) + plan.prefix_offset;
    prm.prefix_o = reinterpret_cast<const float*>(base);
    prm.prefix_lse = reinterpret_cast<const float*>(
        base + align_up(static_cast<size_t>(a.B) * a.Hq * plan.prefix_splits * kHeadDim *
                            sizeof(float), 256));
  }
  if (plan.workspace_bytes > 0) {
    const size_t rows = static_cast<size_t>(a.B) * a.Hq * a.q_len * plan.num_splits;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    prm.ws_count = reinterpret_cast<unsigned*>(ws);
    ws += kCounterRegion;
    prm.ws_o = reinterpret_cast<float*>(ws);
    ws += align_up(rows * kHeadDim * sizeof(float), 256);
    prm.ws_lse = reinterpret_cast<float*>(ws);
  } else {
    prm.ws_o = nullptr;
    prm.ws_lse = nullptr;
    prm.ws_count = nullptr;
  }
  // bf16 pools: the producer-warp form (two blocks per SM either way).  E4M3
  // pools: three blocks per SM of the consumer-issued form, or two of the
  // producer-warp form with a deeper ring; the latter wins once a split is
  // long enough (measured on GB300: 8-block splits of the 32K-128K-token
  // contexts 6% faster, 4-block splits of 512-4096-token contexts 1.5% slower).
  if (a.fp8) {
    const bool prod = plan.split_tokens >= 8 * kBlockSize;
    switch (plan.heads_per_cta) {
      case 8:
        return prod ? launch_g<8, false, true, true>(a, plan, prm, km, vm, stream)
                    : launch_g<8, false, true, false>(a, plan, prm, km, vm, stream);
      case 4:
        return prod ? launch_g<4, false, true, true>(a, plan, prm, km, vm, stream)
                    : launch_g<4, false, true, false>(a, plan, prm, km, vm, stream);
      case 2:
        return prod ? launch_g<2, false, true, true>(a, plan, prm, km, vm, stream)
                    : launch_g<2, false, true, false>(a, plan, prm, km, vm, stream);
      default:
        return prod ? launch_g<1, false, true, true>(a, plan, prm, km, vm, stream)
                    : launch_g<1, false, true, false>(a, plan, prm, km, vm, stream);
    }
  }
  // bf16 single-token batches of one split per sequence under one wave: the
  // producer-warp form with two consumer groups (one block per SM)
  if (plan.consumer_groups == 2 && a.q_len == 1) {
    switch (plan.heads_per_cta) {
      case 8: return launch_g<8, false, false, true, 2>(a, plan, prm, km, vm, stream);
      case 4: return launch_g<4, false, false, true, 2>(a, plan, prm, km, vm, stream);
      case 2: return launch_g<2, false, false, true, 2>(a, plan, prm, km, vm, stream);
      default: return launch_g<1, false, false, true, 2>(a, plan, prm, km, vm, stream);
    }
  }
  // bf16 batches split into 64-token tiles: the 2-stage consumer-issued form
  // (three blocks per SM)
  if (plan.split_tokens < kBlockSize) {
    switch (plan.heads_per_cta) {
      case 8:
        return a.q_len > 1 ? launch_g<8, true, false, false>(a, plan, prm, km, vm, stream)
                           : launch_g<8, false, false, false>(a, plan, prm, km, vm, stream);
      case 4:
        return a.q_len > 1 ? launch_g<4, true, false, false>(a, plan, prm, km, vm, stream)
                           : launch_g<4, false, false, false>(a, plan, prm, km, vm, stream);
      case 2:
        return a.q_len > 1 ? launch_g<2, true, false, false>(a, plan, prm, km, vm, stream)
                           : launch_g<2, false, false, false>(a, plan, prm, km, vm, stream);
      default:
        return a.q_len > 1 ? launch_g<1, true, false, false>(a, plan, prm, km, vm, stream)
                           : launch_g<1, false, false, false>(a, plan, prm, km, vm, stream);
    }
  }
  switch (plan.heads_per_cta) {
    case 8:
      return a.q_len > 1 ? launch_g<8, true, false, true>(a, plan, prm, km, vm, stream)
                         : launch_g<8, false, false, true>(a, plan, prm, km, vm, stream);
    case 4:
      return a.q_len > 1 ? launch_g<4, true, false, true>(a, plan, prm, km, vm, stream)
                         : launch_g<4, false, false, true>(a, plan, prm, km, vm, stream);
    case 2:
      return a.q_len > 1 ? launch_g<2, true, false, true>(a, plan, prm, km, vm, stream)
                         : launch_g<2, false, false, true>(a, plan, prm, km, vm, stream);
    default:
      return a.q_len > 1 ? launch_g<1, true, false, true>(a, plan, prm, km, vm, stream)
                         : launch_g<1, false, false, true>(a, plan, prm, km, vm, stream);
  }
}

}  // namespace pkv
