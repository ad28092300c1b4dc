// store.cu — kv_cache_store, kv_cache_store_fp8 and kv_cache_copy_blocks for
// sm_103a.
//
// Operation: new K/V rows are written into the paged cache through slot_mapping
// ("Nano-vLLM System Architecture Analysis", §2 Core Components, "Attention with
// Paged Cache"; 256-token blocks per "Paged KV Cache").  A slot addresses one
// contiguous [Hkv, D] row of the pool, so a token's K (and V) row is a single
// contiguous 2*Hkv*D-byte copy.
//
// Design: a plain bandwidth kernel.  Consecutive threads move consecutive
// 16-byte pieces of the same row (coalesced reads and writes); the grid is a
// multiple of the SM count and strides over (token, K|V, piece).  Padding slots
// (< 0) are skipped; out-of-range slots are skipped and reported.  The E4M3
// variant converts each 16-element piece to one-byte codes on the way (the
// quantized KV cache that "Why Understand Inference Engine Architecture?",
// Tensor Parallelism Optimization, names); the block copy serves
// copy-on-write ("Paged KV Cache", reference counting).

#include <cuda_bf16.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kStoreThreads = 256;

// VEC: 16-byte pieces (8 bf16); otherwise single elements.
template <bool VEC>
__global__ void __launch_bounds__(kStoreThreads)
kv_store_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                int64_t k_stride, int64_t v_stride, uint16_t* __restrict__ k_cache,
                uint16_t* __restrict__ v_cache, const int32_t* __restrict__ slots, int64_t T,
                int row_elems, int64_t num_slots, unsigned* err) {
  constexpr int kPer = VEC ? 8 : 1;
  const int pieces = row_elems / kPer;
  const int64_t per_token = 2 * static_cast<int64_t>(pieces);
  const int64_t total = T * per_token;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / per_token;
    const int rem = static_cast<int>(i - t * per_token);
    const int which = rem >= pieces;  // 0 = K, 1 = V
    const int piece = rem - which * pieces;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (piece == 0 && which == 0) record_error(err, kErrIndex);
      continue;
    }
    const uint16_t* src = (which ? v + t * v_stride : k + t * k_stride) + piece * kPer;
    uint16_t* dst = (which ? v_cache : k_cache) + s * row_elems + piece * kPer;
    if constexpr (VEC) {
      *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
    } else {
      *dst = __ldg(src);
    }
  }
}

// Whole-block copies for copy-on-write: block dst[i] of both pools becomes a
// bit copy of block src[i].  Consecutive threads move consecutive 16-byte pieces.
__global__ void __launch_bounds__(kStoreThreads)
kv_copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                      const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                      int n_pairs, int64_t block_vecs, int64_t num_blocks, unsigned* err) {
  const int64_t per_pair = 2 * block_vecs;
  const int64_t total = static_cast<int64_t>(n_pairs) * per_pair;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t pair = i / per_pair;
    const int64_t rem = i - pair * per_pair;
    const int which = rem >= block_vecs;
    const int64_t off = rem - which * block_vecs;
    const int64_t s = __ldg(src + pair), d = __ldg(dst + pair);
    if (s < 0 || d < 0 || s >= num_blocks || d >= num_blocks) {
      if (off == 0 && which == 0) record_error(err, kErrIndex);
      continue;
    }
    uint4* cache = which ? v_cache : k_cache;
    cache[d * block_vecs + off] = cache[s * block_vecs + off];
  }
}

// FP8 store: every bf16 element x of a token row becomes the E4M3 code of
// x * inv_scale (inv_scale = 1/scale rounded to fp32 by the host; the product
// rounded to fp32, then to the nearest code, ties to even, saturating at 448).
// VEC: 16 elements per thread (two 16-byte loads, one 16-byte store).
template <bool VEC>
__global__ void __launch_bounds__(kStoreThreads)
kv_store_fp8_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                    int64_t k_stride, int64_t v_stride, uint8_t* __restrict__ k_cache,
                    uint8_t* __restrict__ v_cache, const int32_t* __restrict__ slots, int64_t T,
                    int row_elems, int64_t num_slots, float k_inv, float v_inv, unsigned* err) {
  constexpr int kPer = VEC ? 16 : 1;
  const int pieces = row_elems / kPer;
  const int64_t per_token = 2 * static_cast<int64_t>(pieces);
  const int64_t total = T * per_token;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / per_token;
    const int rem = static_cast<int>(i - t * per_token);
    const int which = rem >= pieces;  // 0 = K, 1 = V
    const int piece = rem - which * pieces;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (piece == 0 && which == 0) record_error(err, kErrIndex);
      continue;
    }
    const uint16_t* src = (which ? v + t * v_stride : k + t * k_stride) + piece * kPer;
    uint8_t* dst = (which ? v_cache : k_cache) + s * row_elems + piece * kPer;
    const float inv = which ? v_inv : k_inv;
    if constexpr (VEC) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c0 = e4m3x2_from_f32(bf16lo(w[2 * j]) * inv, bf16hi(w[2 * j]) * inv);
        const uint32_t c1 =
            e4m3x2_from_f32(bf16lo(w[2 * j + 1]) * inv, bf16hi(w[2 * j + 1]) * inv);
        o[j] = c0 | (c1 << 16);
      }
      *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      const float x = __uint_as_float(static_cast<uint32_t>(__ldg(src)) << 16);
      *dst = static_cast<uint8_t>(e4m3x2_from_f32(x * inv, 0.f) & 0xFFu);
    }
  }
}

}  // namespace

int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                       int n_pairs, int64_t block_bytes, int64_t num_blocks, unsigned* err,
                       cudaStream_t stream) {
  if (n_pairs == 0) return PKV_OK;
  const int64_t vecs = block_bytes / 16;
  const int64_t total = static_cast<int64_t>(n_pairs) * 2 * vecs;
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  int64_t blocks = (total + kStoreThreads - 1) / kStoreThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  kv_copy_blocks_kernel<<<static_cast<unsigned>(blocks), kStoreThreads, 0, stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src, dst, n_pairs, vecs,
      num_blocks, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int launch_store(const StoreArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.T == 0) return PKV_OK;
  const bool vec = (reinterpret_cast<uintptr_t>(a.k) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.v) % 16 == 0) &&
                   ((a.k_tok_stride * 2) % 16 == 0) && ((a.v_tok_stride * 2) % 16 == 0) &&
                   (a.row_elems % 8 == 0);
  const int pieces = vec ? a.row_elems / 8 : a.row_elems;
  const int64_t total = a.T * 2 * static_cast<int64_t>(pieces);
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  int64_t blocks = (total + kStoreThreads - 1) / kStoreThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  const auto* k = static_cast<const uint16_t*>(a.k);
  const auto* v = static_cast<const uint16_t*>(a.v);
  auto* kc = static_cast<uint16_t*>(a.k_cache);
  auto* vc = static_cast<uint16_t*>(a.v_cache);
  if (vec)
    kv_store_kernel<true><<<static_cast<unsigned>(blocks), kStoreThreads, 0, stream>>>(
        k, v, a.k_tok_stride, a.v_tok_stride, kc, vc, a.slot_mapping, a.T, a.row_elems,
        a.num_slots, err);
  else
    kv_store_kernel<false><<<static_cast<unsigned>(blocks), kStoreThreads, 0, stream>>>(
        k, v, a.k_tok_stride, a.v_tok_stride, kc, vc, a.slot_mapping, a.T, a.row_elems,
        a.num_slots, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

int launch_store_fp8(const StoreArgs& a, float k_inv, float v_inv, unsigned* err,
                     cudaStream_t stream) {
  if (a.T == 0) return PKV_OK;
  const bool vec = (reinterpret_cast<uintptr_t>(a.k) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.v) % 16 == 0) &&
                   ((a.k_tok_stride * 2) % 16 == 0) && ((a.v_tok_stride * 2) % 16 == 0) &&
                   (a.row_elems % 16 == 0);
  const int pieces = vec ? a.row_elems / 16 : a.row_elems;
  const int64_t total = a.T * 2 * static_cast<int64_t>(pieces);
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  int64_t blocks = (total + kStoreThreads - 1) / kStoreThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  const auto* k = static_cast<const uint16_t*>(a.k);
  const auto* v = static_cast<const uint16_t*>(a.v);
  auto* kc = static_cast<uint8_t*>(a.k_cache);
  auto* vc = static_cast<uint8_t*>(a.v_cache);
  if (vec)
    kv_store_fp8_kernel<true><<<static_cast<unsigned>(blocks), kStoreThreads, 0, stream>>>(
        k, v, a.k_tok_stride, a.v_tok_stride, kc, vc, a.slot_mapping, a.T, a.row_elems,
        a.num_slots, k_inv, v_inv, err);
  else
    kv_store_fp8_kernel<false><<<static_cast<unsigned>(blocks), kStoreThreads, 0, stream>>>(
        k, v, a.k_tok_stride, a.v_tok_stride, kc, vc, a.slot_mapping, a.T, a.row_elems,
        a.num_slots, k_inv, v_inv, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv
