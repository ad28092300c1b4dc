// pkv_oracle.cpp — CPU oracle for paged KV-cache attention (fp64).
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
// definition that the GPU library is checked against.  Only the test-suite, the
// smoke check and the CPU-baseline leg of the benchmark load it.  It shares no
// code, header, table or helper with the CUDA library, and the CUDA library never
// calls it.
//
// What it computes, and where each step comes from:
//   * "Nano-vLLM System Architecture Analysis", §2 Core Components,
//     "Paged KV Cache": the cache is split into fixed-size blocks of 256 tokens.
//   * same page, §2, "Attention with Paged Cache": new K/V entries are written
//     into the paged cache through slot_mapping; prefill with a prefix cache
//     gathers the cached K/V and concatenates the new ones; decode gathers all of
//     a sequence's cached K/V from its blocks and then runs scaled dot-product
//     attention.
//   * "Why Understand Inference Engine Architecture?", TorchScript Optimization:
//     attention is softmax(q k^T) v.  The 1/sqrt(head_dim) scale is passed in.
//   * "Nano-vLLM System Architecture Analysis", §6 Architecture Support: GQA.
//     Query head h reads kv head h / (Hq / Hkv) (contiguous groups).
//   * same page, §2 "Scheduler" and "Differences", §3: chunked prefill.  New
//     query rows follow the cached prefix, so query row r of a chunk with Lq new
//     tokens over Lk keys may see keys j <= Lk - Lq + r (bottom-right causal).
//
// Readings where the pages are silent (each one is listed in the design notes):
//   * pool layout [num_blocks, block_size, Hkv, D]; a slot = block*block_size +
//     offset indexes one [Hkv, D] row;
//   * a negative slot means "padding, skip"; a slot >= num_blocks*block_size or a
//     repeated slot is an error;
//   * an empty context (L = 0) gives out = 0 and lse = -inf;
//   * lse is the natural log of the sum of exp(scaled scores).
//   * FP8 KV cache: the pages name quantized KV only as "compressed transfers"
//     ("Why Understand Inference Engine Architecture?", Tensor Parallelism
//     Optimization) and give no format.  The reading used here: the
//     OCP FP8 E4M3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa
//     bits, subnormals, no infinity, 0x7F / 0xFF = NaN, largest finite 448) with
//     one scale per tensor; a value x is stored as the code nearest to
//     x * (1 / scale), both factors rounded to binary32 first and the product
//     rounded to binary32, ties to the even code, magnitudes past 448 saturated
//     to 448, and read back as code value * scale.
//
// Arithmetic: every bf16 input is widened exactly to double; scores, softmax and
// the weighted sum of V are in double, summed in ascending index order, so the
// result does not depend on how blocks are placed in the pool.
//
// Parallelism: std::thread over independent (sequence, kv head[, row range])
// items.  The per-item arithmetic is identical whatever the thread count.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// bf16 is the top half of an IEEE binary32; widening is exact.
double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  unsigned hc = std::thread::hardware_concurrency();
  return hc ? static_cast<int>(hc) : 1;
}

// Run fn(item) for item in [0, n_items) on nthreads threads (static striping).
template <class F>
void parallel_for(int64_t n_items, int nthreads, F fn) {
  nthreads = resolve_threads(nthreads);
  if (nthreads > n_items) nthreads = static_cast<int>(n_items > 0 ? n_items : 1);
  if (nthreads <= 1) {
    for (int64_t i = 0; i < n_items; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(nthreads);
  for (int t = 0; t < nthreads; ++t) {
    pool.emplace_back([=]() {
      for (int64_t i = t; i < n_items; i += nthreads) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

// Gather (the pages' "gathers cached K/V from paged blocks"): rebuild the
// contiguous [L, D] key and value rows of one kv head of one sequence from the
// block pool (elements T: bf16 bit patterns, or FP8 codes).  Returns false if a
// block id read for a logical position is out of range.
template <class T>
bool gather_head(const T* k_cache, const T* v_cache,
                 const int32_t* table_row, int64_t L, int Hkv, int D,
                 int block_size, int64_t num_blocks, int kv_head,
                 std::vector<T>& K, std::vector<T>& V) {
  K.resize(static_cast<size_t>(L) * D);
  V.resize(static_cast<size_t>(L) * D);
  for (int64_t j = 0; j < L; ++j) {
    const int32_t blk = table_row[j / block_size];
    if (blk < 0 || blk >= num_blocks) return false;
    const int64_t slot = static_cast<int64_t>(blk) * block_size + j % block_size;
    const int64_t src = (slot * Hkv + kv_head) * D;
    std::memcpy(&K[static_cast<size_t>(j) * D], k_cache + src, sizeof(T) * D);
    std::memcpy(&V[static_cast<size_t>(j) * D], v_cache + src, sizeof(T) * D);
  }
  return true;
}

// Slot rules of a store: negative = padding; a slot past the pool (-2) or a
// slot given twice (-3) is an error.
int check_slots(const int32_t* slot_mapping, int64_t T, int64_t n_slots) {
  std::vector<char> seen(static_cast<size_t>(n_slots), 0);
  for (int64_t t = 0; t < T; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= n_slots) return -2;
    if (seen[s]) return -3;
    seen[s] = 1;
  }
  return 0;
}

// bf16 rows widened exactly to double.
std::vector<double> widen(const std::vector<uint16_t>& x) {
  std::vector<double> y(x.size());
  for (size_t i = 0; i < x.size(); ++i) y[i] = bf16_to_double(x[i]);
  return y;
}

// ---------------------------------------------------------------- FP8 E4M3

// Value of an E4M3 code, from the format's definition.
double e4m3_value(uint8_t code) {
  const int sign = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  double mag;
  if (e == 0)
    mag = std::ldexp(static_cast<double>(m), -9);          // subnormal: m/8 * 2^-6
  else
    mag = std::ldexp(1.0 + m / 8.0, e - 7);                // normal: (1 + m/8) * 2^(e-7)
  return sign ? -mag : mag;
}

// Nearest E4M3 code to v (ties to even), magnitudes beyond 448 (infinity
// included) saturated to 448, NaN to 0x7F.  All arithmetic below is exact in
// double.
uint8_t e4m3_encode(float v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(v));
  if (a == 0.0) return sign;
  if (std::isinf(a)) return sign | 0x7E;
  int e;       // a = f * 2^(e+1), f in [0.5, 1): the binade of a is 2^e
  std::frexp(a, &e);
  e -= 1;
  if (e < -6) e = -6;                           // subnormal range shares 2^-6's spacing
  const double quantum = std::ldexp(1.0, e - 3);  // 3 mantissa bits
  double m = std::nearbyint(a / quantum);       // round half to even
  if (m == 16.0) {                              // rounded up into the next binade
    m = 8.0;
    e += 1;
  }
  // largest finite: e = 8, m = 14 (1.75 * 2^8 = 448); beyond it, saturate
  if (e > 8 || (e == 8 && m > 14.0)) return sign | 0x7E;
  if (m < 8.0) return sign | static_cast<uint8_t>(m);   // subnormal (e == -6)
  return sign | static_cast<uint8_t>(((e + 7) << 3) | (static_cast<int>(m) - 8));
}

// The stored code of a bf16 value x under a tensor scale whose reciprocal is
// inv_scale (already rounded to binary32): the product is rounded to binary32.
uint8_t quantize(uint16_t x_bits, float inv_scale) {
  uint32_t u = static_cast<uint32_t>(x_bits) << 16;
  float x;
  std::memcpy(&x, &u, sizeof x);
  const float v = x * inv_scale;
  return e4m3_encode(v);
}

// Softmax attention of one query row over the first n_keys key / value rows
// (already widened to double).  Writes D outputs and the natural-log LSE.
void attend_row_values(const uint16_t* q_row, const std::vector<double>& K,
                       const std::vector<double>& V, int64_t n_keys, int D, double scale,
                       std::vector<double>& s, double* out, double* lse) {
  if (n_keys <= 0) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    *lse = -std::numeric_limits<double>::infinity();
    return;
  }
  s.resize(static_cast<size_t>(n_keys));
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j < n_keys; ++j) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += bf16_to_double(q_row[d]) * K[static_cast<size_t>(j) * D + d];
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < n_keys; ++j) {
    s[j] = std::exp(s[j] - m);
    l += s[j];
  }
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int64_t j = 0; j < n_keys; ++j)
    for (int d = 0; d < D; ++d) out[d] += s[j] * V[static_cast<size_t>(j) * D + d];
  for (int d = 0; d < D; ++d) out[d] /= l;
  *lse = m + std::log(l);
}

}  // namespace

extern "C" {

// Value of every E4M3 code (256 entries; NaN for 0x7F and 0xFF).
int oracle_e4m3_table(double* out256) {
  for (int c = 0; c < 256; ++c) out256[c] = e4m3_value(static_cast<uint8_t>(c));
  return 0;
}

// E4M3 codes of n bf16 values under reciprocal scale inv_scale (binary32).
int oracle_quantize_e4m3(const uint16_t* x, int64_t n, float inv_scale, uint8_t* codes) {
  if (n < 0) return -1;
  for (int64_t i = 0; i < n; ++i) codes[i] = quantize(x[i], inv_scale);
  return 0;
}

// oracle_store into an FP8 pool: the [Hkv, D] rows of token t are quantized
// (k with k_inv_scale, v with v_inv_scale) and written at slot_mapping[t].
// Same slot rules and status codes as oracle_store.
int oracle_store_fp8(const uint16_t* k, const uint16_t* v, int64_t k_tok_stride,
                     int64_t v_tok_stride, uint8_t* k_cache, uint8_t* v_cache,
                     const int32_t* slot_mapping, int64_t T, int Hkv, int D, int block_size,
                     int64_t num_blocks, float k_inv_scale, float v_inv_scale) {
  if (T < 0 || Hkv <= 0 || D <= 0 || block_size <= 0 || num_blocks < 0) return -1;
  const int st = check_slots(slot_mapping, T, num_blocks * block_size);
  if (st) return st;
  const int64_t row = static_cast<int64_t>(Hkv) * D;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    for (int64_t i = 0; i < row; ++i) {
      k_cache[s * row + i] = quantize(k[t * k_tok_stride + i], k_inv_scale);
      v_cache[s * row + i] = quantize(v[t * v_tok_stride + i], v_inv_scale);
    }
  }
  return 0;
}

// oracle_decode over an FP8 pool: key j of a sequence is value(code) * k_scale
// and value j is value(code) * v_scale (in double); the rest as oracle_decode.
int oracle_decode_fp8(double* out, double* lse, const uint16_t* q, const uint8_t* k_cache,
                      const uint8_t* v_cache, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, int B, int Hq,
                      int Hkv, int D, int block_size, int64_t num_blocks, double scale,
                      double k_scale, double v_scale, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || block_size <= 0)
    return -1;
  for (int b = 0; b < B; ++b) {
    if (context_lens[b] < 0) return -1;
    if (static_cast<int64_t>(context_lens[b]) >
        static_cast<int64_t>(max_blocks_per_seq) * block_size)
      return -6;
  }
  const int g = Hq / Hkv;
  std::vector<int> status(static_cast<size_t>(B) * Hkv, 0);
  parallel_for(static_cast<int64_t>(B) * Hkv, nthreads, [&](int64_t item) {
    const int b = static_cast<int>(item / Hkv);
    const int kvh = static_cast<int>(item % Hkv);
    const int64_t L = context_lens[b];
    std::vector<uint8_t> Kc, Vc;
    if (!gather_head(k_cache, v_cache,
                     block_tables + static_cast<int64_t>(b) * max_blocks_per_seq, L,
                     Hkv, D, block_size, num_blocks, kvh, Kc, Vc)) {
      status[item] = -4;
      return;
    }
    // dequantize: code value * tensor scale, in double
    std::vector<double> K(Kc.size()), V(Vc.size()), s;
    for (size_t i = 0; i < Kc.size(); ++i) {
      K[i] = e4m3_value(Kc[i]) * k_scale;
      V[i] = e4m3_value(Vc[i]) * v_scale;
    }
    for (int hh = 0; hh < g; ++hh) {
      const int64_t r = static_cast<int64_t>(b) * Hq + kvh * g + hh;
      attend_row_values(q + r * D, K, V, L, D, scale, s, out + r * D, lse + r);
    }
  });
  for (int st : status)
    if (st) return st;
  return 0;
}


// Status codes of the oracle (its own; not the library's).
//   0 ok, -1 bad argument, -2 slot out of range, -3 duplicate slot,
//   -4 block id out of range, -5 Lk < Lq, -6 context longer than the table.

// Store: for each token t with slot s = slot_mapping[t] >= 0, copy the [Hkv, D]
// rows of k and v (token stride k_tok_stride / v_tok_stride elements) to slot s
// of k_cache / v_cache ([num_blocks*block_size, Hkv, D]).  Bit copy.
int oracle_store(const uint16_t* k, const uint16_t* v, int64_t k_tok_stride,
                 int64_t v_tok_stride, uint16_t* k_cache, uint16_t* v_cache,
                 const int32_t* slot_mapping, int64_t T, int Hkv, int D,
                 int block_size, int64_t num_blocks) {
  if (T < 0 || Hkv <= 0 || D <= 0 || block_size <= 0 || num_blocks < 0) return -1;
  // Validate first so that an error leaves the caches untouched.
  const int st = check_slots(slot_mapping, T, num_blocks * block_size);
  if (st) return st;
  const int64_t row = static_cast<int64_t>(Hkv) * D;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    const int64_t blk = s / block_size;
    const int64_t off = s % block_size;
    const int64_t dst = (blk * block_size + off) * row;
    std::memcpy(k_cache + dst, k + t * k_tok_stride, sizeof(uint16_t) * row);
    std::memcpy(v_cache + dst, v + t * v_tok_stride, sizeof(uint16_t) * row);
  }
  return 0;
}

// Copy-on-write block copies ("Reference counting for block sharing
// (copy-on-write semantics)", same page, §2 "Paged KV Cache"): for each pair,
// block dst[i] of both caches becomes a copy of block src[i].  Bit copy.
int oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int32_t* src,
                       const int32_t* dst, int64_t n_pairs, int Hkv, int D,
                       int block_size, int64_t num_blocks) {
  if (n_pairs < 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return -1;
  for (int64_t i = 0; i < n_pairs; ++i)
    if (src[i] < 0 || dst[i] < 0 || src[i] >= num_blocks || dst[i] >= num_blocks) return -4;
  const int64_t block_elems = static_cast<int64_t>(block_size) * Hkv * D;
  for (int64_t i = 0; i < n_pairs; ++i) {
    std::memcpy(k_cache + dst[i] * block_elems, k_cache + src[i] * block_elems,
                sizeof(uint16_t) * block_elems);
    std::memcpy(v_cache + dst[i] * block_elems, v_cache + src[i] * block_elems,
                sizeof(uint16_t) * block_elems);
  }
  return 0;
}

// Gather of one sequence into contiguous [L, Hkv, D] K and V (bf16 bits).
// Exposed for the round-trip tests of the addressing.
int oracle_gather(const uint16_t* k_cache, const uint16_t* v_cache,
                  const int32_t* table_row, int64_t L, int Hkv, int D,
                  int block_size, int64_t num_blocks, uint16_t* K_out,
                  uint16_t* V_out) {
  if (L < 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return -1;
  std::vector<uint16_t> K, V;
  for (int h = 0; h < Hkv; ++h) {
    if (!gather_head(k_cache, v_cache, table_row, L, Hkv, D, block_size,
                     num_blocks, h, K, V))
      return -4;
    for (int64_t j = 0; j < L; ++j) {
      std::memcpy(K_out + (j * Hkv + h) * D, &K[static_cast<size_t>(j) * D], sizeof(uint16_t) * D);
      std::memcpy(V_out + (j * Hkv + h) * D, &V[static_cast<size_t>(j) * D], sizeof(uint16_t) * D);
    }
  }
  return 0;
}

// Decode: one query row per (sequence b, query head h); the context is the first
// context_lens[b] logical tokens of sequence b (the token stored this step
// included), read through block_tables[b, :].  No mask.
//   q: [B, Hq, D] bf16; out: [B, Hq, D] double; lse: [B, Hq] double.
int oracle_decode(double* out, double* lse, const uint16_t* q,
                  const uint16_t* k_cache, const uint16_t* v_cache,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                  int block_size, int64_t num_blocks, double scale, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || block_size <= 0)
    return -1;
  for (int b = 0; b < B; ++b) {
    if (context_lens[b] < 0) return -1;
    if (static_cast<int64_t>(context_lens[b]) >
        static_cast<int64_t>(max_blocks_per_seq) * block_size)
      return -6;
  }
  const int g = Hq / Hkv;
  std::vector<int> status(static_cast<size_t>(B) * Hkv, 0);
  parallel_for(static_cast<int64_t>(B) * Hkv, nthreads, [&](int64_t item) {
    const int b = static_cast<int>(item / Hkv);
    const int kvh = static_cast<int>(item % Hkv);
    const int64_t L = context_lens[b];
    std::vector<uint16_t> K, V;
    std::vector<double> s;
    if (!gather_head(k_cache, v_cache,
                     block_tables + static_cast<int64_t>(b) * max_blocks_per_seq, L,
                     Hkv, D, block_size, num_blocks, kvh, K, V)) {
      status[item] = -4;
      return;
    }
    const std::vector<double> Kd = widen(K), Vd = widen(V);
    for (int hh = 0; hh < g; ++hh) {
      const int h = kvh * g + hh;  // query heads of this kv head's group
      const int64_t r = static_cast<int64_t>(b) * Hq + h;
      attend_row_values(q + r * D, Kd, Vd, L, D, scale, s, out + r * D, lse + r);
    }
  });
  for (int st : status)
    if (st) return st;
  return 0;
}

// Prefill / chunked prefill over a prefix-cached pool.  Sequence i has
// Lq = cu_seqlens_q[i+1]-cu_seqlens_q[i] query rows and Lk =
// cu_seqlens_k[i+1]-cu_seqlens_k[i] keys; all Lk keys (cached prefix and the new
// tokens, which the store has already written) are read through
// block_tables[i, :].  Query row r sees keys j <= Lk - Lq + r.
//   q: [sum Lq, Hq, D] bf16; out: [sum Lq, Hq, D] double; lse: [sum Lq, Hq].
int oracle_prefill(double* out, double* lse, const uint16_t* q,
                   const uint16_t* k_cache, const uint16_t* v_cache,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                   int B, int Hq, int Hkv, int D, int block_size,
                   int64_t num_blocks, double scale, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || block_size <= 0)
    return -1;
  for (int i = 0; i < B; ++i) {
    const int64_t Lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
    const int64_t Lk = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
    if (Lq < 0 || Lk < 0) return -1;
    if (Lk < Lq) return -5;
    if (Lk > static_cast<int64_t>(max_blocks_per_seq) * block_size) return -6;
  }
  const int g = Hq / Hkv;
  const int rows_per_item = 64;
  // items: (sequence, kv head, block of query rows)
  std::vector<int64_t> item_seq, item_row0;
  for (int i = 0; i < B; ++i) {
    const int64_t Lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
    for (int64_t r0 = 0; r0 < Lq; r0 += rows_per_item) {
      item_seq.push_back(i);
      item_row0.push_back(r0);
    }
  }
  const int64_t n_row_items = static_cast<int64_t>(item_seq.size());
  std::vector<int> status(static_cast<size_t>(n_row_items) * Hkv, 0);
  parallel_for(n_row_items * Hkv, nthreads, [&](int64_t item) {
    const int64_t ri = item / Hkv;
    const int kvh = static_cast<int>(item % Hkv);
    const int i = static_cast<int>(item_seq[ri]);
    const int64_t r0 = item_row0[ri];
    const int64_t Lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
    const int64_t Lk = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
    const int64_t r1 = r0 + rows_per_item < Lq ? r0 + rows_per_item : Lq;
    std::vector<uint16_t> K, V;
    std::vector<double> s;
    if (!gather_head(k_cache, v_cache,
                     block_tables + static_cast<int64_t>(i) * max_blocks_per_seq, Lk,
                     Hkv, D, block_size, num_blocks, kvh, K, V)) {
      status[item] = -4;
      return;
    }
    const std::vector<double> Kd = widen(K), Vd = widen(V);
    for (int64_t r = r0; r < r1; ++r) {
      const int64_t n_visible = Lk - Lq + r + 1;  // keys 0 .. Lk-Lq+r
      const int64_t row = cu_seqlens_q[i] + r;
      for (int hh = 0; hh < g; ++hh) {
        const int h = kvh * g + hh;
        const int64_t o = row * Hq + h;
        attend_row_values(q + o * D, Kd, Vd, n_visible, D, scale, s, out + o * D, lse + o);
      }
    }
  });
  for (int st : status)
    if (st) return st;
  return 0;
}

int oracle_hardware_threads(void) { return resolve_threads(0); }

}  // extern "C"
