"""Plant plausible mistakes in copies of the oracle (on the CPU) and require the
pins to catch every one.  The oracle source is never modified; each mutant is
compiled from a patched copy in a temporary directory."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.cpp")

# (name, original text, mutated text) — each original must occur exactly once.
MUTANTS = [
    ("gqa-interleaved-heads", "const int h = kvh * g + hh;  // query heads",
     "const int h = hh * Hkv + kvh;  // query heads"),
    ("gather-wrong-block-index", "const int32_t blk = table_row[j / block_size];",
     "const int32_t blk = table_row[j % block_size];"),
    ("gather-offset-off-by-one",
     "const int64_t slot = static_cast<int64_t>(blk) * block_size + j % block_size;",
     "const int64_t slot = static_cast<int64_t>(blk) * block_size + (j + 1) % block_size;"),
    ("causal-off-by-one", "const int64_t n_visible = Lk - Lq + r + 1;",
     "const int64_t n_visible = Lk - Lq + r;"),
    ("causal-top-left", "const int64_t n_visible = Lk - Lq + r + 1;",
     "const int64_t n_visible = r + 1;"),
    ("no-scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("lse-without-max", "*lse = m + std::log(l);", "*lse = std::log(l);"),
    ("lse-log2", "*lse = m + std::log(l);", "*lse = m + std::log2(l);"),
    ("no-normalisation", "for (int d = 0; d < D; ++d) out[d] /= l;",
     "for (int d = 0; d < D; ++d) out[d] /= 1.0;"),
    ("pv-uses-keys", "out[d] += s[j] * V[static_cast<size_t>(j) * D + d];",
     "out[d] += s[j] * K[static_cast<size_t>(j) * D + d];"),
    ("gather-swaps-k-v",
     "std::memcpy(&K[static_cast<size_t>(j) * D], k_cache + src, sizeof(T) * D);",
     "std::memcpy(&K[static_cast<size_t>(j) * D], v_cache + src, sizeof(T) * D);"),
    ("store-swaps-block-offset", "const int64_t dst = (blk * block_size + off) * row;",
     "const int64_t dst = (off * num_blocks + blk) * row;"),
    ("store-k-into-v", "std::memcpy(v_cache + dst, v + t * v_tok_stride, sizeof(uint16_t) * row);",
     "std::memcpy(v_cache + dst, k + t * k_tok_stride, sizeof(uint16_t) * row);"),
    ("store-no-duplicate-check", "if (seen[s]) return -3;", "if (false) return -3;"),
    ("copy-blocks-k-from-v",
     "std::memcpy(k_cache + dst[i] * block_elems, k_cache + src[i] * block_elems,",
     "std::memcpy(k_cache + dst[i] * block_elems, v_cache + src[i] * block_elems,"),
    ("copy-blocks-wrong-direction",
     "std::memcpy(v_cache + dst[i] * block_elems, v_cache + src[i] * block_elems,",
     "std::memcpy(v_cache + src[i] * block_elems, v_cache + dst[i] * block_elems,"),
    ("prefill-wrong-q-row", "const int64_t o = row * Hq + h;",
     "const int64_t o = row * Hq + hh;"),
    ("softmax-max-not-subtracted-from-weights", "s[j] = std::exp(s[j] - m);",
     "s[j] = std::exp(s[j]);"),
    ("e4m3-bias-8", "mag = std::ldexp(1.0 + m / 8.0, e - 7);",
     "mag = std::ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3-subnormal-quantum", "mag = std::ldexp(static_cast<double>(m), -9);",
     "mag = std::ldexp(static_cast<double>(m), -10);"),
    ("e4m3-ties-away-from-zero", "double m = std::nearbyint(a / quantum);",
     "double m = std::round(a / quantum);"),
    ("e4m3-overflow-to-nan", "if (e > 8 || (e == 8 && m > 14.0)) return sign | 0x7E;",
     "if (e > 8 || (e == 8 && m > 14.0)) return sign | 0x7F;"),
    ("e4m3-infinity-not-saturated", "if (std::isinf(a)) return sign | 0x7E;",
     "if (std::isinf(a) && false) return sign | 0x7E;"),
    ("e4m3-subnormal-binade", "if (e < -6) e = -6;", "if (e < -7) e = -7;"),
    ("quantize-divides", "const float v = x * inv_scale;", "const float v = x / inv_scale;"),
    ("fp8-decode-k-uses-v-scale", "K[i] = e4m3_value(Kc[i]) * k_scale;",
     "K[i] = e4m3_value(Kc[i]) * v_scale;"),
    ("fp8-store-v-with-k-scale",
     "v_cache[s * row + i] = quantize(v[t * v_tok_stride + i], v_inv_scale);",
     "v_cache[s * row + i] = quantize(v[t * v_tok_stride + i], k_inv_scale);"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, mut):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor not unique/present: {orig!r}"
    path = tmp_path / f"mut_{name}.cpp"
    path.write_text(src.replace(orig, mut))
    so = oracle.build(str(path), str(tmp_path / f"libmut_{name}.so"))
    lib = oracle.load(so)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError) as e:  # caught by this pin
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
