"""Plants plausible slips in a copy of the oracle source and checks that the
pins in ``test_oracle_pins.py`` catch every one of them.  Runs on the CPU
only; the real oracle is never modified."""

import pytest

import oracle
from tests import test_oracle_pins as pins

# (name, text in pa_oracle.cpp, replacement)
MUTANTS = [
    ("causal_off_by_one", "causal ? pos + 1 : seq", "causal ? pos : seq"),
    ("causal_top_left", "const int64_t pos = ctx + (j - q0);", "const int64_t pos = (j - q0);"),
    ("gqa_strided_groups", "const int h = g * grp + r;\n        const E* qr",
     "const int h = r * Hkv + g;\n        const E* qr"),
    ("key_from_value_half", "const E* krow = pool + (((blk * 2 + 0)", "const E* krow = pool + (((blk * 2 + 1)"),
    ("block_offset_swapped", "const int64_t off = p % bs;", "const int64_t off = (p / bs) % bs;"),
    ("lse_base_two", "*lse = m + std::log(l);", "*lse = m + std::log2(l);"),
    ("scale_dropped", "s[p] = scale * acc;", "s[p] = acc;"),
    ("merge_weight_sign", "const double w = std::exp(l - m);", "const double w = std::exp(m - l);"),
    ("split_chunk_unaligned", "const int64_t chunk = ((per + bs - 1) / bs) * bs;",
     "const int64_t chunk = per;"),
    ("mla_value_from_rope_end", "for (int e = 0; e < dv; ++e) V[p * dv + e] = widen(c[e]);",
     "for (int e = 0; e < dv; ++e) V[p * dv + e] = widen(c[e + rope_dim]);"),
    ("cache_write_value_to_key", "std::memcpy(pool + ((blk * 2 + 1) * block_size + off) * row, value",
     "std::memcpy(pool + ((blk * 2 + 0) * block_size + off) * row, value"),
    ("e4m3_ties_away_from_zero", "double m = std::nearbyint(a / std::ldexp(1.0, e - 3));",
     "double m = std::round(a / std::ldexp(1.0, e - 3));"),
    ("e4m3_overflow_to_nan", "if (a >= 448.0) return sign | 0x7E;",
     "if (a >= 464.0) return sign | 0x7F;"),
    ("e4m3_subnormal_step", "v = std::ldexp(static_cast<double>(m), -9);",
     "v = std::ldexp(static_cast<double>(m), -10);"),
    ("fp8_quantise_multiplies", "kdst[e] = oracle_e4m3_encode(kx / k_scale);",
     "kdst[e] = oracle_e4m3_encode(kx * k_scale);"),
    ("fp8_scales_swapped",
     "const double sc = kv == 0 ? static_cast<double>(k_scale) : static_cast<double>(v_scale);",
     "const double sc = kv == 0 ? static_cast<double>(v_scale) : static_cast<double>(k_scale);"),
    ("mla_write_rope_first", "std::memcpy(dst + kv_lora_rank, k_pe + t * rope_dim",
     "std::memcpy(dst + 0, k_pe + t * rope_dim"),
    ("mla_write_row_stride", "uint16_t* dst = pool + (blk * block_size + off) * width;",
     "uint16_t* dst = pool + (blk * block_size + off) * kv_lora_rank;"),
    ("mla_prefill_unrounded", "if (round_kv) acc = round_bf16(acc);", ""),
    ("mla_prefill_rope_from_latent", "K[p * dk + dn + e] = widen(c[R + e]);",
     "K[p * dk + dn + e] = widen(c[e]);"),
    ("mla_prefill_weight_transposed", "widen(wh[static_cast<int64_t>(e) * R + r])",
     "widen(wh[static_cast<int64_t>(r) * wrow + e])"),
    ("window_one_short", "(window > 0 && visible > window) ? visible - window : 0",
     "(window > 0 && visible > window) ? visible - window + 1 : 0"),
    ("window_one_long", "(window > 0 && visible > window) ? visible - window : 0",
     "(window > 0 && visible > window + 1) ? visible - window - 1 : 0"),
]


def _run_pins():
    """Runs every pin against the currently routed oracle; returns the names
    of the pins that failed."""
    calls = []
    for name in dir(pins):
        fn = getattr(pins, name)
        if not name.startswith("test_") or not callable(fn):
            continue
        if name == "test_m1_paged_equals_contiguous":
            calls += [(name, lambda fn=fn: fn(oracle, [6, 1, 4])),
                      (name, lambda fn=fn: fn(oracle, [7, 3, 5]))]
        elif name == "test_split_then_merge_equals_unsplit":
            calls += [(name, lambda fn=fn, S=S: fn(oracle, S)) for S in (2, 7)]
        else:
            calls.append((name, lambda fn=fn: fn(oracle)))
    failed = set()
    for name, call in calls:
        try:
            call()
        except Exception:      # an assertion or an oracle error both count
            failed.add(name)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_slip(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = oracle.build_variant(src.replace(old, new), str(tmp_path / f"{name}.so"))
    with oracle.using_library(path):
        failed = _run_pins()
    assert failed, f"no pin caught the planted slip {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _run_pins() == set()
