"""CPU tests of the oracle against its pins, and of the pins against planted mistakes."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle_pins as pins
from kv_cache_decode_06_b300.inputs import (
    CONFIGS, T5XXL_SWEEP_GS, bf16_bits_to_f32, f32_to_bf16_bits, make_decode_inputs,
)


@pytest.mark.parametrize("check", pins.DECODE_CHECKS + pins.VARIANT_CHECKS + pins.MEANPOOL_CHECKS,
                         ids=lambda c: c.__name__)
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)


def test_group_map_is_contiguous_blocks(oracle_lib):
    for H, G in ((8, 2), (32, 8), (64, 1), (64, 64), (12, 3)):
        assert [oracle.group_of(i, H, G, lib=oracle_lib) for i in range(H)] == [i // (H // G) for i in range(H)]


def test_oracle_rejects_bad_arguments(oracle_lib):
    inp = make_decode_inputs(CONFIGS["tiny"])
    with pytest.raises(ValueError):   # H % G != 0
        oracle.gqa_decode_f64(inp.q[:, :7], inp.k, inp.v, inp.seq_lens, inp.scale, lib=oracle_lib)
    with pytest.raises(ValueError):   # seq_len > Lmax
        oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens + 1, inp.scale, lib=oracle_lib)


# ------------------------------------------------------------ planted mistakes
# Each mutant edits one expression in a copy of the oracle source; at least one
# pin must then fail.  The mutants are compiled into a temporary directory and
# never replace the real oracle.

MUTANTS = {
    "group_map_modulo": ("return i / (H / G);", "return i % G;"),
    "scale_dropped": ("s[t] = sc * dot;", "s[t] = dot;"),
    "k_and_v_swapped": ("acc += s[t] * bf16_value(vg[(int64_t)t * d + j]);",
                        "acc += s[t] * bf16_value(kg[(int64_t)t * d + j]);"),
    "one_past_the_end": ("*T = seq_lens ? seq_lens[b] : Lmax;",
                         "*T = seq_lens ? (seq_lens[b] < Lmax ? seq_lens[b] + 1 : seq_lens[b]) : Lmax;"),
    "cross_attention_drops_last": ("*T = seq_lens ? seq_lens[b] : Lmax;", "*T = seq_lens ? seq_lens[b] : Lmax - 1;"),
    "window_one_too_wide": ("*t0 = (window > 0 && *T > window) ? *T - window : 0;",
                            "*t0 = (window > 0 && *T > window + 1) ? *T - window - 1 : 0;"),
    "window_ignored": ("*t0 = (window > 0 && *T > window) ? *T - window : 0;", "*t0 = 0;"),
    "gather_page_offset_swapped": ("+ t % page_size) * d;", "+ (t / page_size) % page_size) * d;"),
    "gather_wrong_table_row": ("table[(int64_t)b * max_pages + t / page_size]",
                               "table[(int64_t)(B - 1 - b) * max_pages + t / page_size]"),
    "append_one_row_early": ("* Lmax + (T - 1)) * d", "* Lmax + (T > 1 ? T - 2 : 0)) * d"),
    "normaliser_missing": ("o[j] = acc / l;", "o[j] = acc;"),
    "exp_of_unshifted_sum": ("l += s[t];", "l += s[t] * s[t];"),
    "meanpool_divides_by_H": ("out[(o * G + g) * inner + x] = acc / (float)n;",
                              "out[(o * G + g) * inner + x] = acc / (float)H;"),
    "meanpool_reverse_head_order": (
        "float acc = w[(o * H + (int64_t)g * n) * inner + x];\n"
        "                for (int j = 1; j < n; ++j)\n"
        "                    acc = acc + w[(o * H + (int64_t)g * n + j) * inner + x];",
        "float acc = w[(o * H + (int64_t)g * n + n - 1) * inner + x];\n"
        "                for (int j = 1; j < n; ++j)\n"
        "                    acc = acc + w[(o * H + (int64_t)g * n + n - 1 - j) * inner + x];"),
    "meanpool_sums_in_double": ("float acc = w[(o * H + (int64_t)g * n) * inner + x];",
                                "double acc = w[(o * H + (int64_t)g * n) * inner + x];"),
    "meanpool_interleaved_groups": ("acc = acc + w[(o * H + (int64_t)g * n + j) * inner + x];",
                                    "acc = acc + w[(o * H + (int64_t)j * G + g) * inner + x];"),
    "meanpool_drops_last_member": ("for (int j = 1; j < n; ++j)\n                    acc = acc + w",
                                   "for (int j = 1; j < n - 1; ++j)\n                    acc = acc + w"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutant pattern not found: {old!r}"
    mpath = mutant_dir / f"{name}.c"
    mpath.write_text(src.replace(old, new, 1))
    so = mutant_dir / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(mpath), "-lm"], check=True)
    lib = oracle.load(str(so))
    checks = pins.MEANPOOL_CHECKS if name.startswith("meanpool") else pins.DECODE_CHECKS + pins.VARIANT_CHECKS
    failed = []
    for check in checks:
        try:
            check(lib)
        except (AssertionError, ValueError):
            failed.append(check.__name__)
    assert failed, f"no pin caught mutant {name}"


# ------------------------------------------------------------- input recipe

def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.14159], dtype=np.float32)
    got = bf16_bits_to_f32(f32_to_bf16_bits(x))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa wins (1.0)
    assert got[1] == np.float32(1.0)
    assert got[2] == np.float32(1.0 + 2 ** -6)
    assert got[0] == 1.0 and got[4] == -2.5
    assert abs(float(got[5]) - 3.14159) <= 2 ** -7 * 4


def test_inputs_are_seeded_and_shaped():
    a = make_decode_inputs(CONFIGS["tiny"])
    b = make_decode_inputs(CONFIGS["tiny"])
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k, b.k)
    assert a.q.shape == (1, 8, 64) and a.k.shape == (1, 2, 128, 64) and a.seq_lens.tolist() == [128]
    m = CONFIGS["mistral7b"]
    from kv_cache_decode_06_b300.inputs import draw_seq_lens
    sl = draw_seq_lens(m)
    assert sl.shape == (16,) and sl.min() >= 1024 and sl.max() <= 4096
    for G in T5XXL_SWEEP_GS:
        c = CONFIGS["t5xxl_sweep"].with_G(G)
        assert c.H % c.G == 0


def test_outlier_keys_are_scaled_by_four():
    c = CONFIGS["llama3_70b"].with_(B=2, Lmax=4096, seq_lo=4096, seq_hi=4096)
    inp = make_decode_inputs(c)
    k = bf16_bits_to_f32(inp.k)
    rms = np.sqrt((k.astype(np.float64) ** 2).mean(axis=(1, 3)))   # [B, T]
    big = rms > 2.5
    frac = big.mean()
    assert 0.003 < frac < 0.03
    assert np.all(rms[big] > 3.0)


@pytest.mark.slow
def test_oracle_tiny_config_runs(oracle_lib):
    inp = make_decode_inputs(CONFIGS["tiny"])
    out = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, lib=oracle_lib)
    assert np.isfinite(out).all() and out.shape == (1, 8, 64)


def test_paged_layout_generator_round_trips(oracle_lib):
    """The benchmark's paged layout holds the contiguous cache: the oracle's gather gives it back."""
    from kv_cache_decode_06_b300.inputs import DecodeConfig, make_paged_layout
    cfg = DecodeConfig("pg", 70, B=3, H=8, G=2, d=16, Lmax=200, seq_lo=1, seq_hi=200)
    inp = make_decode_inputs(cfg, seq_lens=[200, 17, 1])
    for ps in (16, 64, 256):
        kp, vp, table = make_paged_layout(inp, ps, spare_pages=2)
        assert table.shape == (3, -(-200 // ps)) and kp.shape[0] == int((table >= 0).sum()) + 2
        kg = oracle.gather_pages(kp, table, inp.seq_lens, cfg.Lmax, lib=oracle_lib)
        vg = oracle.gather_pages(vp, table, inp.seq_lens, cfg.Lmax, lib=oracle_lib)
        for b, T in enumerate(inp.seq_lens):
            assert np.array_equal(kg[b, :, :T], inp.k[b, :, :T]) and np.array_equal(vg[b, :, :T], inp.v[b, :, :T])
