"""Seeded input generators: splitmix64 against its published sequence, recipes."""
import numpy as np
import pytest

from tile_task_transformer_gb300 import synth


def test_splitmix64_published_sequence():
    # sequence of the splitmix64 generator seeded with 1234567 (state advanced by
    # the golden-ratio increment before each output), as published with the
    # algorithm's reference implementations
    g = 0x9E3779B97F4A7C15
    got = [int(synth.splitmix64(np.uint64((1234567 + k * g) % 2 ** 64))) for k in range(5)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_normal_statistics_and_determinism():
    a = synth.normal_f32(5, 3, 200001, 0.02)
    assert a.dtype == np.float32
    assert abs(a.mean()) < 3e-4 and abs(a.std() - 0.02) < 3e-4
    np.testing.assert_array_equal(a[:1000], synth.normal_f32(5, 3, 1000, 0.02))


def test_token_windows_range_and_shape():
    w = synth.token_windows(1, 4, 1024, 50257)
    assert w.shape == (4, 1025) and w.dtype == np.uint16
    assert w.max() < 50257
    # roughly uniform
    assert abs(w.astype(np.float64).mean() - 25128) < 600


def test_param_recipe():
    p = synth.gpt2_params(0, 2, 64, 256, 256, 32)
    names = [n for n, _ in synth.param_names_shapes(2, 64, 256, 256, 32)]
    assert list(p) == names and len(names) == 2 + 12 * 2 + 2
    assert np.all(p["h0.ln1.g"] == 1) and np.all(p["ln_f.b"] == 0)
    assert sum(v.size for v in p.values()) == 118528


@pytest.mark.parametrize("L,d,f,V,S,stated,half_unit", [
    (12, 768, 3072, 50257, 1024, 124.4e6, 0.05e6),  # GPT2-small shape (124.4M)
    (4, 8192, 32768, 50257, 1024, 3.6e9, 0.05e9),   # wide-4, stated as about 3.6B parameters
    (8, 16384, 65536, 50257, 1024, 26.6e9, 0.05e9), # wide-8, stated as about 26.6B parameters
])
def test_parameter_counts_match_the_stated_model_sizes(L, d, f, V, S, stated, half_unit):
    n = sum(int(np.prod(s)) for _, s in synth.param_names_shapes(L, d, f, V, S))
    assert abs(n - stated) <= half_unit, (n, stated)  # equal after rounding to the stated digits


def test_wide4_spread_golden_covers_every_parameter():
    """The stored accumulation spread of the wide-4 parity inputs (written by
    tests/golden/make_wide4_spread.py from the oracle alone) names every
    parameter tensor once, with spreads in (0, 5%)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "wide4_accumulation_spread.json")
    with open(path) as fh:
        d = json.load(fh)
    names = [n for n, _ in synth.param_names_shapes(4, 8192, 32768, 50257, 1024)]
    assert sorted(d["tensors"]) == sorted(names)
    for n, v in d["tensors"].items():
        assert 0 < v["two_norm"] < 0.05 and 0 < v["max_norm"] < 0.05, n
    assert abs(d["loss_fp32"] - d["loss_fp64"]) < 1e-3


def test_wide8_spread_golden_covers_the_compared_tensors():
    """The stored accumulation spread of the wide-8 parity inputs (written by
    tests/golden/make_wide8_spread.py from the oracle alone) covers ln_f, wte,
    wpe and the first and last blocks, with spreads in (0, 20%)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "wide8_accumulation_spread.json")
    with open(path) as fh:
        d = json.load(fh)
    names = [n for n, _ in synth.param_names_shapes(8, 16384, 65536, 50257, 1024)
             if n.startswith(("h0.", "h7.")) or n in ("wte", "wpe", "ln_f.g", "ln_f.b")]
    assert sorted(d["tensors"]) == sorted(names)
    for n, v in d["tensors"].items():
        assert 0 < v["two_norm"] < 0.2 and 0 < v["max_norm"] < 0.2, n
    assert 0 < d["logits"]["max_norm"] < 0.1
