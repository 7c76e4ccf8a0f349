"""Planted mistakes: each pin of the oracle must fail when a plausible mistake is put
into the oracle itself (CPU only).

``oracle.plant(name)`` switches on one deliberate error inside the C++ oracle
library for the enclosed calls.  For every mistake this file runs a pin that
depends on nothing but the pages' definitions (hand-worked values, brute-force
exact arithmetic, closed forms) and expects it to fail; the same pin passes
without the plant (it runs in ``test_oracle_ffn.py`` / ``test_oracle_codecs.py``).
"""
from fractions import Fraction

import numpy as np
import pytest

import brute
import oracle
import test_oracle_codecs as tc
import test_oracle_ffn as tf

PINS = [
    ("gate_up_swapped", tf.test_swiglu_matches_brute_force_and_gate_is_first_half),
    ("e4m3_ties_away", tc.test_e4m3_golden_roundings),
    ("e4m3_no_saturation", tc.test_e4m3_largest_finite_and_saturation),
    ("norm_unrounded_sum", tf.test_rmsnorm_reads_rounded_residual),
    ("gemm_drops_last_k", tf.test_gemm_matches_brute_force_nonsquare),
    ("silu_sign", tf.test_silu_identities),
    ("bf16_truncates", tc.test_bf16_golden_roundings),
    ("dsilu_no_correction", tf.test_swiglu_backward_matches_brute_force_and_layout),
    ("gemv_scale_by_first", tf.test_decode_matches_brute_force),
]


def test_every_plant_has_a_pin():
    assert {p for p, _ in PINS} | {"quant_divides"} == set(oracle.PLANTS)


@pytest.mark.parametrize("plant,pin", PINS, ids=[p for p, _ in PINS])
def test_planted_mistake_is_caught(plant, pin):
    with oracle.plant(plant):
        with pytest.raises(AssertionError):
            pin()
    pin()                                   # and passes again once the plant is gone


def _discriminating_values(amax):
    """bf16 values v whose fp32 product v * (448f / amax) and fp32 quotient v / (amax / 448f)
    round to different E4M3 codes, found by brute force over every positive finite bf16."""
    a = Fraction(float(amax))
    inv = brute.f32(Fraction(448) / a)
    scale = brute.f32(a / 448)
    found = []
    for bits in range(0x0001, 0x7F80):
        v = brute.bf16_value(bits)
        if v > a:
            break
        if brute.round_e4m3_satfinite(brute.f32(v * inv)) != brute.round_e4m3_satfinite(brute.f32(v / scale)):
            found.append(bits)
    return found


def test_quantize_scales_by_a_product_pin():
    """R6: each element is scaled by the fp32 product with 448 / abs-max, not divided by
    the scale.  At abs-max 3.0625 the two forms differ in the E4M3 code of 30 bf16 values;
    the oracle must give the product's codes there, and the planted division must not."""
    amax = np.float32(3.0625)
    vals = _discriminating_values(amax)
    assert vals, "no discriminating value at this abs-max"
    v = np.array(vals, dtype=np.uint16)
    want, scale = brute.quantize([int(b) for b in v], float(amax))
    codes, s = oracle.quantize_with_abs_max(v, amax)
    assert list(codes) == want and Fraction(float(s)) == scale
    with oracle.plant("quant_divides"):
        planted, _ = oracle.quantize_with_abs_max(v, amax)
    assert list(planted) != want


def test_results_do_not_depend_on_the_thread_count():
    """Each output is computed by one thread in a fixed order: 1 thread and all threads agree."""
    from ffn_inputs import PrefillConfig, prefill_inputs
    cfg = PrefillConfig("threads", B=1, T=37, C=256, H=384, eps=1e-5, seed=3)
    inp = prefill_inputs(cfg)
    w1q, w1s = oracle.quantize_tensor(inp["w1"])
    w2q, w2s = oracle.quantize_tensor(inp["w2"])
    n = oracle.max_threads()
    try:
        oracle.set_threads(1)
        one = oracle.ffn_forward(inp["res"], inp["x"], inp["gain"], inp["eps"], w1q, w1s, w2q, w2s, cfg.H)
    finally:
        oracle.set_threads(n)
    many = oracle.ffn_forward(inp["res"], inp["x"], inp["gain"], inp["eps"], w1q, w1s, w2q, w2s, cfg.H)
    for k in one:
        np.testing.assert_array_equal(one[k], many[k], err_msg=k)
