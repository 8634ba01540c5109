"""Pins of the accuracy study's MXFP8 activation quantiser, and the study's
direction on a small layer (CPU only)."""
import numpy as np
import pytest
import torch

import accuracy_study as acc


def test_e4m3_rounding_matches_torch_float8():
    rng = np.random.default_rng(5)
    q = np.concatenate([rng.normal(0, 40, 20000), rng.normal(0, 0.01, 20000),
                        rng.uniform(-600, 600, 5000), [0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10]])
    want = torch.from_numpy(np.clip(q, -448, 448)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = acc.round_to_e4m3(q)
    assert np.array_equal(np.abs(got), np.abs(want))
    assert np.all((got == 0) | (np.sign(got) == np.sign(q)))


def test_mxfp8_quantisation_scale_rule_and_fixed_points():
    # a block of E4M3 values times 2^-5 is representable exactly: unchanged
    vals = np.array([acc.round_to_e4m3(np.array([v]))[0] for v in np.linspace(-448, 448, 32)])
    blk = (vals * 2.0 ** -5)[None, :]
    blk[0, 0] = 448 * 2.0 ** -5  # amax 14 -> scale 2^(3-8)
    assert np.array_equal(acc.quantize_mxfp8(blk), blk)
    # amax = 300 -> scale 2^0; the E4M3 grid above 256 has step 32: 300 -> 288
    v = np.zeros((1, 32))
    v[0, 0] = 300.0
    assert acc.quantize_mxfp8(v)[0, 0] == 288.0
    # all-zero block stays zero
    assert not acc.quantize_mxfp8(np.zeros((2, 64))).any()


def test_bf16_activations_are_closer_than_mxfp8_ones():
    r = acc.study(seed=77, B=2, H=256, I=128, E=16, K=4)
    assert 0 < r["rel_rms_warp_decode"] < r["rel_rms_traditional"]
    assert r["ratio"] > 1.4
