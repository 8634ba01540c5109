"""The seeded input generator: known answers, encoder correctness, recipe.

The generator feeds both the oracle and the CUDA path, so its own mistakes
cannot show up as a parity failure; these tests pin it to outside facts.
"""
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    n = 0
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(t, 16) for t in line.split()]
            ctr, key, want = v[:4], v[4:6], v[6:10]
            got = synth.philox4x32_10(key[0] | (key[1] << 32), ctr)
            assert [int(t) for t in got] == want
            n += 1
    assert n == 3


def test_e4m3_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.uniform(-464, 464, 20000),
        rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 8, 20000),
        # exact ties between neighbouring E4M3 values
        (np.arange(1, 448) + 0.5) * 2.0 ** -9,
        np.arange(0, 2.0 ** -6, 2.0 ** -11),
    ]).astype(np.float32)
    v = v[np.abs(v) < 464]  # torch's cast turns 464 and up into NaN; ours saturates
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = synth.f32_to_e4m3(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(v[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_encoder_saturates():
    got = synth.f32_to_e4m3([464.0, 1000.0, 1e30, -500.0, np.inf])
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]


def test_bf16_encoder_matches_torch_cast():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16(v), ref)


def test_block_scale_rule_and_round_trip():
    """scale = 2^(floor(log2 amax) - 8); decoded elements are within half an
    E4M3 step of the source, except those saturated at 448."""
    rng = np.random.default_rng(2)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for _ in range(300):
        v = (rng.standard_normal(32) * 2.0 ** rng.integers(-30, 30)).astype(np.float32)
        codes, sc = synth.quantise_block(v)
        amax = float(np.abs(v).max())
        assert sc == int(np.floor(np.log2(amax))) - 8 + 127
        scale = 2.0 ** (sc - 127)
        q = v.astype(np.float64) / scale
        dec = e4m3[codes]
        sat = np.abs(q) > 448
        assert np.all(np.abs(dec[sat]) == 448) and np.all(np.sign(dec[sat]) == np.sign(q[sat]))
        ok = ~sat
        # E4M3 spacing at |q| in [2^e, 2^(e+1)) is 2^(e-3); subnormal spacing 2^-9
        e = np.floor(np.log2(np.maximum(np.abs(q[ok]), 2.0 ** -6)))
        assert np.all(np.abs(dec[ok] - q[ok]) <= 2.0 ** (e - 4) + 1e-300)
    codes, sc = synth.quantise_block(np.zeros(32, np.float32))
    assert sc == 127 and not codes.any()


def test_weights_follow_the_recipe():
    H, I, E = 256, 128, 4
    gu, gus, raw = synth.gate_up(99, 0, E, H, I, raw=True)
    dn, dns, rawd = synth.down(99, 0, E, H, I, raw=True)
    # std = 1/sqrt(fan_in): fan_in = H for gate/up, I for down
    assert abs(raw.std() * np.sqrt(H) - 1) < 0.01
    assert abs(rawd.std() * np.sqrt(I) - 1) < 0.01
    assert abs(raw.mean()) < 0.01 / np.sqrt(H) * 10
    # codes and scales are the block quantisation of the raw values
    r = raw.reshape(-1, 32)
    c = gu.reshape(-1, 32)
    s = gus.reshape(-1)
    for i in range(0, r.shape[0], 97):
        cc, ss = synth.quantise_block(r[i])
        assert np.array_equal(cc, c[i]) and ss == s[i]


def test_weight_slices_regenerate_identically():
    H, I, E = 256, 64, 6
    gu, gus = synth.gate_up(5, 3, E, H, I)
    part, parts = synth.gate_up(5, 3, E, H, I, experts=(2, 4), threads=3)
    assert np.array_equal(part[2:4], gu[2:4]) and not part[:2].any()
    assert np.array_equal(parts[2:4], gus[2:4])
    other, _ = synth.gate_up(5, 4, E, H, I)  # another layer draws other numbers
    assert (other != gu).mean() > 0.9


def test_router_uniform_topk_and_weights():
    ids, w, lg = synth.route(1235, 0, 32, 128, 8, logits=True)
    for b in range(32):
        order = np.argsort(-lg[b], kind="stable")[:8]  # stable: ties to the lower id
        assert list(ids[b]) == list(order)
        p = np.exp(lg[b, ids[b]].astype(np.float64) - lg[b].max())
        assert np.allclose(w[b], p / p.sum(), rtol=1e-6)
    assert np.allclose(w.sum(1), 1, atol=1e-6)


def test_router_modes():
    ids, w = synth.route(1237, 0, 32, 128, 8, mode="fixed")
    assert (ids == np.array(synth.FIXED_EXPERTS)).all()
    ids, w = synth.route(1237, 0, 32, 128, 8, mode="disjoint")
    counts = np.bincount(ids.ravel(), minlength=128)
    assert (counts == 2).all()  # two permutations, every expert serves two tokens
    assert len(set(ids[:16].ravel())) == 128 and len(set(ids[16:].ravel())) == 128
    ids, w = synth.route(1237, 0, 32, 128, 8, mode="zipf")
    counts = np.bincount(ids.ravel(), minlength=128)
    assert counts[:4].sum() > counts[64:].sum()  # a few hot experts
    for mode in ("fixed", "disjoint", "zipf"):
        _, w = synth.route(1237, 0, 32, 128, 8, mode=mode)
        assert np.allclose(w.sum(1), 1, atol=1e-6)


def test_x_is_bf16_of_standard_normal():
    xs, raw = synth.x(1235, 0, 4, 2048, raw=True)
    ref = torch.from_numpy(raw).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(xs, ref)
    assert abs(raw.std() - 1) < 0.03


def test_unique_expert_bytes():
    ids = np.array([[1, 2], [2, 3], [-1, 200]], np.int32)
    per = 2 * 768 * 2048 + 2 * 768 * 64 + 2048 * 768 + 2048 * 24
    assert per == 4866048
    assert synth.unique_expert_bytes(ids, 128, 2048, 768) == 3 * per
