"""Pins for the CPU oracle: each test checks it against something other than itself.

- number formats: all 256 E4M3 / E8M0 codes against PyTorch's independent FP8
  decoders and the OCP MX special values (tests/golden/);
- BF16 rounding: against an exhaustive nearest-value search over all 65536
  BF16 patterns;
- SiLU: against scipy's logistic function and the identity silu(g)-silu(-g)=g;
- the layer: against a brute-force dense evaluation over ALL experts with a
  gating matrix that is zero off the top-k (numpy matmuls, its own decode and
  rounding), closed forms, and the invariants the method implies (top-k order,
  zero routing weight, linearity in the routing weights, k=1 equals the dense
  FFN of that expert).

The layer follows the warp-decode blog (Cursor, "用 warp decode 实现更好的 MoE
模型推理"), section 两个 kernel 如何工作 (SiLU(gate)*up, then the down projection
weighted by the routing weights) and section 精度提升 (BF16 activations, wide
accumulation).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ formats --

def _torch_fp8_values(dtype):
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(dtype).to(torch.float64).numpy()


def test_e4m3_all_codes_match_independent_decoder():
    ref = _torch_fp8_values(torch.float8_e4m3fn)
    got = np.array([oracle.e4m3(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))  # -0.0 for 0x80
    assert int(np.isnan(got).sum()) == 2  # only 0x7F and 0xFF


def test_e8m0_all_codes_match_independent_decoder():
    ref = _torch_fp8_values(torch.float8_e8m0fnu)
    got = np.array([oracle.e8m0(c) for c in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_format_special_values_from_the_ocp_spec():
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_e8m0_special_values.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            fmt, code, val = line.split()[:3]
            got = (oracle.e4m3 if fmt == "E4M3" else oracle.e8m0)(int(code, 16))
            want = float(val)
            if math.isnan(want):
                assert math.isnan(got), (fmt, code)
            else:
                assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt, code)
            n += 1
    assert n == 14


def _bf16_table():
    """All finite BF16 values as float64 with their bit patterns, sorted by value."""
    bits = np.arange(65536, dtype=np.uint32)
    f32 = (bits << 16).astype(np.uint32).view(np.float32)
    finite = np.isfinite(f32) & (bits != 0x8000)  # keep +0 only
    vals = np.where(finite, f32, 0).astype(np.float64)
    bits, vals = bits[finite], vals[finite]
    order = np.argsort(vals, kind="stable")
    return vals[order], bits[order]


def _nearest_bf16(v, table):
    """Exhaustive search: nearest BF16 value, ties to the even bit pattern."""
    vals, bits = table
    i = np.searchsorted(vals, v)
    out = []
    for vi, ii in zip(v, i):
        cands = [j for j in (ii - 1, ii) if 0 <= j < len(vals)]
        best = min(cands, key=lambda j: (abs(vals[j] - vi), bits[j] & 1))
        # magnitude beyond the largest finite + half an ulp rounds to infinity
        maxv = vals[-1]
        if abs(vi) >= maxv + 2.0 ** (127 - 8):
            out.append(0x7F80 | (0x8000 if vi < 0 else 0))
            continue
        b = int(bits[best])
        if vals[best] == 0.0 and vi < 0:
            b = 0x8000
        out.append(b)
    return np.array(out, dtype=np.uint16)


def test_bf16_rounding_matches_exhaustive_nearest_search():
    rng = np.random.default_rng(7)
    table = _bf16_table()
    vals, _ = table
    # exact midpoints between neighbours (ties), and one FP64 ulp either side
    mids = (vals[:-1] + vals[1:]) / 2
    pick = rng.choice(mids.size, 3000, replace=False)
    m = mids[pick]
    cases = [m, np.nextafter(m, np.inf), np.nextafter(m, -np.inf)]
    cases.append(rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000))
    cases.append(rng.uniform(-2.0 ** -126, 2.0 ** -126, 2000))  # subnormal range
    cases.append(np.array([0.0, 1.0, -1.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135,
                           3.3895313892515355e38, 3.3961775292304563e38, -3.3961775292304563e38]))
    v = np.concatenate(cases)
    want = _nearest_bf16(v, table)
    got = np.array([oracle.f64_to_bf16(t) for t in v], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(v[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_bf16_to_f64_is_exact_widening():
    b = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(t)) for t in b[::97]])
    r = ref[::97]
    same = (got == r) | (np.isnan(got) & np.isnan(r))
    assert same.all()


def test_silu_against_scipy_and_odd_identity():
    from scipy.special import expit

    g = np.concatenate([np.linspace(-30, 30, 301), [0.0, 1e-300, -745.0, 745.0]])
    got = np.array([oracle.silu(t) for t in g])
    assert np.allclose(got, g * expit(g), rtol=1e-14, atol=1e-300)
    # silu(g) - silu(-g) = g for every g (sigma(g) + sigma(-g) = 1)
    neg = np.array([oracle.silu(-t) for t in g])
    assert np.allclose(got - neg, g, rtol=1e-13, atol=1e-13)
    assert oracle.silu(0.0) == 0.0


# ---------------------------------------------------------------- the layer --

def _random_layer(rng, B, H, I, E, K, scale_spread=3, distinct=True):
    """Random codes over the whole finite E4M3 range (subnormals included)."""
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    gu = rng.choice(finite, (E, 2 * I, H))
    dn = rng.choice(finite, (E, H, I))
    # scales near 2^-8 so that products stay O(1); spread tests the per-block indexing
    gus = (127 - 8 + rng.integers(-scale_spread, scale_spread + 1, (E, 2 * I, H // 32))).astype(np.uint8)
    dns = (127 - 8 + rng.integers(-scale_spread, scale_spread + 1, (E, H, I // 32))).astype(np.uint8)
    xb = torch.from_numpy(rng.standard_normal((B, H)).astype(np.float32)).to(torch.bfloat16)
    x = xb.view(torch.int16).numpy().view(np.uint16)
    if distinct:
        ids = np.stack([rng.choice(E, K, replace=False) for _ in range(B)]).astype(np.int32)
    else:
        ids = rng.integers(0, E, (B, K)).astype(np.int32)
    w = rng.dirichlet(np.ones(K), B).astype(np.float32)
    return x, ids, w, gu, gus, dn, dns


def _dequant(codes, scales):
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = torch.from_numpy(scales).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    return v * np.repeat(s, 32, axis=-1)


_TABLE = None


def _bf16_round_vec(v):
    """Round FP64 values to BF16 (returned as FP64) by nearest-value search in
    the sorted table of all finite BF16 values; ties go to the even pattern.
    Inputs must lie within the finite BF16 range."""
    global _TABLE
    if _TABLE is None:
        _TABLE = _bf16_table()
    vals, bits = _TABLE
    v = np.asarray(v, np.float64)
    i = np.clip(np.searchsorted(vals, v), 1, vals.size - 1)
    lo, hi = vals[i - 1], vals[i]
    dlo, dhi = np.abs(v - lo), np.abs(hi - v)
    pick_lo = (dlo < dhi) | ((dlo == dhi) & ((bits[i - 1] & 1) == 0))
    return np.where(pick_lo, lo, hi)


def _brute_force(x, ids, w, gu, gus, dn, dns, I, E):
    """Dense evaluation over every expert with a [B,E] gating matrix."""
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    WG, WD = _dequant(gu, gus), _dequant(dn, dns)
    B, K = ids.shape
    G = np.zeros((B, E))
    for b in range(B):
        for k in range(K):
            G[b, ids[b, k]] += float(w[b, k])
    y = np.zeros((B, x.shape[1]))
    hs = {}
    for e in range(E):
        g = X @ WG[e, :I].T
        u = X @ WG[e, I:].T
        hb = _bf16_round_vec(g / (1.0 + np.exp(-g)) * u)
        hs[e] = hb
        y += G[:, e:e + 1] * (hb @ WD[e].T)
    return y, hs


def test_bf16_helper_of_the_brute_force_agrees_with_exhaustive_search():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(4000) * 10.0 ** rng.integers(-20, 20, 4000)
    want = _nearest_bf16(v, _bf16_table())
    got = _bf16_round_vec(v).astype(np.float32).view(np.uint32) >> 16
    assert np.array_equal(got.astype(np.uint16), want)


@pytest.mark.parametrize("B,H,I,E,K,distinct", [(3, 64, 32, 4, 2, True), (2, 96, 64, 5, 3, True),
                                                (4, 64, 32, 3, 3, False)])
def test_layer_matches_brute_force_dense_evaluation(B, H, I, E, K, distinct):
    rng = np.random.default_rng(B * 1000 + H + I + E + K)
    x, ids, w, gu, gus, dn, dns = _random_layer(rng, B, H, I, E, K, distinct=distinct)
    out, h, y, bad = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    assert bad == 0
    y_ref, hs = _brute_force(x, ids, w, gu, gus, dn, dns, I, E)
    # h: the brute force's BF16 value of the same (token, expert) neuron
    hv = oracle.bf16_bits_to_f64(h)
    for b in range(B):
        for k in range(K):
            assert np.array_equal(hv[b, k], hs[ids[b, k]][b]), (b, k)
    scale = np.abs(y_ref).max()
    assert np.allclose(y, y_ref, rtol=0, atol=1e-12 * scale)
    # out is y rounded once
    assert np.array_equal(oracle.bf16_bits_to_f64(out), _bf16_round_vec(y))


def test_split_projections_compose_to_the_layer():
    rng = np.random.default_rng(11)
    I, E = 32, 4
    x, ids, w, gu, gus, dn, dns = _random_layer(rng, 2, 64, I, E, 2)
    out, h, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    h2 = oracle.gate_up(x, ids, gu, gus, I, E)
    out2 = oracle.down(h2, ids, w, dn, dns, 64, E)
    assert np.array_equal(h, h2) and np.array_equal(out, out2)


def test_closed_form_constant_weights():
    """gate = a, up = c, down = 1 everywhere, x = t: every neuron sees g = H a t,
    u = H c t, so y[d] = sum_k w_k * I * bf16(silu(g) u) for every d."""
    B, H, I, E, K = 1, 64, 32, 3, 2
    gu = np.zeros((E, 2 * I, H), np.uint8)
    gu[:, :I, :] = 0x30   # 0.5
    gu[:, I:, :] = 0x3C   # 1.5
    gus = np.full((E, 2 * I, H // 32), 127, np.uint8)
    dn = np.full((E, H, I), 0x38, np.uint8)     # 1.0
    dns = np.full((E, H, I // 32), 126, np.uint8)  # scale 0.5 -> down weight 0.5
    t = 0.1875  # exact in BF16
    x = np.full((B, H), 0, np.uint16)
    x[:] = torch.tensor([t], dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
    ids = np.array([[2, 0]], np.int32)
    w = np.array([[0.75, 0.25]], np.float32)
    out, h, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    g, u = H * 0.5 * t, H * 1.5 * t
    hval = g / (1 + math.exp(-g)) * u
    hb = float(torch.tensor([hval], dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
               .to(torch.float64)[0])
    assert np.all(oracle.bf16_bits_to_f64(h) == hb)
    assert np.allclose(y, (0.75 + 0.25) * I * 0.5 * hb, rtol=1e-15)


def test_closed_form_single_nonzero_weights_pick_the_right_operands():
    """One nonzero weight per matrix checks every index: gate row n, up row I+n,
    column j, the scale of column block j/32, and down row d column i."""
    B, H, I, E, K = 1, 64, 32, 2, 1
    n, j, d = 5, 37, 50
    i = n  # the down column that meets the only nonzero neuron
    gu = np.zeros((E, 2 * I, H), np.uint8)
    gus = np.full((E, 2 * I, H // 32), 127, np.uint8)
    dn = np.zeros((E, H, I), np.uint8)
    dns = np.full((E, H, I // 32), 127, np.uint8)
    e = 1
    gu[e, n, j] = 0x40        # 2.0
    gus[e, n, j // 32] = 128  # x2 -> gate weight 4
    gu[e, I + n, j] = 0xB8    # -1.0
    gus[e, I + n, 1 - j // 32] = 200  # a scale of the OTHER block must not matter
    dn[e, d, i] = 0x48        # 4.0
    dns[e, d, i // 32] = 125  # /4 -> down weight 1
    dn[e, d + 1, i + 1] = 0x48  # meets a zero neuron: must not contribute
    x = np.zeros((B, H), np.uint16)
    x[0, j] = 0x3F80          # 1.0
    ids = np.array([[e]], np.int32)
    w = np.array([[0.5]], np.float32)
    out, h, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    g, u = 4.0, -1.0
    hval = g / (1 + math.exp(-g)) * u
    hv = oracle.bf16_bits_to_f64(h)
    assert hv[0, 0, n] == _bf16_round_vec([hval])[0]
    assert np.count_nonzero(hv) == 1
    want = np.zeros(H)
    want[d] = 0.5 * 1.0 * hv[0, 0, n]
    assert np.array_equal(y[0], want)


def test_invariant_topk_order_does_not_matter():
    rng = np.random.default_rng(5)
    I, E, K = 32, 6, 4
    x, ids, w, gu, gus, dn, dns = _random_layer(rng, 3, 64, I, E, K)
    out, _, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    perm = rng.permutation(K)
    out2, _, y2, _ = oracle.moe_decode(x, ids[:, perm], w[:, perm], gu, gus, dn, dns, I, E,
                                       with_f64=True)
    assert np.allclose(y, y2, rtol=0, atol=1e-13 * np.abs(y).max())
    # BF16 outputs agree except where y sits within a few FP64 ulps of a rounding tie
    assert np.mean(out == out2) > 0.99


def test_invariant_zero_weight_expert_contributes_nothing():
    rng = np.random.default_rng(6)
    I, E, K = 32, 6, 3
    x, ids, w, gu, gus, dn, dns = _random_layer(rng, 2, 64, I, E, K)
    w[:, 1] = 0.0
    _, _, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    ids2 = ids.copy()
    ids2[:, 1] = np.array([e for e in range(E) if e not in ids[0]][0])  # another expert
    ids2[1, 1] = np.array([e for e in range(E) if e not in ids[1]][0])
    _, _, y2, _ = oracle.moe_decode(x, ids2, w, gu, gus, dn, dns, I, E, with_f64=True)
    assert np.array_equal(y, y2)


def test_invariant_linear_in_routing_weights():
    rng = np.random.default_rng(8)
    I, E, K = 32, 5, 3
    x, ids, w, gu, gus, dn, dns = _random_layer(rng, 2, 64, I, E, K)
    _, _, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    _, _, y4, _ = oracle.moe_decode(x, ids, w * 4, gu, gus, dn, dns, I, E, with_f64=True)
    assert np.array_equal(y4, 4 * y)  # a power of two scales exactly
    w2 = rng.dirichlet(np.ones(K), 2).astype(np.float32)
    _, _, ya, _ = oracle.moe_decode(x, ids, w2, gu, gus, dn, dns, I, E, with_f64=True)
    _, _, yab, _ = oracle.moe_decode(x, ids, (w.astype(np.float64) + w2).astype(np.float32),
                                     gu, gus, dn, dns, I, E, with_f64=True)
    # (w + w2) is rounded to FP32, so compare within that rounding
    assert np.allclose(yab, y + ya, rtol=0, atol=1e-6 * np.abs(yab).max())


def test_invariant_k1_unit_weight_is_the_dense_ffn_of_that_expert():
    rng = np.random.default_rng(9)
    B, H, I, E = 3, 64, 32, 4
    x, _, _, gu, gus, dn, dns = _random_layer(rng, B, H, I, E, 1)
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    WG, WD = _dequant(gu, gus), _dequant(dn, dns)
    for e in range(E):
        ids = np.full((B, 1), e, np.int32)
        w = np.ones((B, 1), np.float32)
        _, _, y, _ = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
        g, u = X @ WG[e, :I].T, X @ WG[e, I:].T
        dense = _bf16_round_vec(g / (1 + np.exp(-g)) * u) @ WD[e].T
        assert np.allclose(y, dense, rtol=0, atol=1e-12 * np.abs(dense).max())


def test_duplicate_ids_sum_their_weights():
    rng = np.random.default_rng(10)
    I, E = 32, 4
    x, _, _, gu, gus, dn, dns = _random_layer(rng, 1, 64, I, E, 2)
    _, _, y2, _ = oracle.moe_decode(x, np.array([[1, 1]], np.int32), np.array([[0.25, 0.5]], np.float32),
                                    gu, gus, dn, dns, I, E, with_f64=True)
    _, _, y1, _ = oracle.moe_decode(x, np.array([[1]], np.int32), np.array([[0.75]], np.float32),
                                    gu, gus, dn, dns, I, E, with_f64=True)
    assert np.allclose(y2, y1, rtol=0, atol=1e-14 * np.abs(y1).max())


def test_out_of_range_ids_contribute_nothing_and_are_counted():
    rng = np.random.default_rng(12)
    I, E, K = 32, 4, 3
    x, ids, w, gu, gus, dn, dns = _random_layer(rng, 2, 64, I, E, K)
    bad_ids = ids.copy()
    bad_ids[0, 1], bad_ids[1, 2] = -1, E
    out, h, y, bad = oracle.moe_decode(x, bad_ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    assert bad == 2
    assert np.all(h[0, 1] == 0) and np.all(h[1, 2] == 0)
    w0 = w.copy()
    w0[0, 1] = w0[1, 2] = 0.0
    _, _, y0, _ = oracle.moe_decode(x, ids, w0, gu, gus, dn, dns, I, E, with_f64=True)
    assert np.array_equal(y, y0)
