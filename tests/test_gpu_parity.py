"""GPU parity: the CUDA kernels through the C-ABI against the CPU oracle.

Every case compares element by element with the tolerance in tests/parity.py,
on seeded synthetic inputs (synth/), at sizes that span several CTAs and leave
ragged tails, and on the Qwen-3-style layer (H=2048, I=768, E=128, K=8) at
B = 1..32 with the routing patterns of the benchmark.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_decode_gate_gb300 as wd

from parity import bf16_bits_to_f64, compare, from_dev_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

_WEIGHTS = {}


def weights(wl, layer=0):
    key = (wl.seed, layer, wl.H, wl.I, wl.E)
    if key not in _WEIGHTS:
        gu, gus = synth.gate_up(wl.seed, layer, wl.E, wl.H, wl.I)
        dn, dns = synth.down(wl.seed, layer, wl.E, wl.H, wl.I)
        _WEIGHTS.clear()  # keep one full layer in host memory at a time
        _WEIGHTS[key] = (gu, gus, dn, dns)
    return _WEIGHTS[key]


def inputs(wl, B, layer=0):
    xs = synth.x(wl.seed, layer, B, wl.H)
    ids, w = synth.route(wl.seed, layer, B, wl.E, wl.K, mode=wl.route)
    return xs, ids, w


def run_layer(dev, xs, ids, w, gu, gus, dn, dns, stream=None):
    B, K = ids.shape
    I = gu.shape[1] // 2
    layer = wd.MoEDecodeLayer(gu, gus, dn, dns, K=K, max_batch=B, device=dev)
    out = torch.empty((B, gu.shape[2]), dtype=torch.bfloat16, device=dev)
    layer(to_dev_bf16(xs, dev), to_dev(ids, dev), to_dev(w, dev), out=out, stream=stream)
    torch.cuda.synchronize(dev)
    h = layer.workspace[256:256 + B * K * I * 2].view(torch.int16).view(B, K, I)
    flag = wd.wd_moe_read_error_flag(layer.workspace)
    return from_dev_bf16(out), h.cpu().numpy().view(np.uint16), flag


def check_layer(dev, xs, ids, w, gu, gus, dn, dns, what):
    I, E = gu.shape[1] // 2, gu.shape[0]
    want, want_h, _, bad = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    got, got_h, flag = run_layer(dev, xs, ids, w, gu, gus, dn, dns)
    compare(got_h.reshape(-1, I), want_h.reshape(-1, I), what + " h")
    stats = compare(got, want, what + " out")
    assert flag == (1 if bad else 0)
    return stats


def test_tiny_layer(cuda_device):
    wl = synth.WORKLOADS["tiny"]
    s = check_layer(cuda_device, *inputs(wl, 1), *weights(wl), "tiny")
    assert s["frac_equal"] > 0.9


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 32])
def test_qwen3_layer_batch_sweep(cuda_device, B):
    wl = synth.WORKLOADS["qwen3_sweep"]
    s = check_layer(cuda_device, *inputs(wl, B), *weights(wl), f"sweep B={B}")
    assert s["frac_equal"] > 0.9


@pytest.mark.parametrize("name", ["qwen3_zipf", "qwen3_fixed", "qwen3_disjoint"])
def test_qwen3_routing_stress_b32(cuda_device, name):
    wl = synth.WORKLOADS[name]
    check_layer(cuda_device, *inputs(wl, 32), *weights(wl), name)


# The batches of the crossover sweep, beyond decode (B = 128 and 256 on the
# full-size layer, the built-in plan the bench times there): the GPU runs every
# token, the oracle a seeded sample of them.  A token's h rows and output
# depend only on its own x row, ids and weights, so the sampled rows are
# compared element by element.
@pytest.mark.parametrize("B", [128, 256])
def test_crossover_batches_on_sampled_tokens(cuda_device, B):
    wl = synth.WORKLOADS["qwen3_sweep"]
    xs, ids, w = inputs(wl, B)
    gu, gus, dn, dns = weights(wl)
    got, got_h, flag = run_layer(cuda_device, xs, ids, w, gu, gus, dn, dns)
    pick = np.sort(np.random.default_rng(B).choice(B, 12, replace=False))
    want, want_h, _, bad = oracle.moe_decode(xs[pick], ids[pick], w[pick], gu, gus, dn, dns,
                                             wl.I, wl.E, with_f64=True)
    what = f"B={B} sampled tokens {pick.tolist()} ({wd.wd_moe_describe_plan(B, wl.H, wl.I, wl.E, wl.K)})"
    compare(got_h[pick].reshape(-1, wl.I), want_h.reshape(-1, wl.I), what + " h")
    compare(got[pick], want, what + " out")
    assert flag == 0 and bad == 0


def test_gate_up_kernel_alone(cuda_device):
    wl = synth.WORKLOADS["qwen3_b1"]
    gu, gus, _, _ = weights(wl)
    for B in (1, 3):
        xs, ids, _ = inputs(wl, B)
        want = oracle.gate_up(xs, ids, gu, gus, wl.I, wl.E)
        h = torch.empty((B, wl.K, wl.I), dtype=torch.bfloat16, device=cuda_device)
        flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        wd.wd_moe_gate_up(to_dev_bf16(xs, cuda_device), to_dev(ids, cuda_device),
                          to_dev(gu, cuda_device), to_dev(gus, cuda_device), h, error_flag=flag)
        torch.cuda.synchronize()
        compare(from_dev_bf16(h).reshape(-1, wl.I), want.reshape(-1, wl.I), f"gate_up B={B}")
        assert int(flag.item()) == 0


def test_down_kernel_alone_on_oracle_h(cuda_device):
    """The second kernel gets the ORACLE's h, so its parity does not depend on the first."""
    wl = synth.WORKLOADS["qwen3_b1"]
    gu, gus, dn, dns = weights(wl)
    B = 4
    xs, ids, w = inputs(wl, B)
    h = oracle.gate_up(xs, ids, gu, gus, wl.I, wl.E)
    want = oracle.down(h, ids, w, dn, dns, wl.H, wl.E)
    out = torch.empty((B, wl.H), dtype=torch.bfloat16, device=cuda_device)
    wd.wd_moe_down(to_dev_bf16(h, cuda_device), to_dev(ids, cuda_device), to_dev(w, cuda_device),
                   to_dev(dn, cuda_device), to_dev(dns, cuda_device), out)
    torch.cuda.synchronize()
    compare(from_dev_bf16(out), want, "down")


def _random_case(seed, B, H, I, E, K, route="uniform"):
    wl = synth.Workload(f"ragged{seed}", seed, H, I, E, K, (B,), route=route)
    gu, gus = synth.gate_up(seed, 0, E, H, I)
    dn, dns = synth.down(seed, 0, E, H, I)
    return inputs(wl, B) + (gu, gus, dn, dns)


@pytest.mark.parametrize("B,H,I,E,K", [
    (1, 32, 32, 1, 1),        # smallest legal layer: one block per row
    (3, 288, 96, 5, 3),       # 9 and 3 blocks per row: most lanes idle, ragged
    (5, 1056, 160, 7, 2),     # 33 blocks per gate row: one lane gets two
    (2, 4096, 256, 4, 4),     # 128 blocks per gate row: four passes per lane
    (7, 2048, 2048, 6, 6),    # K2 virtual stream of 384 blocks: several passes
    (33, 512, 768, 16, 8),    # odd batch above 32
    (64, 2048, 768, 128, 8),  # batch 64 on the full-size layer
    (2, 128, 64, 3, 3),       # K == E: every expert routed
])
def test_ragged_and_edge_shapes(cuda_device, B, H, I, E, K):
    case = _random_case(100 + B + H + I, B, H, I, E, K)
    check_layer(cuda_device, *case, f"B={B} H={H} I={I} E={E} K={K}")


def test_bad_expert_ids_are_skipped_and_flagged(cuda_device):
    xs, ids, w, gu, gus, dn, dns = _random_case(7, 4, 256, 128, 8, 3)
    ids = ids.copy()
    ids[0, 1], ids[2, 0], ids[3, 2] = -1, 8, 1 << 30
    want, want_h, _, bad = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, 128, 8, with_f64=True)
    assert bad == 3
    got, got_h, flag = run_layer(cuda_device, xs, ids, w, gu, gus, dn, dns)
    assert flag == 1
    assert not got_h[0, 1].any() and not got_h[2, 0].any()
    compare(got, want, "bad ids")


def test_error_flag_clears_after_read(cuda_device):
    xs, ids, w, gu, gus, dn, dns = _random_case(8, 2, 256, 128, 8, 2)
    bad_ids = ids.copy()
    bad_ids[1, 1] = -5
    layer = wd.MoEDecodeLayer(gu, gus, dn, dns, K=2, max_batch=2, device=cuda_device)
    x_d = to_dev_bf16(xs, cuda_device)
    w_d = to_dev(w, cuda_device)
    layer(x_d, to_dev(bad_ids, cuda_device), w_d)
    assert wd.wd_moe_read_error_flag(layer.workspace) == 1
    layer(x_d, to_dev(ids, cuda_device), w_d)
    assert wd.wd_moe_read_error_flag(layer.workspace) == 0


def test_duplicate_ids_and_zero_weights(cuda_device):
    xs, ids, w, gu, gus, dn, dns = _random_case(9, 6, 512, 256, 8, 4)
    ids = ids.copy()
    w = w.copy()
    ids[0, :] = 3           # one expert four times
    ids[1, 1] = ids[1, 0]   # a duplicate pair
    w[2, :] = 0.0           # a token with all-zero routing weights
    w[3, 1] = 0.0
    check_layer(cuda_device, xs, ids, w, gu, gus, dn, dns, "duplicates / zero weights")


def test_extreme_block_scales(cuda_device):
    """Scales far from 1 (2^-40 .. 2^+20) and subnormal E4M3 codes in every block."""
    xs, ids, w, gu, gus, dn, dns = _random_case(10, 3, 512, 128, 6, 3)
    rng = np.random.default_rng(0)
    gus = (127 + rng.integers(-40, 8, gus.shape)).astype(np.uint8)
    dns = (127 + rng.integers(-20, 20, dns.shape)).astype(np.uint8)
    gu = gu.copy()
    gu[..., ::32] = rng.integers(1, 8, gu[..., ::32].shape)  # subnormal codes
    check_layer(cuda_device, xs, ids, w, gu, gus, dn, dns, "extreme scales")


def test_deterministic_and_stream_ordered(cuda_device):
    wl = synth.WORKLOADS["qwen3_sweep"]
    xs, ids, w = inputs(wl, 8)
    gu, gus, dn, dns = weights(wl)
    s = torch.cuda.Stream(device=cuda_device)
    with torch.cuda.stream(s):
        a, _, _ = run_layer(cuda_device, xs, ids, w, gu, gus, dn, dns, stream=s)
    b, _, _ = run_layer(cuda_device, xs, ids, w, gu, gus, dn, dns)
    assert np.array_equal(a, b)  # no atomics in any reduction: bit-identical reruns


def test_captured_in_a_cuda_graph(cuda_device):
    wl = synth.WORKLOADS["qwen3_sweep"]
    xs, ids, w = inputs(wl, 4)
    gu, gus, dn, dns = weights(wl)
    layer = wd.MoEDecodeLayer(gu, gus, dn, dns, K=wl.K, max_batch=4, device=cuda_device)
    x_d, ids_d, w_d = to_dev_bf16(xs, cuda_device), to_dev(ids, cuda_device), to_dev(w, cuda_device)
    out = torch.empty((4, wl.H), dtype=torch.bfloat16, device=cuda_device)
    s = torch.cuda.Stream(device=cuda_device)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer(x_d, ids_d, w_d, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    want = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, wl.I, wl.E)
    compare(from_dev_bf16(out), want, "graph replay")


def test_smaller_batch_reuses_a_larger_workspace(cuda_device):
    wl = synth.WORKLOADS["qwen3_sweep"]
    gu, gus, dn, dns = weights(wl)
    layer = wd.MoEDecodeLayer(gu, gus, dn, dns, K=wl.K, max_batch=32, device=cuda_device)
    for B in (32, 3):
        xs, ids, w = inputs(wl, B)
        out = layer(to_dev_bf16(xs, cuda_device), to_dev(ids, cuda_device), to_dev(w, cuda_device))
        torch.cuda.synchronize()
        want = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, wl.I, wl.E)
        compare(from_dev_bf16(out), want, f"shared workspace B={B}")
    assert wd.wd_moe_read_error_flag(layer.workspace) == 0


# every compiled kernel instance, selected through the plan override
PLANS = [
    "gu=batched:1:1,dn=1:1",
    "gu=batched:1:2,dn=1:2",
    "gu=batched:2:1,dn=2:1",
    "gu=batched:2:1,dn=2:3",
    "gu=rowshare:1:1,dn=4:1",
    "gu=rowshare:1:2,dn=4:2",
    "gu=rowshare:2:1,dn=2:2",
    "gu=rowshare:2:2,dn=1:6",
    "gu=batched:1:1,dn=1:4",
    "gu=persist:2:2,dn=4:1",
    "gu=persist:2:1,dn=2:2",
    "gu=persist:1:1,dn=2:3",
    "gu=persist:1:2,dn=dimblock",
    "gu=mma,dn=4:1",
    "gu=mma:2:16,dn=4:1",
    "gu=mma,dn=dimblock",
    "gu=mma,dn=dimblock:2:1:3:2",
    "gu=mma,dn=dimblock:4:3:1:2",
    "gu=mma,dn=dimblock:1:2:8:1",
    "gu=batched:2:1,dn=dimblock,pdl=0",
]

PLAN_SHAPES = [
    (3, 288, 96, 5, 3, "uniform"),
    (5, 1056, 160, 7, 2, "uniform"),
    (2, 4096, 256, 4, 4, "uniform"),
    (7, 2048, 2048, 6, 6, "uniform"),
    (33, 512, 768, 16, 8, "uniform"),
    (32, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "fixed"),
    (9, 512, 128, 8, 3, "uniform"),       # smallest shape both streamed kernels accept
    (17, 1024, 832, 20, 5, "uniform"),    # I = 832: ragged lane slices in both
    (12, 8192, 64, 3, 2, "uniform"),      # H = 8192: x of 3 tokens staged at a time, ~8 per expert
    (20, 1024, 96, 6, 4, "uniform"),      # smallest H the bulk-copy ring accepts, ~13 tokens per expert
]


@pytest.fixture
def plan_reset():
    yield
    wd.wd_moe_set_plan(None)


@pytest.mark.parametrize("B,H,I,E,K,route", PLAN_SHAPES)
def test_every_kernel_instance_matches_the_oracle(cuda_device, plan_reset, B, H, I, E, K, route):
    xs, ids, w, gu, gus, dn, dns = _random_case(300 + B + H + I + E, B, H, I, E, K, route=route)
    want, want_h, _, _ = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, I, E, with_f64=True)
    for plan in PLANS:
        wd.wd_moe_set_plan(plan)
        got, got_h, flag = run_layer(cuda_device, xs, ids, w, gu, gus, dn, dns)
        compare(got_h.reshape(-1, I), want_h.reshape(-1, I), f"{plan} h")
        compare(got, want, f"{plan} out")
        assert flag == 0, plan


@pytest.mark.parametrize("plan", ["gu=rowshare:2:2,rowshare_min_b=1,dn=2:3",
                                  "gu=persist:2:2,dn=4:1",
                                  "gu=mma,dn=4:1",
                                  "gu=batched:2:1,dn=dimblock",
                                  "gu=mma,dn=dimblock"])
def test_routing_table_kernels_handle_bad_ids(cuda_device, plan_reset, plan):
    wd.wd_moe_set_plan(plan)
    xs, ids, w, gu, gus, dn, dns = _random_case(17, 9, 512, 128, 8, 3)
    ids = ids.copy()
    ids[0, 1], ids[4, 0], ids[8, 2] = -1, 8, 99
    want, want_h, _, bad = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, 128, 8, with_f64=True)
    got, got_h, flag = run_layer(cuda_device, xs, ids, w, gu, gus, dn, dns)
    assert bad == 3 and flag == 1
    assert not got_h[0, 1].any() and not got_h[4, 0].any() and not got_h[8, 2].any()
    compare(got_h.reshape(-1, 128), want_h.reshape(-1, 128), "rowshare bad ids h")
    compare(got, want, "rowshare bad ids")


# moe_gate_up_mma: B*K <= 256, H % 512 == 0, H <= 2048, I % 16 == 0.  Shapes:
# the full-size layer at B = 8..32 with every routing pattern of the benchmark
# (fixed: 32 tokens per expert, four groups of 8 staged tokens; disjoint: 2 per
# expert), B*K = 256 (the table limit), two 256-column chunks per row (six
# consumer warps idle), six chunks (H = 1536), ~13 tokens per expert (two
# groups, the second partly empty), K == E, and a single token.
MMA_SHAPES = [
    (8, 2048, 768, 128, 8, "uniform"),
    (16, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "zipf"),
    (32, 2048, 768, 128, 8, "fixed"),
    (32, 2048, 768, 128, 8, "disjoint"),
    (64, 2048, 768, 128, 4, "uniform"),
    (5, 512, 64, 4, 2, "uniform"),
    (10, 1536, 32, 4, 2, "uniform"),
    (40, 1024, 128, 6, 2, "uniform"),
    (3, 1024, 256, 3, 3, "uniform"),
    (1, 2048, 768, 128, 8, "uniform"),
]


@pytest.mark.parametrize("warps", [8, 16])
@pytest.mark.parametrize("B,H,I,E,K,route", MMA_SHAPES)
def test_gate_up_mma_matches_the_oracle(cuda_device, plan_reset, B, H, I, E, K, route, warps):
    wd.wd_moe_set_plan(f"gu=mma:0:{warps},dn=4:1")
    assert f"gate_up=moe_gate_up_mma<{warps}," in wd.wd_moe_describe_plan(B, H, I, E, K)
    xs, ids, w, gu, gus, dn, dns = _random_case(900 + B + H + I + E, B, H, I, E, K, route=route)
    check_layer(cuda_device, xs, ids, w, gu, gus, dn, dns, f"gu=mma B={B} H={H} I={I} {route}")


def test_gate_up_mma_activation_range(cuda_device, plan_reset):
    """Tokens are re-encoded in FP16 with a per-token power-of-two scale: an
    ordinary token; one of magnitude 1e-15 (scaled up); one of 1e+15 (scaled
    down); all zeros; BF16 subnormals only; and a wide dynamic range (1e-12
    next to 1e+3), whose smallest values sit below the FP16 grid."""
    wd.wd_moe_set_plan("gu=mma,dn=4:1")
    xs, ids, w, gu, gus, dn, dns = _random_case(31, 6, 1024, 256, 8, 3)
    xf = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).float()
    xf[1] *= 1e-15
    xf[2] *= 1e15
    xf[3, :] = 0.0
    xf[4] = torch.sign(xf[4]) * 2.0 ** -130
    xf[5, ::2] *= 1e-12
    xf[5, 1] = 1e3
    xs = xf.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    I, E = 256, 8
    want_h = oracle.gate_up(xs, ids, gu, gus, I, E)
    h = torch.empty((6, 3, I), dtype=torch.bfloat16, device=cuda_device)
    wd.wd_moe_gate_up(to_dev_bf16(xs, cuda_device), to_dev(ids, cuda_device),
                      to_dev(gu, cuda_device), to_dev(gus, cuda_device), h)
    torch.cuda.synchronize()
    got_h = from_dev_bf16(h)
    for t in range(6):  # per token: each has its own output scale
        compare(got_h[t].reshape(-1, I), want_h[t].reshape(-1, I), f"gu=mma token {t}")


def test_gate_up_mma_special_scale_codes(cuda_device, plan_reset):
    """E8M0 code 0 (2^-127) on whole rows and code 255 (NaN) on one block: the
    NaN reaches exactly the outputs of that row, the rest matches the oracle."""
    wd.wd_moe_set_plan("gu=mma,dn=4:1")
    B, H, I, E, K = 4, 512, 128, 4, 2
    xs, ids, w, gu, gus, dn, dns = _random_case(33, B, H, I, E, K)
    ids = np.array([[0, 1], [1, 2], [0, 3], [2, 1]], dtype=np.int32)
    gus = gus.copy()
    gu = gu.copy()
    gus[1, 5, :] = 0        # gate row 5 of expert 1: every block at 2^-127
    gu[1, 5, :] = 0x70      # E4M3 128: products of ~2^-120 |x|
    gus[2, I + 7, 3] = 255  # up row 7 of expert 2: one NaN block
    want_h = oracle.gate_up(xs, ids, gu, gus, I, E)
    h = torch.empty((B, K, I), dtype=torch.bfloat16, device=cuda_device)
    wd.wd_moe_gate_up(to_dev_bf16(xs, cuda_device), to_dev(ids, cuda_device),
                      to_dev(gu, cuda_device), to_dev(gus, cuda_device), h)
    torch.cuda.synchronize()
    got = bf16_bits_to_f64(from_dev_bf16(h)).reshape(B, K, I)
    want = bf16_bits_to_f64(want_h).reshape(B, K, I)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.isnan(want).sum() == 2  # tokens 1 and 3 route expert 2 once each
    tiny = [(0, 1, 5), (1, 0, 5), (3, 1, 5)]  # (token, slot, neuron) through gate row 5 of expert 1
    for t, k, n in tiny:
        assert 0.0 < abs(want[t, k, n]) < 2.0 ** -100
        assert abs(got[t, k, n] - want[t, k, n]) <= 2.0 ** -7 * abs(want[t, k, n])
    got[np.isnan(got)] = 0.0
    want[np.isnan(want)] = 0.0
    err = np.abs(got - want).max()
    assert err <= 1e-2 * np.abs(want).max() + 2e-3


# moe_down_dimblock (after moe_h_encode): B <= 64, B*K <= 256, H % 16 == 0,
# I % 128 == 0, I <= 2048.  Shapes: the full-size layer at B = 8..64 with every
# routing pattern (fixed: 32 pairs per expert, six steps of up to 6; disjoint:
# 2 per expert), two CTAs (H = 32) and six (H = 96), I = 128 (four blocks per
# step), I = 2048 (a two-stage ring, one consumer warp), ~13 pairs per expert
# (a third, partly empty step), duplicate-prone K == E, and a single token;
# each with the built-in shape (at I = 768: 4 step groups of 2 warps, 3 stages
# per group, 8 pairs per step) and with (groups, stages per group, pairs,
# warps per step) = (2, 2, 8, 2), (1, 3, 3, 2) and (4, 2, 5, 1) where they fit
# (the built-in shape where they do not).
DN_SHAPES = [
    (8, 2048, 768, 128, 8, "uniform"),
    (16, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "zipf"),
    (32, 2048, 768, 128, 8, "fixed"),
    (32, 2048, 768, 128, 8, "disjoint"),
    (64, 2048, 768, 128, 4, "uniform"),
    (2, 32, 128, 2, 2, "uniform"),
    (3, 96, 256, 3, 3, "uniform"),
    (40, 1024, 128, 6, 2, "uniform"),
    (7, 512, 2048, 6, 6, "uniform"),
    (3, 512, 384, 3, 3, "uniform"),
    (1, 2048, 768, 128, 8, "uniform"),
]


@pytest.mark.parametrize("plan", ["dn=dimblock", "dn=dimblock:2:2:8:2", "dn=dimblock:1:3:3:2",
                                  "dn=dimblock:4:2:5:1"])
@pytest.mark.parametrize("B,H,I,E,K,route", DN_SHAPES)
def test_down_dimblock_matches_the_oracle(cuda_device, plan_reset, B, H, I, E, K, route, plan):
    wd.wd_moe_set_plan(plan)
    assert "down=moe_down_dimblock<" in wd.wd_moe_describe_plan(B, H, I, E, K)
    xs, ids, w, gu, gus, dn, dns = _random_case(1100 + B + H + I + E, B, H, I, E, K, route=route)
    check_layer(cuda_device, xs, ids, w, gu, gus, dn, dns, f"{plan} B={B} H={H} I={I} {route}")


def _down_alone(dev, h_bits, ids, w, dn, dns, H, E):
    """The down stage alone, on a given h, through wd_moe_down_workspace."""
    B, K, I = h_bits.shape
    want = oracle.down(h_bits, ids, w, dn, dns, H, E)
    out = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(wd.wd_moe_workspace_size(B, K, I), dtype=torch.uint8, device=dev)
    wd.wd_moe_workspace_init(ws)
    wd.wd_moe_down_workspace(to_dev_bf16(h_bits, dev), to_dev(ids, dev), to_dev(w, dev),
                             to_dev(dn, dev), to_dev(dns, dev), out, ws)
    torch.cuda.synchronize()
    return from_dev_bf16(out), want, wd.wd_moe_read_error_flag(ws)


@pytest.mark.parametrize("plan", ["dn=dimblock", "dn=4:1"])
def test_down_h_range_and_duplicates(cuda_device, plan_reset, plan):
    """h rows are re-encoded per (token, slot) as FP16 times a power of two:
    ordinary rows, rows of magnitude 1e-20 and 1e+20, an all-zero row, BF16
    subnormals only, a row spanning 1e-12 .. 1e+3; a token routed twice to one
    expert and a zero routing weight."""
    wd.wd_moe_set_plan(plan)
    B, H, I, E, K = 6, 256, 256, 4, 3
    xs, ids, w, gu, gus, dn, dns = _random_case(41, B, H, I, E, K)
    ids, w = ids.copy(), w.copy()
    ids[0, 2] = ids[0, 1]
    w[3, 0] = 0.0
    h = oracle.gate_up(xs, ids, gu, gus, I, E)
    hf = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float()
    hf[1] *= 1e-20
    hf[2] *= 1e20
    hf[3, 1, :] = 0.0
    hf[4, 0] = torch.sign(hf[4, 0]) * 2.0 ** -130
    hf[5, 2, ::2] *= 1e-12
    hf[5, 2, 1] = 1e3
    hb = hf.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got, want, flag = _down_alone(cuda_device, hb, ids, w, dn, dns, H, E)
    assert flag == 0
    for t in range(B):  # per token: the rows differ by up to 40 orders of magnitude
        compare(got[t:t + 1], want[t:t + 1], f"{plan} token {t}")


@pytest.mark.parametrize("plan", ["dn=dimblock", "dn=4:1"])
def test_down_special_scale_codes_and_bad_ids(cuda_device, plan_reset, plan):
    """E8M0 codes far from 1 (2^-40 .. 2^+19), 0 (2^-127) on a whole row and 255
    (NaN) on one block; an out-of-range id contributes nothing and is flagged."""
    wd.wd_moe_set_plan(plan)
    B, H, I, E, K = 4, 128, 256, 4, 2
    xs, ids, w, gu, gus, dn, dns = _random_case(43, B, H, I, E, K)
    ids = np.array([[0, 1], [1, 2], [0, 9], [2, 3]], dtype=np.int32)
    rng = np.random.default_rng(5)
    dns = (127 + rng.integers(-40, 20, dns.shape)).astype(np.uint8)
    dn = dn.copy()
    dn[..., ::32] = rng.integers(1, 8, dn[..., ::32].shape)  # subnormal E4M3 codes
    dns[3, 7, :] = 0       # expert 3, output dim 7: every block at 2^-127
    dns[1, 20, 2] = 255    # expert 1, output dim 20: one NaN block
    h = oracle.gate_up(xs, ids, gu, gus, I, E)
    got_b, want_b, flag = _down_alone(cuda_device, h, ids, w, dn, dns, H, E)
    assert flag == wd.FLAG_BAD_EXPERT_ID
    got, want = bf16_bits_to_f64(got_b), bf16_bits_to_f64(want_b)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.isnan(want[:, 20]).sum() == 2  # tokens 0 and 1 route expert 1
    got[np.isnan(got)] = 0.0
    want[np.isnan(want)] = 0.0
    err = np.abs(got - want).max()
    assert err <= 1e-2 * np.abs(want).max() + 2e-3


def test_down_workspace_matches_the_layer(cuda_device, plan_reset):
    """wd_moe_down_workspace on the layer's own h gives the layer's output, bit
    for bit (the same kernels in the same order)."""
    wl = synth.WORKLOADS["qwen3_sweep"]
    gu, gus, dn, dns = weights(wl)
    for B in (4, 16):
        xs, ids, w = inputs(wl, B)
        layer = wd.MoEDecodeLayer(gu, gus, dn, dns, K=wl.K, max_batch=B, device=cuda_device)
        ids_d, w_d = to_dev(ids, cuda_device), to_dev(w, cuda_device)
        out = layer(to_dev_bf16(xs, cuda_device), ids_d, w_d)
        h = layer.workspace[256:256 + B * wl.K * wl.I * 2].view(torch.bfloat16).view(B, wl.K, wl.I)
        h = h.clone()
        out2 = torch.empty_like(out)
        ws = torch.empty(wd.wd_moe_workspace_size(B, wl.K, wl.I), dtype=torch.uint8, device=cuda_device)
        wd.wd_moe_workspace_init(ws)
        wd.wd_moe_down_workspace(h, ids_d, w_d, layer.down, layer.down_scale, out2, ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), f"B={B}"


def test_error_flag_bits_map_to_statuses(cuda_device):
    """The flag read reports the raw mask and the status of its worst bit: a
    bounded wait that ran out (bit 1) wins over a skipped expert id (bit 0).
    The bits are planted with a device fill, no kernel has to fail."""
    ws = torch.empty(wd.wd_moe_workspace_size(1, 8, 768), dtype=torch.uint8, device=cuda_device)
    wd.wd_moe_workspace_init(ws)
    flag_word = ws[:4].view(torch.int32)
    for planted, status in ((0, 0), (1, 5), (2, 6), (3, 6)):
        flag_word.fill_(planted)
        mask, st = wd.wd_moe_read_error_flag(ws, with_status=True)
        assert (mask, wd.wd_status_string(st)) == (planted, wd.wd_status_string(status))
        assert wd.wd_moe_read_error_flag(ws) == 0  # cleared by the read
