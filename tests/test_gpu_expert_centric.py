"""GPU parity of the expert-centric comparison layer (wd_bench_expert_centric).

The comparison path of Cursor, "用 warp decode 实现更好的 MoE 模型推理",
section 传统的 MoE 路径 (The traditional MoE path): tokens gathered per expert
into padded expert-major buffers, grouped GEMVs, a per-expert output buffer in
BF16, and a weighted combine.  Its definition is the layer's, with each
expert's contribution rounded to BF16 in the per-expert buffer before the
combine; the expected values are assembled here from the oracle's own
functions: h = oracle.gate_up (one BF16 rounding), Y_k = oracle.down of slot k
alone with weight 1 (the BF16 per-expert output), out = bf16(sum_k w_k Y_k).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_decode_gate_gb300 as wd

from parity import compare, from_dev_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def expert_centric_expected(xs, ids, w, gu, gus, dn, dns, I, E):
    """out = bf16(sum_k w[b,k] * bf16(Wd[e_k] h[b,k])) from oracle functions."""
    B, K = ids.shape
    H = dn.shape[1]
    h = oracle.gate_up(xs, ids, gu, gus, I, E)
    y = np.zeros((B, H))
    ones = np.ones((B, 1), np.float32)
    for k in range(K):
        yk = oracle.down(np.ascontiguousarray(h[:, k:k + 1, :]), np.ascontiguousarray(ids[:, k:k + 1]),
                         ones, dn, dns, H, E)
        valid = ((ids[:, k] >= 0) & (ids[:, k] < E))[:, None]
        y += np.where(valid, w[:, k:k + 1].astype(np.float64) * oracle.bf16_bits_to_f64(yk), 0.0)
    return np.array([oracle.f64_to_bf16(float(v)) for v in y.ravel()], np.uint16).reshape(B, H)


def run_expert_centric(dev, xs, ids, w, gu, gus, dn, dns):
    B, K = ids.shape
    E, two_i, H = gu.shape
    ws = torch.empty(wd.wd_bench_expert_centric_workspace_size(B, H, two_i // 2, E, K),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    wd.wd_bench_expert_centric(to_dev_bf16(xs, dev), to_dev(ids, dev), to_dev(w, dev), to_dev(gu, dev),
                               to_dev(gus, dev), to_dev(dn, dev), to_dev(dns, dev), out, ws)
    torch.cuda.synchronize(dev)
    return from_dev_bf16(out)


def _case(seed, B, H, I, E, K, route="uniform"):
    wl = synth.Workload(f"ec{seed}", seed, H, I, E, K, (B,), route=route)
    gu, gus = synth.gate_up(seed, 0, E, H, I)
    dn, dns = synth.down(seed, 0, E, H, I)
    xs = synth.x(seed, 0, B, H)
    ids, w = synth.route(seed, 0, B, E, K, mode=route)
    return xs, ids, w, gu, gus, dn, dns


# the full-size layer at decode batches and under every routing pattern of the
# benchmark (fixed: 32 tokens on 8 experts, padded lists of 32; disjoint: no
# sharing), a batch above the decode range, ragged and tiny shapes, K == E
@pytest.mark.parametrize("B,H,I,E,K,route", [
    (1, 2048, 768, 128, 8, "uniform"),
    (4, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "uniform"),
    (32, 2048, 768, 128, 8, "zipf"),
    (32, 2048, 768, 128, 8, "fixed"),
    (32, 2048, 768, 128, 8, "disjoint"),
    (96, 1024, 256, 16, 4, "uniform"),
    (3, 288, 96, 5, 3, "uniform"),
    (5, 1056, 160, 7, 2, "uniform"),
    (1, 32, 32, 1, 1, "uniform"),
    (2, 128, 64, 3, 3, "uniform"),
    (2, 4096, 4096, 4, 2, "uniform"),
])
def test_expert_centric_layer_matches_its_definition(cuda_device, B, H, I, E, K, route):
    xs, ids, w, gu, gus, dn, dns = _case(500 + B + H + I + E, B, H, I, E, K, route)
    got = run_expert_centric(cuda_device, xs, ids, w, gu, gus, dn, dns)
    compare(got, expert_centric_expected(xs, ids, w, gu, gus, dn, dns, I, E),
            f"expert-centric B={B} H={H} I={I} {route}")


# The largest batch of the crossover sweep on the full-size layer: the GPU
# runs all 256 tokens, the definition is assembled for a seeded sample (each
# token's output depends only on its own row, ids and weights).
def test_expert_centric_crossover_batch_on_sampled_tokens(cuda_device):
    B, H, I, E, K = 256, 2048, 768, 128, 8
    xs, ids, w, gu, gus, dn, dns = _case(900, B, H, I, E, K)
    got = run_expert_centric(cuda_device, xs, ids, w, gu, gus, dn, dns)
    pick = np.sort(np.random.default_rng(B).choice(B, 8, replace=False))
    want = expert_centric_expected(np.ascontiguousarray(xs[pick]), np.ascontiguousarray(ids[pick]),
                                   np.ascontiguousarray(w[pick]), gu, gus, dn, dns, I, E)
    compare(got[pick], want, f"expert-centric B={B} sampled tokens {pick.tolist()}")


def test_expert_centric_skips_bad_ids(cuda_device):
    xs, ids, w, gu, gus, dn, dns = _case(41, 4, 256, 128, 8, 3)
    ids = ids.copy()
    ids[0, 1], ids[2, 0], ids[3, 2] = -1, 8, 1 << 30
    got = run_expert_centric(cuda_device, xs, ids, w, gu, gus, dn, dns)
    compare(got, expert_centric_expected(xs, ids, w, gu, gus, dn, dns, 128, 8), "expert-centric bad ids")


def test_expert_centric_is_close_to_warp_decode(cuda_device):
    """The two paths differ only by the per-expert BF16 rounding: on the
    full-size layer at B = 8 their outputs agree to the parity bar."""
    xs, ids, w, gu, gus, dn, dns = _case(42, 8, 2048, 768, 128, 8)
    got = run_expert_centric(cuda_device, xs, ids, w, gu, gus, dn, dns)
    compare(got, oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, 768, 128), "expert-centric vs warp decode")
