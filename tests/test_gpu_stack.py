"""GPU parity of the 48-layer decode stack, in the launch configuration bench.py
times: the stack's device-resident weights, one CUDA graph of all layers'
launches (at B=32: moe_gate_up_mma, moe_h_encode and moe_down_dimblock per
layer, each a programmatic dependent of the one before), the built-in launch
plan, B=32.

Tokens are independent through the stack (there is no attention), so the
oracle follows a few sampled tokens through every layer on its own, with only
their routed experts' weights generated, and the GPU's rows for those tokens
are compared with it.

Three checks:
  - chained: the GPU's own activations flow through the first layers (graphs
    of 1 and 3 layers), compared with the oracle's chain after layers 0, 1, 2;
  - per layer: layer l of the device-resident 48-layer stack run on the
    ORACLE's input of layer l, for l in 0..7, 16, 32, 47, compared with the
    oracle's output of layer l;
  - the full 48-layer chained graph output.
Chained comparisons stop at layer 2 because, with no norm between layers, a
layer is close to quadratic in its input once activations are small
(SiLU(g) ~ g/2), so relative rounding differences roughly double per layer;
the per-layer checks cover the deeper layers instead.  The activations shrink
to exactly zero within about eight layers, which both sides must reproduce.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import synth
import moe_decode_gate_gb300 as wd

from parity import compare, from_dev_bf16

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["qwen3_stack48"]
B = 32
SAMPLE = (0, 13, 31)


def oracle_chain(layers, tokens):
    """Oracle outputs of the sampled tokens after each of the first `layers` layers."""
    H, I, E, K = WL.H, WL.I, WL.E, WL.K
    x = synth.x(WL.seed, 0, B, H)[list(tokens)]
    outs = []
    for l in range(layers):
        ids, w = synth.route(WL.seed, l, B, E, K)
        ids, w = ids[list(tokens)], w[list(tokens)]
        gu = np.zeros((E, 2 * I, H), np.uint8)
        gus = np.zeros((E, 2 * I, H // 32), np.uint8)
        dn = np.zeros((E, H, I), np.uint8)
        dns = np.zeros((E, H, I // 32), np.uint8)
        for e in np.unique(ids):
            synth.gate_up(WL.seed, l, E, H, I, experts=(int(e), int(e) + 1), out=(gu, gus))
            synth.down(WL.seed, l, E, H, I, experts=(int(e), int(e) + 1), out=(dn, dns))
        x = oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E)
        outs.append(x.copy())
    return outs


def run_stack(dev, layers):
    stack = bench.Stack(torch, wd, dev, layers, B, lambda m: None)
    buf = stack.buffers(B)
    g, s = stack.graph(buf)
    g.replay()
    torch.cuda.synchronize(dev)
    return stack, buf


def test_stack_chained_first_layers(cuda_device):
    want = oracle_chain(3, SAMPLE)
    stack1, buf1 = run_stack(cuda_device, 1)
    compare(from_dev_bf16(buf1["act"][0])[list(SAMPLE)], want[0], "chained layer 0")
    del stack1, buf1
    stack3, buf3 = run_stack(cuda_device, 3)
    for l in (1, 2):
        got = from_dev_bf16(buf3["act"][l % 2])[list(SAMPLE)]
        compare(got, want[l], f"chained layer {l}")
    assert wd.wd_moe_read_error_flag(stack3.workspace) == 0


def test_stack_layers_on_oracle_inputs(cuda_device):
    """Layer l of the 48-layer stack on the oracle's input of layer l."""
    want = oracle_chain(WL.layers, SAMPLE)
    stack = bench.Stack(torch, wd, cuda_device, WL.layers, B, lambda m: None)
    buf = stack.buffers(B)
    x0 = synth.x(WL.seed, 0, B, WL.H)
    for l in (0, 1, 2, 3, 4, 5, 6, 7, 16, 32, 47):
        xin = x0.copy()
        if l > 0:
            xin[list(SAMPLE)] = want[l - 1]
        x_d = torch.from_numpy(xin.view(np.int16)).view(torch.bfloat16).to(cuda_device)
        out = torch.empty_like(x_d)
        gu, gus, dn, dns = stack.weights[l]
        wd.wd_moe_decode(x_d, buf["ids"][l], buf["w"][l], gu, gus, dn, dns, out, stack.workspace)
        torch.cuda.synchronize(cuda_device)
        compare(from_dev_bf16(out)[list(SAMPLE)], want[l], f"stack layer {l} on oracle input")
    assert wd.wd_moe_read_error_flag(stack.workspace) == 0


def test_full_48_layer_stack_output(cuda_device):
    want = oracle_chain(WL.layers, SAMPLE)
    stack, buf = run_stack(cuda_device, WL.layers)
    got = from_dev_bf16(buf["act"][(WL.layers - 1) % 2])[list(SAMPLE)]
    wv = oracle.bf16_bits_to_f64(want[-1])
    gv = oracle.bf16_bits_to_f64(got)
    if not np.any(wv):
        # the activations have collapsed to exactly zero, on both sides
        assert not np.any(gv), "GPU stack output should be exactly zero"
    else:
        compare(got, want[-1], "stack layer 47")
    assert wd.wd_moe_read_error_flag(stack.workspace) == 0
