"""wd_moe_decode_no_alloc: the layer for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns all device memory and forbids
allocation while it runs, or a latency-critical loop that cannot pay for
cudaMalloc's possible implicit synchronisation) cannot hand the library a
workspace.  This entry point keeps the layer's scratch in a 2 MiB array
compiled into the library instead.  The test drives it through the C-ABI on
two calls in a row (different batches and plans, so the second call must not
see anything the first one left in the shared array) and checks each against
the CPU oracle with the parity tolerance of the other GPU tests, and against
wd_moe_decode bit for bit: both run the same kernels in the same order.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import moe_decode_gate_gb300 as wd

from parity import compare, from_dev_bf16, to_dev, to_dev_bf16

WD_OK, WD_ERR_WORKSPACE_TOO_SMALL = 0, 3
A32 = 0x10000  # fake 32-byte-aligned address: the size check rejects before any use


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_no_alloc_rejects_batches_beyond_its_scratch_on_the_host():
    # the workspace layout must fit in 2 MiB: B=85 fits at K=8, I=768; B=86 does not
    lib = wd.lib()
    assert lib.wd_moe_decode_no_alloc(A32, A32, A32, A32, A32, A32, A32, A32,
                                      86, 2048, 768, 128, 8, None) == WD_ERR_WORKSPACE_TOO_SMALL
    assert lib.wd_moe_decode_no_alloc(A32, A32, A32, A32, A32, A32, A32, A32,
                                      1, 2048, 16384, 128, 64, None) == WD_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.gpu
def test_no_alloc_matches_wd_moe_decode_on_two_calls_in_a_row(cuda_device):
    dev = cuda_device
    lib = wd.lib()
    wl = synth.WORKLOADS["qwen3_sweep"]
    H, I, E, K = wl.H, wl.I, wl.E, wl.K
    gu, gus = synth.gate_up(wl.seed, 0, E, H, I)
    dn, dns = synth.down(wl.seed, 0, E, H, I)
    gu_d, gus_d, dn_d, dns_d = (to_dev(a, dev) for a in (gu, gus, dn, dns))
    workspace = torch.empty(wd.wd_moe_workspace_size(32, K, I), dtype=torch.uint8, device=dev)
    wd.wd_moe_workspace_init(workspace)
    stream = torch.cuda.current_stream(dev)

    # B=32 runs the shared-row kernels (three launches), B=5 the per-token ones
    for call, (B, layer) in enumerate(((32, 0), (5, 1))):
        xs = synth.x(wl.seed, layer, B, H)
        ids, w = synth.route(wl.seed, layer, B, E, K)
        x_d, ids_d, w_d = to_dev_bf16(xs, dev), to_dev(ids, dev), to_dev(w, dev)
        ref = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
        wd.wd_moe_decode(x_d, ids_d, w_d, gu_d, gus_d, dn_d, dns_d, ref, workspace)
        out = torch.full((B, H), float("nan"), dtype=torch.bfloat16, device=dev)
        st = lib.wd_moe_decode_no_alloc(_ptr(x_d), _ptr(ids_d), _ptr(w_d), _ptr(gu_d), _ptr(gus_d),
                                        _ptr(dn_d), _ptr(dns_d), _ptr(out), B, H, I, E, K,
                                        ctypes.c_void_p(stream.cuda_stream))
        assert st == WD_OK, wd.wd_status_string(st)
        torch.cuda.synchronize(dev)
        got, want = from_dev_bf16(out), from_dev_bf16(ref)
        expect = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, I, E)
        compare(got, expect, f"no-alloc call {call + 1} (B={B}) vs the oracle")
        assert np.array_equal(got, want), f"call {call + 1}: differs from wd_moe_decode"
