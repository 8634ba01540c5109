"""Accuracy of keeping activations in BF16 versus re-quantising them to MXFP8
between the stages of the layer, on the synthetic Qwen-3-style layer.

Cursor, "用 warp decode 实现更好的 MoE 模型推理", section 精度提升 (Accuracy
gains): the expert-centric path re-quantises activations to MXFP8 on the way
into each grouped GEMM, while warp decode keeps them in BF16 and accumulates
in FP32; the page reports the warp-decode output about 1.4x closer to an FP32
reference, without saying how the distance is measured.  This study measures
it here, with the plainest reading of each path (all in FP64 arithmetic so that
only the activation formats differ):

  reference    x (BF16 input) -> g, u exact -> h = silu(g) u exact -> y exact
  warp decode  ... h rounded once to BF16 ...                -> y   (this library's definition)
  traditional  x quantised to MXFP8 -> ... h quantised to MXFP8 -> y

MXFP8 quantisation of an activation vector follows the OCP Microscaling
Formats (MX) v1.0 conversion: per block of 32 consecutive elements the shared
scale is 2^(floor(log2(amax)) - 8) (8 = the exponent of E4M3's largest
normal), and each element is rounded to the nearest E4M3 value (ties to an even
mantissa) after dividing by the scale, saturating at +-448.  The distance is the
relative RMS error of y against the reference over all outputs of the batch.

Test infrastructure: the study reads the oracle (oracle/) and the generator
(synth/); gpu_column also runs this library's CUDA path on the same layer and
measures its own error against the same reference (the test in
tests/test_gpu_accuracy.py).  `python tests/accuracy_study.py [--gpu]` prints
the table quoted in the design notes.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

_E4M3_POS = None  # (values, codes) of the non-negative finite E4M3 codes, ascending


def _e4m3_positive():
    global _E4M3_POS
    if _E4M3_POS is None:
        codes = np.arange(0x7F, dtype=np.int64)  # 0x00 .. 0x7E (0x7F is NaN)
        vals = np.array([oracle.e4m3(int(c)) for c in codes])
        _E4M3_POS = (vals, codes)
    return _E4M3_POS


def round_to_e4m3(q: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value of each element (ties to the even mantissa), saturated at +-448."""
    vals, codes = _e4m3_positive()
    a = np.minimum(np.abs(q), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0) & (hi != lo))
    r = np.where(pick_hi, vals[hi], vals[lo])
    return np.copysign(r, q)


def quantize_mxfp8(v: np.ndarray) -> np.ndarray:
    """The values an activation tensor (last axis a multiple of 32) takes after
    MXFP8 quantisation with one E8M0 scale per 32 elements."""
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    amax = np.max(np.abs(blocks), axis=-1, keepdims=True)
    safe = np.where(amax > 0, amax, 1.0)
    scale = np.where(amax > 0, np.exp2(np.floor(np.log2(safe)) - 8), 1.0)
    return (round_to_e4m3(blocks / scale) * scale).reshape(v.shape)


def _dequant(codes, scales):
    vals = np.array([oracle.e4m3(c) for c in range(256)])
    sc = np.array([oracle.e8m0(c) for c in range(256)])
    r = vals[codes.astype(np.int64)]
    s = sc[scales.astype(np.int64)]
    return (r.reshape(r.shape[:-1] + (r.shape[-1] // 32, 32)) * s[..., None]).reshape(r.shape)


def _down_f64(h, ids, w, dn, dns, E):
    """y[b,d] = sum_k w[b,k] * Wd[e_k][d,:] . h[b,k,:] in FP64, h given as values."""
    B, K, I = h.shape
    H = dn.shape[1]
    y = np.zeros((B, H))
    for e in np.unique(ids):
        if not 0 <= e < E:
            continue
        wd = _dequant(dn[e], dns[e])  # [H, I]
        for b, k in zip(*np.nonzero(ids == e)):
            y[b] += float(w[b, k]) * (wd @ h[b, k])
    return y


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    return np.array([oracle.f64_to_bf16(float(t)) for t in v.ravel()], np.uint16).reshape(v.shape)


def layer_inputs(seed=1236, B=4, H=2048, I=768, E=128, K=8):
    """One seeded layer: x (BF16 bits), ids, w and the MXFP8 weights."""
    gu, gus = synth.gate_up(seed, 0, E, H, I)
    dn, dns = synth.down(seed, 0, E, H, I)
    x = synth.x(seed, 0, B, H)
    ids, w = synth.route(seed, 0, B, E, K)
    return x, ids, w, gu, gus, dn, dns


def reference_y(x, ids, w, gu, gus, dn, dns, I, E):
    """The unrounded reference output: FP64 throughout, h not rounded."""
    _, h_f64, _ = oracle.gate_up(x, ids, gu, gus, I, E, with_f64=True)
    return _down_f64(h_f64, ids, w, dn, dns, E)


def rel_rms(y, y_ref):
    """Relative RMS distance of y from y_ref over all outputs."""
    return float(np.sqrt(np.mean((y - y_ref) ** 2)) / np.sqrt(np.mean(y_ref ** 2)))


def study(seed=1236, B=4, H=2048, I=768, E=128, K=8):
    """Relative RMS error of y for the warp-decode and traditional activation
    formats against the unrounded reference, on one seeded layer."""
    x, ids, w, gu, gus, dn, dns = layer_inputs(seed, B, H, I, E, K)
    # reference and warp decode share the first projection
    h_bits, h_f64, _ = oracle.gate_up(x, ids, gu, gus, I, E, with_f64=True)
    y_ref = _down_f64(h_f64, ids, w, dn, dns, E)
    _, y_wd, _ = oracle.down(h_bits, ids, w, dn, dns, H, E, with_f64=True)
    # traditional: MXFP8 activations into both projections
    xq = quantize_mxfp8(oracle.bf16_bits_to_f64(x))
    _, hq_f64, _ = oracle.gate_up(_bf16_bits(xq), ids, gu, gus, I, E, with_f64=True)
    y_tr = _down_f64(quantize_mxfp8(hq_f64), ids, w, dn, dns, E)
    # each re-quantisation alone
    y_x_only = _down_f64(hq_f64, ids, w, dn, dns, E)
    y_h_only = _down_f64(quantize_mxfp8(h_f64), ids, w, dn, dns, E)

    def rel(y):
        return rel_rms(y, y_ref)

    e_wd, e_tr = rel(y_wd), rel(y_tr)
    return {"B": B, "rel_rms_warp_decode": e_wd, "rel_rms_traditional": e_tr,
            "ratio": e_tr / e_wd, "rel_rms_x_only": rel(y_x_only), "rel_rms_h_only": rel(y_h_only)}


def gpu_column(seed=1236, B=4, H=2048, I=768, E=128, K=8, device="cuda:0"):
    """This library's CUDA output (BF16, the built-in plan) on the same layer:
    its relative RMS error against the unrounded reference, next to the
    oracle's own output rounded to BF16 the same way (the error a perfect
    implementation of this path would show)."""
    import torch

    import moe_decode_gate_gb300 as wd

    x, ids, w, gu, gus, dn, dns = layer_inputs(seed, B, H, I, E, K)
    y_ref = reference_y(x, ids, w, gu, gus, dn, dns, I, E)
    dev = torch.device(device)
    layer = wd.MoEDecodeLayer(gu, gus, dn, dns, K=K, max_batch=B, device=dev)
    out = layer(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev),
                torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev))
    torch.cuda.synchronize(dev)
    y_gpu = out.float().cpu().double().numpy()
    y_oracle = oracle.bf16_bits_to_f64(oracle.moe_decode(x, ids, w, gu, gus, dn, dns, I, E))
    return {"B": B, "rel_rms_gpu": rel_rms(y_gpu, y_ref), "rel_rms_oracle_bf16": rel_rms(y_oracle, y_ref),
            "plan": wd.wd_moe_describe_plan(B, H, I, E, K)}


if __name__ == "__main__":
    gpu = "--gpu" in sys.argv
    print("| B | BF16 h (this path, FP64) | MXFP8 x and h | ratio | MXFP8 x only | MXFP8 h only |"
          + (" CUDA path (BF16 out) | oracle, BF16 out |" if gpu else ""))
    print("|---|---|---|---|---|---|" + ("---|---|" if gpu else ""))
    for B in (1, 4, 8, 32):
        r = study(B=B)
        line = (f"| {B} | {r['rel_rms_warp_decode']:.3e} | {r['rel_rms_traditional']:.3e} "
                f"| {r['ratio']:.1f} | {r['rel_rms_x_only']:.3e} | {r['rel_rms_h_only']:.3e} |")
        if gpu:
            g = gpu_column(B=B)
            line += f" {g['rel_rms_gpu']:.3e} | {g['rel_rms_oracle_bf16']:.3e} |"
        print(line, flush=True)
