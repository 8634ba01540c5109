"""Helpers for GPU-vs-oracle parity tests.

Tolerance (the layer's accuracy contract): for every token, cosine similarity
between the GPU and oracle output rows >= 0.99999, and
max |gpu - oracle| <= 1e-2 * max |oracle| + 2e-3 over the compared values.
The GPU accumulates in FP32 in a different order than the FP64 oracle and
both round h and out to BF16, so isolated 1-ulp BF16 differences are expected;
the bound admits those and nothing systematic.
"""
import numpy as np
import torch

COS_MIN = 0.99999
REL_TOL = 1e-2
ABS_TOL = 2e-3


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def to_dev_bf16(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def from_dev_bf16(t):
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def compare(got_bits, want_bits, what=""):
    """Assert the parity bar row by row (rows = tokens or (token, slot) pairs)."""
    got = bf16_bits_to_f64(got_bits).reshape(-1, np.asarray(got_bits).shape[-1])
    want = bf16_bits_to_f64(want_bits).reshape(got.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU values"
    err = np.abs(got - want).max()
    tol = REL_TOL * np.abs(want).max() + ABS_TOL
    assert err <= tol, f"{what}: max |gpu - oracle| = {err:.4g} > {tol:.4g}"
    for r in range(got.shape[0]):
        ng, nw = np.linalg.norm(got[r]), np.linalg.norm(want[r])
        if nw == 0.0:
            assert ng == 0.0, f"{what}: row {r} should be zero"
            continue
        cos = float(got[r] @ want[r] / (ng * nw))
        assert cos >= COS_MIN, f"{what}: row {r} cosine {cos:.7f} < {COS_MIN}"
    return dict(max_err=float(err), tol=float(tol),
                frac_equal=float(np.mean(np.asarray(got_bits) == np.asarray(want_bits))))
