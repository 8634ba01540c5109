"""Seeded synthetic inputs for the MoE decode layer.

The one module that both the CPU oracle and the CUDA path consume.  It holds
none of the layer's arithmetic: it draws activations, router outputs and FP32
expert weights from a counter-based generator (Philox4x32-10) and encodes the
weights to MXFP8 codes the way a checkpoint producer would.  The C source,
``wd_synth.c``, documents the exact recipe.

Workloads (Qwen-3-style shapes: 128 experts, top-8, hidden 2048, expert
intermediate 768; warp-decode blog (Cursor), section "传统的 MoE 路径"):

=====================  =====================================================
name                   description
=====================  =====================================================
``tiny``               B=1, H=256, I=128, E=16, K=4, uniform routing
``qwen3_b1``           B=1, H=2048, I=768, E=128, K=8, uniform routing
``qwen3_sweep``        same layer, B in {1,2,4,8,16,32}
``qwen3_zipf``         B=32, logits biased by a Zipf(1.2) prior over experts
``qwen3_fixed``        B=32, every token on experts {5,8,14,19,33,71,90,127}
``qwen3_disjoint``     B=32, disjoint 8-sets from two seeded permutations
``qwen3_stack48``      48 layers with their own weights, B in {1,8,32}
=====================  =====================================================
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wd_synth.c")
_SO = os.path.join(_HERE, "libwd_synth.so")
_LOCK = threading.Lock()
_LIB = None

ROUTE_MODES = {"uniform": 0, "zipf": 1, "fixed": 2, "disjoint": 3}
FIXED_EXPERTS = (5, 8, 14, 19, 33, 71, 90, 127)


def build(force: bool = False) -> str:
    """Compile ``libwd_synth.so`` next to its source (gcc, no GPU needed)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-ffp-contract=off", "-fno-math-errno", "-fno-semantic-interposition", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            u64, u32, i32 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
            lib.wd_synth_philox4x32_10.argtypes = [u64, P, P]
            lib.wd_synth_philox4x32_10.restype = None
            lib.wd_synth_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.wd_synth_f32_to_bf16.restype = ctypes.c_uint16
            lib.wd_synth_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.wd_synth_f32_to_e4m3.restype = ctypes.c_uint8
            lib.wd_synth_quantise_block.argtypes = [P, i32, P, P]
            lib.wd_synth_quantise_block.restype = None
            for fn in (lib.wd_synth_gate_up, lib.wd_synth_down):
                fn.argtypes = [u64, u32, i32, i32, i32, i32, P, P, P, i32]
                fn.restype = i32
            lib.wd_synth_x.argtypes = [u64, u32, i32, i32, P, P]
            lib.wd_synth_x.restype = i32
            lib.wd_synth_route.argtypes = [u64, u32, i32, i32, i32, i32, ctypes.c_double, P, P, P, P]
            lib.wd_synth_route.restype = i32
            _LIB = lib
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(n):
    return int(n) if n else max(1, os.cpu_count() or 1)


def philox4x32_10(seed: int, ctr) -> np.ndarray:
    """Raw Philox4x32-10 output (4 x uint32) for one 128-bit counter."""
    c = np.asarray(ctr, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _lib().wd_synth_philox4x32_10(seed, _ptr(c), _ptr(out))
    return out


def f32_to_e4m3(v) -> np.ndarray:
    """Element-wise FP32 -> E4M3 code (round to nearest even, saturating)."""
    v = np.asarray(v, dtype=np.float32).ravel()
    f = _lib().wd_synth_f32_to_e4m3
    return np.array([f(float(t)) for t in v], dtype=np.uint8)


def f32_to_bf16(v) -> np.ndarray:
    v = np.asarray(v, dtype=np.float32).ravel()
    f = _lib().wd_synth_f32_to_bf16
    return np.array([f(float(t)) for t in v], dtype=np.uint16)


def quantise_block(v):
    """(codes[32], scale_code) for one block of 32 FP32 values."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.zeros(v.size, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.uint8)
    _lib().wd_synth_quantise_block(_ptr(v), v.size, _ptr(codes), _ptr(scale))
    return codes, int(scale[0])


def gate_up(seed, layer, E, H, I, experts=None, raw=False, threads=None, out=None):
    """MXFP8 gate_up weights: codes uint8 [E, 2I, H], scales uint8 [E, 2I, H/32].

    Rows [0, I) of each expert are the gate projection, rows [I, 2I) the up
    projection.  ``experts`` = (e0, e1) generates only that expert range (the
    rest stays zero).  ``raw`` also returns the FP32 values before quantisation.
    """
    e0, e1 = experts if experts is not None else (0, E)
    codes, scales = out if out is not None else (np.zeros((E, 2 * I, H), np.uint8),
                                                 np.zeros((E, 2 * I, H // 32), np.uint8))
    r = np.zeros((E, 2 * I, H), np.float32) if raw else None
    rc = _lib().wd_synth_gate_up(seed, layer, e0, e1, H, I, _ptr(codes), _ptr(scales), _ptr(r),
                                 _threads(threads))
    if rc:
        raise ValueError("wd_synth_gate_up: bad shape")
    return (codes, scales, r) if raw else (codes, scales)


def down(seed, layer, E, H, I, experts=None, raw=False, threads=None, out=None):
    """MXFP8 down weights: codes uint8 [E, H, I], scales uint8 [E, H, I/32]."""
    e0, e1 = experts if experts is not None else (0, E)
    codes, scales = out if out is not None else (np.zeros((E, H, I), np.uint8),
                                                 np.zeros((E, H, I // 32), np.uint8))
    r = np.zeros((E, H, I), np.float32) if raw else None
    rc = _lib().wd_synth_down(seed, layer, e0, e1, H, I, _ptr(codes), _ptr(scales), _ptr(r),
                              _threads(threads))
    if rc:
        raise ValueError("wd_synth_down: bad shape")
    return (codes, scales, r) if raw else (codes, scales)


def x(seed, layer, B, H, raw=False):
    """Activations as BF16 bit patterns, uint16 [B, H] (N(0,1) rounded to BF16)."""
    out = np.zeros((B, H), np.uint16)
    r = np.zeros((B, H), np.float32) if raw else None
    _lib().wd_synth_x(seed, layer, B, H, _ptr(out), _ptr(r))
    return (out, r) if raw else out


def route(seed, layer, B, E, K, mode="uniform", zipf_s=1.2, fixed=FIXED_EXPERTS, logits=False):
    """Router outputs: topk_ids int32 [B, K], topk_w float32 [B, K]."""
    ids = np.zeros((B, K), np.int32)
    w = np.zeros((B, K), np.float32)
    fx = np.asarray(fixed if fixed is not None else [0] * K, np.int32)
    if mode == "fixed" and fx.size != K:
        raise ValueError("fixed routing needs exactly K ids")
    lg = np.zeros((B, E), np.float32) if logits else None
    rc = _lib().wd_synth_route(seed, layer, B, E, K, ROUTE_MODES[mode], zipf_s, _ptr(fx), _ptr(ids),
                               _ptr(w), _ptr(lg))
    if rc:
        raise ValueError(f"wd_synth_route: bad arguments (B={B}, E={E}, K={K}, mode={mode})")
    return (ids, w, lg) if logits else (ids, w)


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    H: int
    I: int
    E: int
    K: int
    batches: tuple
    route: str = "uniform"
    layers: int = 1
    note: str = ""


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 1234, 256, 128, 16, 4, (1,), note="tiny layer, B=1"),
        Workload("qwen3_b1", 1235, 2048, 768, 128, 8, (1,), note="Qwen-3-style layer, B=1"),
        Workload("qwen3_sweep", 1236, 2048, 768, 128, 8, (1, 2, 4, 8, 16, 32),
                 note="Qwen-3-style layer, batch sweep"),
        Workload("qwen3_zipf", 1237, 2048, 768, 128, 8, (32,), route="zipf",
                 note="B=32, Zipf(1.2) prior over experts"),
        Workload("qwen3_fixed", 1237, 2048, 768, 128, 8, (32,), route="fixed",
                 note="B=32, all tokens on experts {5,8,14,19,33,71,90,127}"),
        Workload("qwen3_disjoint", 1237, 2048, 768, 128, 8, (32,), route="disjoint",
                 note="B=32, disjoint expert sets from two seeded permutations"),
        Workload("qwen3_stack48", 1238, 2048, 768, 128, 8, (1, 8, 32), layers=48,
                 note="48 layers, own weights each, output of layer l feeds layer l+1"),
    )
}


@dataclass
class Layer:
    """One layer's inputs as host arrays (codes and bit patterns, not values)."""
    x: np.ndarray          # uint16 [B, H] (BF16 bits)
    ids: np.ndarray        # int32 [B, K]
    w: np.ndarray          # float32 [B, K]
    gate_up: np.ndarray    # uint8 [E, 2I, H]
    gate_up_scale: np.ndarray  # uint8 [E, 2I, H/32]
    down: np.ndarray       # uint8 [E, H, I]
    down_scale: np.ndarray     # uint8 [E, H, I/32]
    dims: dict = field(default_factory=dict)


def make_layer(wl: Workload, B: int, layer: int = 0, threads=None, weights=True) -> Layer:
    """Generate one layer of a workload at batch B."""
    H, I, E, K = wl.H, wl.I, wl.E, wl.K
    xs = x(wl.seed, layer, B, H)
    ids, w = route(wl.seed, layer, B, E, K, mode=wl.route)
    if weights:
        gu, gus = gate_up(wl.seed, layer, E, H, I, threads=threads)
        dn, dns = down(wl.seed, layer, E, H, I, threads=threads)
    else:
        gu = gus = dn = dns = None
    return Layer(xs, ids, w, gu, gus, dn, dns, dict(B=B, H=H, I=I, E=E, K=K))


def unique_expert_bytes(ids: np.ndarray, E: int, H: int, I: int) -> int:
    """Weight bytes touched by a routing: each distinct valid expert once (codes + scales)."""
    uniq = np.unique(ids[(ids >= 0) & (ids < E)])
    per_expert = 2 * I * H + 2 * I * (H // 32) + H * I + H * (I // 32)
    return int(uniq.size) * per_expert
