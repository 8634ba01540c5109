"""CPU oracle for the MoE decode layer (TEST INFRASTRUCTURE).

Plain FP64 C loops (``wd_oracle.c``) behind ctypes.  The tests, the smoke check
and the benchmark's CPU-baseline leg are the only callers; the library and its
Python binding never import this package, and it imports nothing from them.
It builds its own shared object with gcc (FMA contraction off, so the FP64
arithmetic is the same on every host).

Every function is pinned by tests that do not re-run the oracle's own formula:
see ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wd_oracle.c")
_SO = os.path.join(_HERE, "libwd_oracle.so")
_LOCK = threading.Lock()
_LIB = None


def build(force: bool = False) -> str:
    """Compile ``libwd_oracle.so`` next to its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            P, i32 = ctypes.c_void_p, ctypes.c_int
            lib.oracle_e4m3.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3.restype = ctypes.c_double
            lib.oracle_e8m0.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_gate_up.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_gate_up.restype = ctypes.c_long
            lib.oracle_down.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_down.restype = ctypes.c_long
            lib.oracle_moe_decode.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, P, P, P]
            lib.oracle_moe_decode.restype = ctypes.c_long
            _LIB = lib
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def e4m3(code: int) -> float:
    return _lib().oracle_e4m3(int(code))


def e8m0(code: int) -> float:
    return _lib().oracle_e8m0(int(code))


def bf16_to_f64(bits: int) -> float:
    return _lib().oracle_bf16_to_f64(int(bits))


def f64_to_bf16(v: float) -> int:
    return int(_lib().oracle_f64_to_bf16(float(v)))


def silu(g: float) -> float:
    return _lib().oracle_silu(float(g))


def gate_up(x, ids, gate_up_codes, gate_up_scale, I, E, with_f64=False):
    """h [B,K,I] as BF16 bits (and the FP64 values before rounding)."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    B, H = x.shape
    K = ids.shape[1]
    gu, gus = _c(gate_up_codes, np.uint8), _c(gate_up_scale, np.uint8)
    assert gu.shape == (E, 2 * I, H) and gus.shape == (E, 2 * I, H // 32)
    h = np.zeros((B, K, I), np.uint16)
    hf = np.zeros((B, K, I), np.float64) if with_f64 else None
    bad = _lib().oracle_gate_up(_p(x), _p(ids), _p(gu), _p(gus), B, H, I, E, K, _p(h), _p(hf))
    return (h, hf, bad) if with_f64 else h


def down(h, ids, w, down_codes, down_scale, H, E, with_f64=False):
    """out [B,H] as BF16 bits (and y [B,H] in FP64 before rounding)."""
    h = _c(h, np.uint16)
    ids, w = _c(ids, np.int32), _c(w, np.float32)
    B, K, I = h.shape
    dn, dns = _c(down_codes, np.uint8), _c(down_scale, np.uint8)
    assert dn.shape == (E, H, I) and dns.shape == (E, H, I // 32)
    out = np.zeros((B, H), np.uint16)
    y = np.zeros((B, H), np.float64) if with_f64 else None
    bad = _lib().oracle_down(_p(h), _p(ids), _p(w), _p(dn), _p(dns), B, H, I, E, K, _p(out), _p(y))
    return (out, y, bad) if with_f64 else out


def moe_decode(x, ids, w, gate_up_codes, gate_up_scale, down_codes, down_scale, I, E,
               with_f64=False):
    """The whole layer: out [B,H] BF16 bits; with_f64 adds (h bits, y FP64, bad-id count)."""
    x = _c(x, np.uint16)
    ids, w = _c(ids, np.int32), _c(w, np.float32)
    B, H = x.shape
    K = ids.shape[1]
    gu, gus = _c(gate_up_codes, np.uint8), _c(gate_up_scale, np.uint8)
    dn, dns = _c(down_codes, np.uint8), _c(down_scale, np.uint8)
    assert gu.shape == (E, 2 * I, H) and gus.shape == (E, 2 * I, H // 32)
    assert dn.shape == (E, H, I) and dns.shape == (E, H, I // 32)
    h = np.zeros((B, K, I), np.uint16)
    out = np.zeros((B, H), np.uint16)
    y = np.zeros((B, H), np.float64) if with_f64 else None
    bad = _lib().oracle_moe_decode(_p(x), _p(ids), _p(w), _p(gu), _p(gus), _p(dn), _p(dns),
                                   B, H, I, E, K, _p(h), _p(out), _p(y))
    return (out, h, y, bad) if with_f64 else out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Vectorised BF16 bits -> values (for comparisons in tests)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
