"""ctypes binding of the C-ABI in include/wd_moe.h and include/wd_bench.h.

Argument marshalling only: shapes are read off the tensors, pointers and the
current CUDA stream are passed through, and a non-OK status raises WdError.
Every step of the layer runs in the library's CUDA kernels; there is no
fallback path.  If the library cannot be loaded the import of this module
fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

WD_OK = 0
STATUS_NAMES = {0: "WD_OK", 1: "WD_ERR_INVALID_ARG", 2: "WD_ERR_UNSUPPORTED_SHAPE",
                3: "WD_ERR_WORKSPACE_TOO_SMALL", 4: "WD_ERR_CUDA", 5: "WD_ERR_BAD_EXPERT_ID",
                6: "WD_ERR_PIPELINE_TIMEOUT"}
# bits of the workspace error flag (wd_moe_read_error_flag)
FLAG_BAD_EXPERT_ID = 1
FLAG_PIPELINE_TIMEOUT = 2

# (name, restype, argtypes) for every symbol the headers declare
_P, _I, _SZ, _U32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint32
SIGNATURES = {
    "wd_status_string": (ctypes.c_char_p, [_I]),
    "wd_moe_workspace_size": (_SZ, [_I, _I, _I]),
    "wd_moe_workspace_init": (_I, [_P, _SZ, _P]),
    "wd_moe_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _P]),
    "wd_moe_gate_up": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "wd_moe_down": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "wd_moe_down_workspace": (_I, [_P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _P]),
    "wd_moe_launches": (_I, [_I, _I, _I, _I, _I]),
    "wd_moe_h_encode": (_I, [_P, _P, _P, _I, _I, _P]),
    "wd_moe_down_encoded": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "wd_moe_read_error_flag": (_I, [_P, _SZ, _P, ctypes.POINTER(_I)]),
    "wd_moe_launches_per_call": (_I, []),
    "wd_moe_decode_no_alloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "wd_moe_set_plan": (_I, [ctypes.c_char_p]),
    "wd_last_error_string": (ctypes.c_char_p, []),
    "wd_moe_describe_plan": (_I, [ctypes.c_int] * 5 + [ctypes.c_char_p, ctypes.c_size_t]),
    "wd_bench_copy": (_I, [_P, _P, _SZ, _I, _P]),
    "wd_bench_read": (_I, [_P, _SZ, _P, _I, _P]),
    "wd_bench_fill": (_I, [_P, _SZ, _U32, _I, _P]),
    "wd_bench_hold": (_I, [_U32, _P]),
    "wd_bench_expert_centric_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "wd_bench_expert_centric": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I,
                                     _P]),
    "wd_bench_sm_count": (_I, []),
    "wd_bench_spec_gbs": (ctypes.c_double, []),
}


class WdError(RuntimeError):
    def __init__(self, fn, status, detail=None):
        self.status = status
        extra = f" ({detail})" if detail else ""
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}{extra}")


def library_path() -> str:
    return _build.OUT


def lib() -> ctypes.CDLL:
    """Load libwd_moe.so (compiling it first if a source is newer)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.build() if _build.stale() else _build.OUT
            if not os.path.exists(path):
                raise RuntimeError(f"native library missing: {path}")
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = handle
    return _LIB


def _check(fn, status):
    if status != WD_OK:
        detail = None
        if STATUS_NAMES.get(status) == "WD_ERR_CUDA":
            detail = lib().wd_last_error_string().decode()
        raise WdError(fn, status, detail)


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dims(x, topk_ids, gate_up):
    B, H = x.shape
    K = topk_ids.shape[1]
    E, I2, H2 = gate_up.shape
    if H2 != H or topk_ids.shape[0] != B or I2 % 2:
        raise ValueError("inconsistent shapes")
    return B, H, I2 // 2, E, K


# --------------------------------------------------------------- wd_moe.h ---

def wd_status_string(status: int) -> str:
    return lib().wd_status_string(status).decode()


def wd_moe_workspace_size(B: int, K: int, I: int) -> int:
    return int(lib().wd_moe_workspace_size(B, K, I))


def wd_moe_workspace_init(workspace, stream=None):
    _check("wd_moe_workspace_init",
           lib().wd_moe_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))


def wd_moe_decode(x, topk_ids, topk_w, gate_up, gate_up_scale, down, down_scale, out, workspace,
                  stream=None):
    """out[B,H] (bf16) = the MoE decode layer; see include/wd_moe.h."""
    B, H, I, E, K = _dims(x, topk_ids, gate_up)
    _check("wd_moe_decode", lib().wd_moe_decode(
        _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(gate_up), _ptr(gate_up_scale), _ptr(down),
        _ptr(down_scale), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        B, H, I, E, K, _stream(stream)))


def wd_moe_gate_up(x, topk_ids, gate_up, gate_up_scale, h, error_flag=None, stream=None):
    """h[B,K,I] (bf16) from the first kernel alone."""
    B, H, I, E, K = _dims(x, topk_ids, gate_up)
    _check("wd_moe_gate_up", lib().wd_moe_gate_up(
        _ptr(x), _ptr(topk_ids), _ptr(gate_up), _ptr(gate_up_scale), _ptr(h), _ptr(error_flag),
        B, H, I, E, K, _stream(stream)))


def wd_moe_down(h, topk_ids, topk_w, down, down_scale, out, error_flag=None, stream=None):
    """out[B,H] (bf16) from the second kernel alone, given h[B,K,I]."""
    B, K, I = h.shape
    E, H, I2 = down.shape
    if I2 != I or topk_ids.shape != (B, K):
        raise ValueError("inconsistent shapes")
    _check("wd_moe_down", lib().wd_moe_down(
        _ptr(h), _ptr(topk_ids), _ptr(topk_w), _ptr(down), _ptr(down_scale), _ptr(out),
        _ptr(error_flag), B, H, I, E, K, _stream(stream)))


def wd_moe_down_workspace(h, topk_ids, topk_w, down, down_scale, out, workspace, stream=None):
    """out[B,H] (bf16) from the down stage alone with a workspace (the plan's
    down kernels, as wd_moe_decode runs them), given h[B,K,I]."""
    B, K, I = h.shape
    E, H, I2 = down.shape
    if I2 != I or topk_ids.shape != (B, K):
        raise ValueError("inconsistent shapes")
    _check("wd_moe_down_workspace", lib().wd_moe_down_workspace(
        _ptr(h), _ptr(topk_ids), _ptr(topk_w), _ptr(down), _ptr(down_scale), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, I, E, K,
        _stream(stream)))


def wd_moe_h_encode(h, h16, hk, stream=None):
    """h16 (fp16, h's shape) and hk (int32 per row) from h [..., I] (bf16)."""
    I = h.shape[-1]
    rows = h.numel() // I
    _check("wd_moe_h_encode", lib().wd_moe_h_encode(_ptr(h), _ptr(h16), _ptr(hk), rows, I,
                                                    _stream(stream)))


def wd_moe_down_encoded(h16, hk, topk_ids, topk_w, down, down_scale, out, error_flag=None,
                        stream=None):
    """out[B,H] (bf16) from moe_down_dimblock alone, given moe_h_encode's output."""
    B, K, I = h16.shape
    E, H, I2 = down.shape
    if I2 != I or topk_ids.shape != (B, K):
        raise ValueError("inconsistent shapes")
    _check("wd_moe_down_encoded", lib().wd_moe_down_encoded(
        _ptr(h16), _ptr(hk), _ptr(topk_ids), _ptr(topk_w), _ptr(down), _ptr(down_scale), _ptr(out),
        _ptr(error_flag), B, H, I, E, K, _stream(stream)))


def wd_moe_read_error_flag(workspace, stream=None, with_status=False):
    """The error-flag bit mask accumulated since the last read, then cleared
    (synchronises): bit 0 (FLAG_BAD_EXPERT_ID) an out-of-range expert id was
    skipped; bit 1 (FLAG_PIPELINE_TIMEOUT) a kernel's bounded wait ran out and
    that call's output is invalid.  With ``with_status`` also the C status."""
    flag = ctypes.c_int(0)
    st = lib().wd_moe_read_error_flag(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream), ctypes.byref(flag))
    if st not in (WD_OK, 5, 6):
        raise WdError("wd_moe_read_error_flag", st)
    return (flag.value, st) if with_status else flag.value


def wd_moe_launches_per_call() -> int:
    """The most kernel launches one wd_moe_decode call issues."""
    return int(lib().wd_moe_launches_per_call())


def wd_moe_launches(B, H, I, E, K) -> int:
    """Kernel launches wd_moe_decode issues for this shape under the current plan."""
    return int(lib().wd_moe_launches(B, H, I, E, K))


def wd_moe_set_plan(spec=None):
    """Override the launch plan (see include/wd_moe.h); None restores the default."""
    _check("wd_moe_set_plan", lib().wd_moe_set_plan(None if spec is None else spec.encode()))


def wd_last_error_string() -> str:
    """Name of the CUDA error behind this thread's last WD_ERR_CUDA ("none" if none)."""
    return lib().wd_last_error_string().decode()


def wd_moe_describe_plan(B, H, I, E, K) -> str:
    """The kernels wd_moe_decode would launch for this shape, e.g.
    "gate_up=moe_gate_up_persist<2,1> down=moe_down_3d_batched<4,1>"."""
    buf = ctypes.create_string_buffer(256)
    _check("wd_moe_describe_plan", lib().wd_moe_describe_plan(B, H, I, E, K, buf, 256))
    return buf.value.decode()


def wd_moe_decode_no_alloc(x, topk_ids, topk_w, gate_up, gate_up_scale, down, down_scale, out,
                           stream=None):
    """The layer without a workspace, for callers that cannot allocate device
    memory: its scratch lives in a 2 MiB array inside the library
    (wd_moe_workspace_size(B, K, I) <= 2 MiB, i.e. B <= 85 at K=8, I=768).
    Calls that may overlap on the GPU share that array and must not be issued."""
    B, H, I, E, K = _dims(x, topk_ids, gate_up)
    _check("wd_moe_decode_no_alloc", lib().wd_moe_decode_no_alloc(
        _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(gate_up), _ptr(gate_up_scale), _ptr(down),
        _ptr(down_scale), _ptr(out), B, H, I, E, K, _stream(stream)))


# ------------------------------------------------------------- wd_bench.h ---

def wd_bench_copy(dst, src, nbytes=None, blocks=0, stream=None):
    n = nbytes if nbytes is not None else src.numel() * src.element_size()
    _check("wd_bench_copy", lib().wd_bench_copy(_ptr(dst), _ptr(src), n, blocks, _stream(stream)))


def wd_bench_read(src, sink, nbytes=None, blocks=0, stream=None):
    n = nbytes if nbytes is not None else src.numel() * src.element_size()
    _check("wd_bench_read", lib().wd_bench_read(_ptr(src), n, _ptr(sink), blocks, _stream(stream)))


def wd_bench_fill(buf, value=0, nbytes=None, blocks=0, stream=None):
    n = nbytes if nbytes is not None else buf.numel() * buf.element_size()
    _check("wd_bench_fill", lib().wd_bench_fill(_ptr(buf), n, value, blocks, _stream(stream)))


def wd_bench_hold(microseconds, stream=None):
    """Occupy `stream` for `microseconds` of device time (one thread)."""
    _check("wd_bench_hold", lib().wd_bench_hold(int(microseconds), _stream(stream)))


def wd_bench_expert_centric_workspace_size(B, H, I, E, K) -> int:
    return int(lib().wd_bench_expert_centric_workspace_size(B, H, I, E, K))


def wd_bench_expert_centric(x, topk_ids, topk_w, gate_up, gate_up_scale, down, down_scale, out,
                            workspace, stream=None):
    """The expert-centric comparison layer (include/wd_bench.h); shapes as wd_moe_decode."""
    B, H = x.shape
    E, two_i, _ = gate_up.shape
    K = topk_ids.shape[1]
    _check("wd_bench_expert_centric", lib().wd_bench_expert_centric(
        _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(gate_up), _ptr(gate_up_scale), _ptr(down),
        _ptr(down_scale), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        B, H, two_i // 2, E, K, _stream(stream)))


def wd_bench_sm_count() -> int:
    return int(lib().wd_bench_sm_count())


def wd_bench_spec_gbs() -> float:
    return float(lib().wd_bench_spec_gbs())
