"""The C-ABI library without a GPU: it loads, exports every symbol the headers
declare, and rejects bad arguments on the host before any launch.

Every call below fails host validation, so nothing reaches the GPU even on a
machine that has one.
"""
import ctypes
import os
import re

import pytest

import moe_decode_gate_gb300 as wd
from moe_decode_gate_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in ("wd_moe.h", "wd_bench.h")]

OK, INVALID, SHAPE, SMALL, CUDA, BADID, TIMEOUT = 0, 1, 2, 3, 4, 5, 6


def declared_symbols():
    names = []
    for h in HEADERS:
        text = open(h).read()
        names += re.findall(r"^WD_API\s+[\w\s\*]+?\b(wd_\w+)\s*\(", text, flags=re.M)
    return names


def test_headers_declare_the_expected_entry_points():
    names = set(declared_symbols())
    for n in ("wd_moe_decode", "wd_moe_gate_up", "wd_moe_down", "wd_moe_down_workspace",
              "wd_moe_workspace_size", "wd_moe_workspace_init", "wd_moe_read_error_flag",
              "wd_status_string", "wd_moe_launches", "wd_bench_copy", "wd_bench_read",
              "wd_bench_fill", "wd_bench_hold"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = wd.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, name  # and the binding knows its signature


def test_library_was_built_for_sm_103a_only():
    from moe_decode_gate_gb300 import build

    assert "arch=compute_103a,code=sm_103a" in build.ARCH
    assert os.path.exists(wd.library_path())


def test_status_strings():
    for code, name in _native.STATUS_NAMES.items():
        assert wd.wd_status_string(code) == name
    assert wd.wd_status_string(TIMEOUT) == "WD_ERR_PIPELINE_TIMEOUT"
    assert wd.wd_status_string(99) == "WD_ERR_UNKNOWN"


def test_workspace_size():
    # 256-byte flag slot + bf16 h [B, K, I] + its FP16 re-encoding [B, K, I] +
    # int32 exponents [B, K], each rounded up to 256 bytes
    assert wd.wd_moe_workspace_size(1, 8, 768) == 256 + 2 * 12288 + 256
    assert wd.wd_moe_workspace_size(32, 8, 768) == 256 + 2 * 32 * 8 * 768 * 2 + 1024
    assert wd.wd_moe_workspace_size(1, 1, 32) == 256 + 256 + 256 + 256
    assert wd.wd_moe_workspace_size(0, 8, 768) == 0
    assert wd.wd_moe_workspace_size(1, -1, 768) == 0


A32 = 0x10000  # a 32-byte-aligned fake address: never dereferenced (validation fails first)


def _decode(x=A32, ids=A32, w=A32, gu=A32, gus=A32, dn=A32, dns=A32, out=A32, ws=A32,
            ws_bytes=1 << 20, B=1, H=2048, I=768, E=128, K=8):
    return wd.lib().wd_moe_decode(x, ids, w, gu, gus, dn, dns, out, ws, ws_bytes,
                                  B, H, I, E, K, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), INVALID), (dict(ids=None), INVALID), (dict(w=None), INVALID),
    (dict(gu=None), INVALID), (dict(gus=None), INVALID), (dict(dn=None), INVALID),
    (dict(dns=None), INVALID), (dict(out=None), INVALID), (dict(ws=None), INVALID),
    (dict(B=0), INVALID), (dict(B=4097), INVALID), (dict(K=0), INVALID), (dict(K=65, E=128), INVALID),
    (dict(K=9, E=8), INVALID), (dict(E=0), INVALID),
    (dict(H=2047), SHAPE), (dict(H=2064), SHAPE), (dict(I=770), SHAPE), (dict(I=16), SHAPE),
    (dict(H=16416), SHAPE),
    (dict(x=A32 + 16), INVALID), (dict(gu=A32 + 16), INVALID), (dict(dn=A32 + 8), INVALID),
    (dict(ids=A32 + 2), INVALID), (dict(w=A32 + 1), INVALID), (dict(out=A32 + 2), INVALID),
    (dict(ws=A32 + 128), INVALID),
    (dict(ws_bytes=256 + 2 * 12288 + 255), SMALL), (dict(ws_bytes=0), SMALL),
])
def test_decode_rejects_bad_arguments_on_the_host(kw, status):
    assert _decode(**kw) == status


def test_split_kernels_reject_bad_arguments():
    lib = wd.lib()
    # gate_up: null h, misaligned x, bad shape
    assert lib.wd_moe_gate_up(A32, A32, A32, A32, None, None, 1, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_gate_up(A32 + 4, A32, A32, A32, A32, None, 1, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_gate_up(A32, A32, A32, A32, A32, None, 1, 2000, 768, 128, 8, None) == SHAPE
    assert lib.wd_moe_gate_up(A32, A32, A32, A32, A32, A32 + 1, 1, 2048, 768, 128, 8, None) == INVALID
    # down: h must be 32-byte aligned
    assert lib.wd_moe_down(A32 + 16, A32, A32, A32, A32, A32, None, 1, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_down(A32, A32, None, A32, A32, A32, None, 1, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_down(A32, A32, A32, A32, A32, A32, None, 1, 2048, 100, 128, 8, None) == SHAPE
    # down with a workspace: aligned h and workspace, and a large enough workspace
    ws = wd.wd_moe_workspace_size(32, 8, 768)
    assert lib.wd_moe_down_workspace(A32 + 16, A32, A32, A32, A32, A32, A32, ws,
                                     32, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_down_workspace(A32, A32, A32, A32, A32, A32, A32 + 64, ws,
                                     32, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_down_workspace(A32, A32, A32, A32, A32, A32, None, ws,
                                     32, 2048, 768, 128, 8, None) == INVALID
    assert lib.wd_moe_down_workspace(A32, A32, A32, A32, A32, A32, A32, ws - 1,
                                     32, 2048, 768, 128, 8, None) == SMALL


def test_workspace_calls_reject_bad_arguments():
    lib = wd.lib()
    flag = ctypes.c_int(7)
    assert lib.wd_moe_workspace_init(None, 1 << 20, None) == INVALID
    assert lib.wd_moe_workspace_init(A32 + 32, 1 << 20, None) == INVALID
    assert lib.wd_moe_workspace_init(A32, 16, None) == SMALL
    assert lib.wd_moe_read_error_flag(A32, 1 << 20, None, None) == INVALID
    assert lib.wd_moe_read_error_flag(A32 + 64, 1 << 20, None, ctypes.byref(flag)) == INVALID
    assert lib.wd_moe_read_error_flag(A32, 8, None, ctypes.byref(flag)) == SMALL
    assert flag.value == 7  # untouched on error


def test_bench_kernels_reject_unaligned_buffers():
    lib = wd.lib()
    einval = 1  # cudaErrorInvalidValue
    assert lib.wd_bench_copy(A32, A32 + 16, 1024, 0, None) == einval
    assert lib.wd_bench_copy(A32, A32, 1000, 0, None) == einval
    assert lib.wd_bench_read(A32, 1024, None, 0, None) == einval
    assert lib.wd_bench_fill(None, 1024, 0, 0, None) == einval
    assert lib.wd_bench_hold(1000001, None) == einval  # longer than a second


def test_expert_centric_arguments_and_workspace():
    lib = wd.lib()
    size = wd.wd_bench_expert_centric_workspace_size
    assert size(32, 2048, 768, 128, 8) > 2 * (2 * 32 * 8) * (2048 + 768 + 2048)  # three buffers
    assert size(64, 2048, 768, 128, 8) > size(32, 2048, 768, 128, 8)
    assert size(0, 2048, 768, 128, 8) == 0 and size(1, 2048, 768, 8192, 8) == 0
    assert size(1, 8192, 768, 128, 8) == 0  # H above 4096
    einval = 1
    n = size(2, 256, 128, 8, 2)
    assert lib.wd_bench_expert_centric(None, None, None, None, None, None, None, None, None, n,
                                       2, 256, 128, 8, 2, None) == einval
    assert lib.wd_bench_expert_centric(A32, A32, A32, A32, A32, A32, A32, A32, A32, n - 1,
                                       2, 256, 128, 8, 2, None) == einval  # workspace too small
    assert lib.wd_bench_expert_centric(A32, A32, A32, A32, A32, A32, A32, A32, A32 + 16, n,
                                       2, 256, 128, 8, 2, None) == einval  # misaligned workspace


def test_last_error_string_starts_empty():
    assert wd.wd_last_error_string() == "none"


def test_launch_count():
    assert wd.wd_moe_launches_per_call() == 3
    wd.wd_moe_set_plan(None)
    q = dict(H=2048, I=768, E=128, K=8)
    assert [wd.wd_moe_launches(B, **q) for B in (1, 2, 4, 8, 16, 32, 64)] == [2, 2, 2, 2, 3, 3, 2]
    assert wd.wd_moe_launches(0, **q) == 0


def test_built_in_plan_by_batch():
    """The kernels the built-in plan picks on the Qwen-3-style shape (host only)."""
    wd.wd_moe_set_plan(None)
    q = dict(H=2048, I=768, E=128, K=8)
    assert wd.wd_moe_describe_plan(1, **q) == \
        "gate_up=moe_gate_up_3d_batched<1,1> down=moe_down_3d_batched<1,6> pdl=3 launches=2"
    assert wd.wd_moe_describe_plan(2, **q) == \
        "gate_up=moe_gate_up_3d_batched<1,1> down=moe_down_3d_batched<2,3> pdl=3 launches=2"
    assert wd.wd_moe_describe_plan(4, **q) == \
        "gate_up=moe_gate_up_3d_batched<1,1> down=moe_down_3d_batched<4,1> pdl=3 launches=2"
    # tokens share experts: tensor-core gate/up; from B*K >= E on, each routed
    # down row is read once for all of its pairs
    assert wd.wd_moe_describe_plan(8, **q) == \
        "gate_up=moe_gate_up_mma<8,0> down=moe_down_3d_batched<4,1> pdl=1 launches=2"
    for B in (16, 32):
        assert wd.wd_moe_describe_plan(B, **q) == \
            "gate_up=moe_gate_up_mma<8,0> down=moe_down_dimblock<4,3,8,2> pdl=7 launches=3"
    # H above the tensor-core gate/up kernel's limit: the CUDA-core persistent kernel
    assert wd.wd_moe_describe_plan(32, 4096, 768, 128, 8).startswith(
        "gate_up=moe_gate_up_persist<2,1> down=moe_down_dimblock<4,3,8,2>")
    # B*K above the persistent kernels' routing tables: shared-row gate/up, batched down
    assert wd.wd_moe_describe_plan(64, **q) == \
        "gate_up=moe_gate_up_rowshare<2,2> down=moe_down_3d_batched<4,1> pdl=3 launches=2"
    # I not a multiple of 128: no tensor-map slabs for the down rows
    assert "down=moe_down_3d_batched<4,1>" in wd.wd_moe_describe_plan(32, 2048, 800, 128, 8)
    wd.wd_moe_set_plan("gu=mma,dn=4:1,pdl=1")
    try:
        assert wd.wd_moe_describe_plan(32, **q) == \
            "gate_up=moe_gate_up_mma<8,0> down=moe_down_3d_batched<4,1> pdl=1 launches=2"
    finally:
        wd.wd_moe_set_plan(None)
    # the shared-row down on request even where tokens rarely share experts
    wd.wd_moe_set_plan("dn=dimblock:1:3:3:2")
    try:
        assert wd.wd_moe_describe_plan(2, **q).endswith("down=moe_down_dimblock<1,3,3,2> pdl=7 launches=3")
        assert "down=moe_down_3d_batched<4,1>" in wd.wd_moe_describe_plan(128, 2048, 768, 128, 2)
    finally:
        wd.wd_moe_set_plan(None)
    lib = wd.lib()
    buf = ctypes.create_string_buffer(64)
    assert lib.wd_moe_describe_plan(32, 2048, 768, 128, 8, buf, 64) == INVALID
    buf = ctypes.create_string_buffer(128)
    assert lib.wd_moe_describe_plan(0, 2048, 768, 128, 8, buf, 128) == INVALID


def test_plan_override_parser():
    lib = wd.lib()
    assert lib.wd_moe_set_plan(b"gu=rowshare:2:1,dn=4:1,rowshare_min_b=4") == OK
    assert lib.wd_moe_set_plan(b"gu=batched:2:1") == OK
    assert lib.wd_moe_set_plan(b"gu=batched:2:1x") == INVALID
    assert lib.wd_moe_set_plan(b"gu=batched:1:1:2") == INVALID
    assert lib.wd_moe_set_plan(b"gu=persist:2:2,dn=4:1") == OK
    assert lib.wd_moe_set_plan(b"gu=mma,pdl=3") == OK
    assert lib.wd_moe_set_plan(b"gu=mma:2,pdl=0") == OK
    assert lib.wd_moe_set_plan(b"gu=mma:2:16,dn=dimblock") == OK
    assert lib.wd_moe_set_plan(b"dn=dimblock:4:2:6:2,pdl=7") == OK
    assert lib.wd_moe_set_plan(b"dn=dimblock:4:2:6") == INVALID
    assert lib.wd_moe_set_plan(b"dn=dimblock:4:2:6:1:1") == INVALID
    # kernels that are no longer part of the library
    for gone in (b"gu=tma", b"gu=ring:2", b"dn=emma", b"dn=shared:2", b"dn=persist:4:1"):
        assert lib.wd_moe_set_plan(gone) == INVALID
    assert lib.wd_moe_set_plan(b"pdl=8") == INVALID
    assert lib.wd_moe_set_plan(b"nonsense") == INVALID
    assert lib.wd_moe_set_plan(b"dn=2") == INVALID
    assert lib.wd_moe_set_plan(None) == OK
    assert lib.wd_moe_set_plan(b"") == OK
