"""GB300-native small-batch MoE decode layer on MXFP8 weights ("warp decode").

Two hand-written sm_103a CUDA kernels behind a C-ABI (include/wd_moe.h):
``moe_gate_up_3d_batched`` (one warp per token x routed expert x neuron group)
and ``moe_down_3d_batched`` (one warp per token x output-dim group, all K
experts folded into one FP32 register accumulator); for batches whose tokens
share experts the gate/up stage runs ``moe_gate_up_persist``, which reads and
dequantises each routed expert row once for all of its tokens
(``wd_moe_describe_plan`` names the kernels a shape gets).  This package is the
thin Python binding over that library; PyTorch only supplies device memory and
streams.

    from moe_decode_gate_gb300 import wd_moe_decode, wd_moe_workspace_size
"""
from ._native import (  # noqa: F401
    SIGNATURES,
    WdError,
    library_path,
    lib,
    wd_bench_copy,
    wd_bench_fill,
    wd_bench_read,
    wd_bench_sm_count,
    wd_bench_spec_gbs,
    wd_moe_decode,
    wd_moe_decode_no_alloc,
    wd_moe_describe_plan,
    wd_last_error_string,
    wd_moe_down,
    wd_moe_gate_up,
    wd_moe_launches_per_call,
    wd_moe_read_error_flag,
    wd_moe_set_plan,
    wd_moe_workspace_init,
    wd_moe_workspace_size,
    wd_status_string,
)
from .layer import MoEDecodeLayer  # noqa: F401
