"""GB300-native small-batch MoE decode layer on MXFP8 weights ("warp decode").

Hand-written sm_103a CUDA kernels behind a C-ABI (include/wd_moe.h).  While
tokens rarely share experts (2*B*K < E) the layer is the pages' two kernels:
``moe_gate_up_3d_batched`` (one warp per token x routed expert x neuron group)
and ``moe_down_3d_batched`` (one warp per token x output-dim group, all K
experts folded into one FP32 register accumulator).  Once they share experts
each routed row is read and dequantised once for all of its tokens:
``moe_gate_up_mma`` (tensor-core products, one CTA per SM), then
``moe_h_encode`` and ``moe_down_dimblock`` (one CTA per 16 output dims over
every routed expert); ``wd_moe_describe_plan`` names the kernels a shape gets.
This package is the thin Python binding over that library; PyTorch only
supplies device memory and streams.

    from moe_decode_gate_gb300 import wd_moe_decode, wd_moe_workspace_size
"""
from ._native import (  # noqa: F401
    FLAG_BAD_EXPERT_ID,
    FLAG_PIPELINE_TIMEOUT,
    SIGNATURES,
    WdError,
    library_path,
    lib,
    wd_bench_copy,
    wd_bench_expert_centric,
    wd_bench_expert_centric_workspace_size,
    wd_bench_fill,
    wd_bench_hold,
    wd_bench_read,
    wd_bench_sm_count,
    wd_bench_spec_gbs,
    wd_moe_decode,
    wd_moe_decode_no_alloc,
    wd_moe_describe_plan,
    wd_last_error_string,
    wd_moe_down,
    wd_moe_down_encoded,
    wd_moe_down_workspace,
    wd_moe_h_encode,
    wd_moe_launches,
    wd_moe_gate_up,
    wd_moe_launches_per_call,
    wd_moe_read_error_flag,
    wd_moe_set_plan,
    wd_moe_workspace_init,
    wd_moe_workspace_size,
    wd_status_string,
)
from .layer import MoEDecodeLayer  # noqa: F401
