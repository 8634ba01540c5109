"""The CUDA path's own accuracy against the FP64 unrounded reference, next to
the accuracy study's formats (Cursor, "用 warp decode 实现更好的 MoE 模型推理",
section 精度提升: keeping activations in BF16 with FP32 accumulation is closer
to full precision than re-quantising them to MXFP8).

On the seeded Qwen-3-style layer of the study, the library's BF16 output must
be about as close to the unrounded reference as the oracle's own output rounded
to BF16 (the only rounding the path defines besides h), and well inside the
error of the MXFP8-activation path.
"""
import pytest

import accuracy_study as acc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [1, 8, 32])
def test_cuda_path_error_matches_the_bf16_path(cuda_device, B):
    g = acc.gpu_column(B=B, device=str(cuda_device))
    r = acc.study(B=B)
    print(f"B={B}: CUDA {g['rel_rms_gpu']:.4e}, oracle BF16 out {g['rel_rms_oracle_bf16']:.4e}, "
          f"MXFP8 activations {r['rel_rms_traditional']:.4e} ({g['plan']})")
    # FP32 accumulation in another order adds a little to the oracle's own error
    assert g["rel_rms_gpu"] <= 1.05 * g["rel_rms_oracle_bf16"]
    assert g["rel_rms_gpu"] * 10 < r["rel_rms_traditional"]
