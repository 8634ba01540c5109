// wd_mma.cuh - pieces shared by the tensor-core kernels (moe_gate_up_mma,
// moe_down_dimblock): E4M3 -> FP16 conversion into MMA fragments, the
// warp-level m16n8k16 MMA, 3-D tensor-map copies into shared memory, the
// swizzled layout those copies produce, FP16 re-encoding of BF16 activations
// by a power of two, and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "wd_pipeline.cuh"

namespace wd {

// Byte offset of (row, col) in a 128-byte-swizzled slab [cols/128][16][128]:
// 16-byte chunk q of a 128-byte line is stored at q ^ (row % 8).
__device__ __forceinline__ uint32_t slab_offset(int row, int col) {
  return (uint32_t)((col >> 7) * 2048 + row * 128 + ((((col & 127) >> 4) ^ (row & 7)) << 4) +
                    (col & 15));
}

// Which of 8 slab rows MMA tile row g (0..7, the lane's group) reads: tile rows
// 0..3 take the even rows and 4..7 the odd ones, so that the 16 lanes of a
// half-warp (tile rows 0..3 or 4..7) read 8-byte pieces of one 32-column block
// from rows whose swizzle moves them to 8 different 16-byte chunks: the
// fragment loads are free of bank conflicts (with rows g, the rows g and g^1
// share a chunk pair and every load took two passes).
__device__ __forceinline__ int slab_row(int g) { return ((g & 3) << 1) | (g >> 2); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Two E4M3 codes (low 16 bits of w) -> f16x2, element 0 in the low half (exact).
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\t}"
      : "=r"(r)
      : "r"(w));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}"
      : "=r"(r)
      : "r"(w));
  return r;
}

// d = A(16x16, f16) * B(16x8, f16), FP32 accumulate from zero.
__device__ __forceinline__ void mma_f16_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}
// d += A * B.
__device__ __forceinline__ void mma_f16_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// 16 bytes of activations written by an earlier kernel: coherent load; `p`
// must depend on grid_dependency_wait()'s token.
__device__ __forceinline__ uint4 ld_act_16B(const void* p) {
  uint4 r;
  asm("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

// Exponent k such that 2^k times the largest magnitude (BF16 bits `mx`,
// sign cleared) lies in [2^14, 2^15); 0 for an all-zero row or a row holding
// Inf or NaN (whose results are not finite anyway).
__device__ __forceinline__ int fp16_row_exponent(uint32_t mx) {
  if (mx == 0u || mx >= 0x7F80u) return 0;
  const int ef = (int)(mx >> 7);
  const int e = ef ? ef - 127 : (31 - __clz((int)mx)) - 133;  // floor(log2(largest magnitude))
  return 14 - e;
}

// 2^k for k in [-126, 127].
__device__ __forceinline__ float exp2_int(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }


// True if any byte of w is an E8M0 code whose 8 bits are all equal: 0x00
// (2^-127) or 0xFF (NaN), the two codes that do not decode as code << 23.
__device__ __forceinline__ bool e8m0x4_any_special(uint32_t w) {
  const uint32_t d = (w ^ (w >> 1)) & 0x7F7F7F7Fu;  // per byte: 0 iff all 8 bits are equal
  return ((d + 0x7F7F7F7Fu) & 0x80808080u) != 0x80808080u;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Host: the driver's tensor-map encoder, looked up once (null if unavailable).
inline PFN_cuTensorMapEncodeTiled_v12000 mma_tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Host: a row-major byte matrix [rows][cols] (cols a multiple of 128) as the
// 3-D tensor {128, rows, cols/128} with strides {cols, 128}, so that one box
// {128, 16, box_cols/128} is box_cols columns of 16 rows (whole rows when
// box_cols is 0 or cols), stored in shared memory as [box_cols/128][16][128]
// with the 128-byte swizzle (slab_offset).
inline bool encode_row_slab_map(CUtensorMap* map, const void* base, uint64_t rows, int cols,
                                int box_cols = 0) {
  if (box_cols <= 0) box_cols = cols;
  PFN_cuTensorMapEncodeTiled_v12000 enc = mma_tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, rows, (cuuint64_t)(cols / 128)};
  const cuuint64_t strides[2] = {(cuuint64_t)cols, 128};
  const cuuint32_t box[3] = {128, 16, (cuuint32_t)(box_cols / 128)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host: a row-major byte matrix [rows][cols] (cols a multiple of 16) as the
// 3-D tensor {16, rows, cols/16} with strides {cols, 16}, so that one box
// {16, 16, cols/16} is 16 whole rows stored in shared memory as
// [cols/16][16][16]: the 16-byte groups of consecutive rows are adjacent.
inline bool encode_scale_group_map(CUtensorMap* map, const void* base, uint64_t rows, int cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = mma_tensor_map_encoder();
  if (!enc || cols % 16 != 0 || cols / 16 > 256) return false;
  const cuuint64_t dims[3] = {16, rows, (cuuint64_t)(cols / 16)};
  const cuuint64_t strides[2] = {(cuuint64_t)cols, 16};
  const cuuint32_t box[3] = {16, 16, (cuuint32_t)(cols / 16)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace wd
