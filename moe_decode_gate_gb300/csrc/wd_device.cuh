// wd_device.cuh - device helpers shared by the two MoE decode kernels.
//
// Loads: weight rows are streamed once per use with 256-bit (32-byte) vector
// loads through the read-only path without allocating in L1, so one lane
// fetches exactly one MXFP8 block (32 E4M3 codes) per instruction and a warp
// covers 1 KiB of a row per instruction.  Activations (x, h) are small, reused
// by many warps and written by the preceding kernel, so they use plain coherent
// loads that may allocate in L1.
//
// Dequantisation follows the MXFP8 definition (OCP MX v1.0): value =
// E4M3(code) * 2^(scale - 127).  The E4M3 -> FP16 conversion is exact (every
// finite E4M3 value is an FP16 normal), FP16 -> FP32 is exact, and the
// power-of-two block scale is applied once to the FP32 partial sum of the
// block's 32 products, which equals scaling every element (barring FP32
// overflow or underflow of the partial).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace wd {

struct U32x8 {
  uint32_t v[8];
};

// The load helpers below are plain (non-volatile) asm with no memory clobber,
// so the compiler may schedule them freely: hoist them above arithmetic, batch
// them and overlap their latencies.  Weights and scales are read-only for the
// whole launch, so that is always safe.  Activations may be written by the
// kernel before this one on the stream: their addresses must carry the token
// returned by grid_dependency_wait() (a zero that the compiler cannot see
// through), which keeps every such load after the wait.

// 32 bytes of a weight row: read-only for the kernel's lifetime, no L1 allocation.
__device__ __forceinline__ U32x8 ld_weights_32B(const void* p) {
  U32x8 r;
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]),
                 "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
               : "l"(p));
  return r;
}

// 32 bytes of an activation vector (written by an earlier kernel): coherent
// load; `p` must depend on grid_dependency_wait()'s token.
__device__ __forceinline__ U32x8 ld_act_32B(const void* p) {
  U32x8 r;
  asm("ld.global.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
        "=r"(r.v[6]), "=r"(r.v[7])
      : "l"(p));
  return r;
}

// One scale byte, read-only, no L1 allocation.
__device__ __forceinline__ uint32_t ld_scale(const uint8_t* p) {
  uint16_t r;
  asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// E8M0 scale code -> FP32 2^(code-127).  Code 0 is 2^-127 (an FP32 subnormal),
// code 255 is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
  const uint32_t bits = code == 0u ? 0x00400000u : (code == 255u ? 0x7FC00000u : code << 23);
  return __uint_as_float(bits);
}

// Four E4M3 codes (little-endian bytes of `w`, element 0 in bits 0..7) -> FP32,
// via the hardware e4m3x2 -> f16x2 conversion.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float2& lo, float2& hi) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  lo = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  hi = __half22float2(*reinterpret_cast<const __half2*>(&h23));
}

// Two BF16 values packed in a word (element 0 in the low half) -> FP32 pair.
__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// 32 activations (64 bytes, two 32-byte loads) -> 16 FP32 pairs.
__device__ __forceinline__ void unpack_act32(const U32x8& a, const U32x8& b, float2 (&xf)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) xf[i] = bf16x2_to_f32(a.v[i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) xf[8 + i] = bf16x2_to_f32(b.v[i]);
}

// Sum over one MXFP8 block of 32 codes times 32 FP32 activations, unscaled.
__device__ __forceinline__ float block_dot(const U32x8& w, const float2 (&xf)[16]) {
  float2 p0 = make_float2(0.f, 0.f), p1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float2 lo, hi;
    e4m3x4_to_f32(w.v[i], lo, hi);
    p0 = __ffma2_rn(lo, xf[2 * i], p0);
    p1 = __ffma2_rn(hi, xf[2 * i + 1], p1);
  }
  return (p0.x + p1.x) + (p0.y + p1.y);
}

// Butterfly all-reduce over the 32 lanes (shfl.sync.bfly): every lane ends
// with the full sum, with no shared memory and no barrier.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// Programmatic dependent launch controls (no-ops when launched without it).
// The wait returns a token equal to 0; adding it to an activation address
// makes that load data-dependent on the wait.
__device__ __forceinline__ uint32_t grid_dependency_wait() {
  uint32_t token;
  asm volatile("griddepcontrol.wait;\n\tmov.u32 %0, 0;" : "=r"(token) : : "memory");
  return token;
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

}  // namespace wd
