// wd_down_wmma.cu - moe_down_3d_mma: the pages' down kernel with each warp's
// dot products done by warp-level tensor-core MMAs.
//
// Same organisation as moe_down_3d_batched (Cursor, "用 warp decode 实现更好的
// MoE 模型推理", section 两个 kernel 如何工作, down paragraph): one warp per
// (token b, group of output dims), which walks the K routed experts of b,
// folds w[b,k] * (down rows . h[b,k,:]) for all k into register accumulators,
// and writes each of its outputs once as BF16.  No routing tables, no shared
// expert rows, no cross-warp combine.
//
// What changes is how a warp forms its dot products.  The group is 16 output
// dims, the 16 rows of one m16n8k16 MMA tile; all 8 columns of the tile carry
// the same (token, slot) activations, so column 0 of the result is the 16 dot
// products (the other columns repeat it).  Per weight element this costs half a
// cvt (E4M3x2 -> F16x2, exact, straight into the A fragment) and a share of an
// MMA, where the CUDA-core kernel widens every element to FP32 and multiplies
// it (~2.5 instructions per element and per (token, slot)).
//
// Each warp streams its K routed row pairs as one pipeline of 8-block passes:
// the next pass's weight loads are in flight while the current pass is
// computed, and the next slot's h row while the current slot's passes are.
//
// Activations: per routed slot the warp stages h[b,k,:] in shared memory as
// FP16 scaled by a power of two 2^p so that its largest magnitude lies in
// [2^14, 2^15) (exact for every BF16 value within 2^31 of that magnitude,
// smaller ones rounded to a 2^-38 grid of it, below the FP32 accumulation's own
// rounding); the slot's sum is multiplied by w[b,k] * 2^-p.  Block scales
// multiply each 32-column tile's partial sum in FP32 (exact barring FP32
// over/underflow).
#include "wd_launch.h"
#include "wd_mma.cuh"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kWWarps = 8;   // warps per CTA
constexpr int kWRows = 16;   // output dims per warp
constexpr int kWBlocks = 8;  // 32-column blocks per pass (two passes of loads in flight)

// 8 bytes of a weight row or of its scale codes: read-only for the whole
// launch, no L1 allocation.  Volatile, so that a pass's loads stay where the
// pipeline issues them (one pass ahead) instead of moving next to their use.
__device__ __forceinline__ uint2 ld_nc_8B(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}


}  // namespace

__global__ void __launch_bounds__(32 * kWWarps, 2) moe_down_3d_mma(
    const __nv_bfloat16* __restrict__ h, const int32_t* __restrict__ topk_ids,
    const float* __restrict__ topk_w, const uint8_t* __restrict__ down,
    const uint8_t* __restrict__ down_scale, __nv_bfloat16* __restrict__ out,
    uint32_t* __restrict__ error_flag, int B, int H, int I, int E, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  grid_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const long long gw = (long long)blockIdx.x * kWWarps + warp;
  if (gw >= (long long)(H / kWRows) * B) return;
  const int tile = (int)(gw / B), b = (int)(gw - (long long)tile * B);
  const int d0 = tile * kWRows;
  const int nbi = I >> 5, P = nbi / kWBlocks, NP = K * P;  // passes per row, in all
  const int nch = I >> 3;  // 16-byte chunks of 8 BF16 values per h row (<= 128)
  // this warp's two FP16 buffers for the staged h rows of consecutive slots
  const uint32_t hs = smem_u32(smem) + (uint32_t)(warp * I * 4);
  const int32_t* ids = topk_ids + (size_t)b * K;
  float y0 = 0.0f, y1 = 0.0f;  // output dims d0 + g and d0 + g + 8
  float a0 = 0.0f, a1 = 0.0f;  // the current slot's sums
  bool bad = false;
  // h may come from the kernel before this one on the stream
  const uint32_t wait_token = grid_dependency_wait();
  const uint8_t* hg = reinterpret_cast<const uint8_t*>(h) + wait_token;

  // lane k holds slot k's expert and weight (K <= 32), so addresses never wait on a load
  const int my_e = lane < K ? __ldg(ids + lane) : -1;
  const float my_w = lane < K ? __ldg(topk_w + (size_t)b * K + lane) : 0.0f;
  auto expert = [&](int k) {
    const int e = __shfl_sync(0xFFFFFFFFu, my_e, k);
    return (e >= 0 && e < E) ? e : -1;
  };
  // pass n: blocks jp*kWBlocks .. of the rows d0 + g, d0 + g + 8 of slot n / P's expert
  // (expert 0's rows for an out-of-range id: loaded, never used)
  auto load_pass = [&](int n, uint2 (&w0)[kWBlocks], uint2 (&w1)[kWBlocks], uint2& c0,
                       uint2& c1) {
    const int k = n / P, jp = n - k * P;
    const int e = max(expert(k), 0);
    const uint8_t* r0 = down + ((size_t)e * H + d0 + g) * I + tig * 8 + jp * kWBlocks * 32;
    const uint8_t* r1 = r0 + (size_t)8 * I;
#pragma unroll
    for (int j = 0; j < kWBlocks; ++j) {
      w0[j] = ld_nc_8B(r0 + 32 * j);
      w1[j] = ld_nc_8B(r1 + 32 * j);
    }
    const uint8_t* sc = down_scale + ((size_t)e * H + d0 + g) * nbi + jp * kWBlocks;
    c0 = ld_nc_8B(sc);  // the pass's 8 block scales of each row
    c1 = ld_nc_8B(sc + (size_t)8 * nbi);
  };
  // h row of slot k into registers (all chunks of this lane)
  uint4 hv[4];
  auto load_h = [&](int k) {
    const uint8_t* hrow = hg + ((size_t)b * K + k) * I * 2;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      hv[t] = (lane + 32 * t < nch) ? ld_act_16B(hrow + (lane + 32 * t) * 16)
                                    : make_uint4(0u, 0u, 0u, 0u);
  };
  // the registers' h row -> FP16 times 2^p in buffer `buf`; returns p
  auto stage_h = [&](int buf) {
    __syncwarp();  // the slot that used `buf` two slots ago is computed by every lane
    uint32_t mx = 0u;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      mx = max(mx, max(max(max_abs_bf16x2(hv[t].x), max_abs_bf16x2(hv[t].y)),
                       max(max_abs_bf16x2(hv[t].z), max_abs_bf16x2(hv[t].w))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    const int p = fp16_row_exponent(mx);
    const float f1 = exp2_int(p >> 1), f2 = exp2_int(p - (p >> 1));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (lane + 32 * t >= nch) break;
      const uint32_t in[4] = {hv[t].x, hv[t].y, hv[t].z, hv[t].w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = bf16x2_to_f32(in[q]);
        const __half2 v = __floats2half2_rn((f.x * f1) * f2, (f.y * f1) * f2);
        o[q] = *reinterpret_cast<const uint32_t*>(&v);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(hs + buf * I * 2 + (lane + 32 * t) * 16),
                   "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                   : "memory");
    }
    __syncwarp();
    return p;
  };
  // pass n from its registers, against the staged h of its slot
  auto compute_pass = [&](int n, const uint2 (&w0)[kWBlocks], const uint2 (&w1)[kWBlocks],
                          uint2 c0, uint2 c1) {
    const int k = n / P, jp = n - k * P;
    const uint32_t hb = hs + (k & 1) * I * 2 + (uint32_t)((jp * kWBlocks * 32 + tig * 8) * 2);
#pragma unroll
    for (int j = 0; j < kWBlocks; ++j) {
      const uint4 bv = lds_u32x4(hb + 64 * j);
      float cc[4];
      mma_f16_zero(cc, e4m3x2_lo_to_f16x2(w0[j].x), e4m3x2_lo_to_f16x2(w1[j].x),
                   e4m3x2_hi_to_f16x2(w0[j].x), e4m3x2_hi_to_f16x2(w1[j].x), bv.x, bv.y);
      mma_f16_acc(cc, e4m3x2_lo_to_f16x2(w0[j].y), e4m3x2_lo_to_f16x2(w1[j].y),
                  e4m3x2_hi_to_f16x2(w0[j].y), e4m3x2_hi_to_f16x2(w1[j].y), bv.z, bv.w);
      const uint32_t q0 = j < 4 ? c0.x : c0.y, q1 = j < 4 ? c1.x : c1.y;
      a0 = fmaf(cc[0], e8m0_to_f32((q0 >> (8 * (j & 3))) & 0xFFu), a0);
      a1 = fmaf(cc[2], e8m0_to_f32((q1 >> (8 * (j & 3))) & 0xFFu), a1);
    }
  };
  int p_cur = 0;
  // after the last pass of slot k: fold its sums into the outputs
  auto finish_slot = [&](int k) {
    if (expert(k) >= 0) {
      const float wv = __shfl_sync(0xFFFFFFFFu, my_w, k);
      const float f1 = exp2_int(-(p_cur >> 1)), f2 = exp2_int(-(p_cur - (p_cur >> 1)));
      y0 += ((a0 * wv) * f1) * f2;
      y1 += ((a1 * wv) * f1) * f2;
    } else {
      bad = true;
    }
    a0 = a1 = 0.0f;
  };

  // software pipeline over the NP passes: pass n + 1's rows are in flight
  // while pass n is computed, and the next slot's h row while the current
  // slot's passes are
  uint2 wA0[kWBlocks], wA1[kWBlocks], wB0[kWBlocks], wB1[kWBlocks];
  uint2 cA0, cA1, cB0, cB1;
  load_h(0);
  load_pass(0, wA0, wA1, cA0, cA1);
  p_cur = stage_h(0);
  if (K > 1) load_h(1);
  auto after_pass = [&](int n) {  // slot boundary after pass n
    if ((n + 1) % P != 0) return;
    const int k = n / P;
    finish_slot(k);
    if (k + 1 < K) {
      p_cur = stage_h((k + 1) & 1);
      if (k + 2 < K) load_h(k + 2);
    }
  };
  for (int n = 0; n < NP; n += 2) {
    if (n + 1 < NP) load_pass(n + 1, wB0, wB1, cB0, cB1);
    compute_pass(n, wA0, wA1, cA0, cA1);
    after_pass(n);
    if (n + 1 >= NP) break;
    if (n + 2 < NP) load_pass(n + 2, wA0, wA1, cA0, cA1);
    compute_pass(n + 1, wB0, wB1, cB0, cB1);
    after_pass(n + 1);
  }
  if (tig == 0) {
    out[(size_t)b * H + d0 + g] = __float2bfloat16_rn(y0);
    out[(size_t)b * H + d0 + g + 8] = __float2bfloat16_rn(y1);
  }
  if (bad && lane == 0 && error_flag) atomicOr(error_flag, 1u);
}

bool down_3d_mma_supported(int B, int H, int I, int E, int K) {
  (void)E;
  (void)B;
  return H % kWRows == 0 && I % (32 * kWBlocks) == 0 && I <= 1024 && K <= 32 &&
         I * 4 * kWWarps <= 48 * 1024;
}

cudaError_t launch_down_3d_mma(const DownArgs& a, const DownPlan& p, cudaStream_t stream,
                               bool pdl) {
  (void)p;
  if (!down_3d_mma_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  const long long warps = (long long)(a.H / kWRows) * a.B;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + kWWarps - 1) / kWWarps));
  cfg.blockDim = dim3(32 * kWWarps);
  cfg.dynamicSmemBytes = (size_t)(a.I * 4 * kWWarps);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_3d_mma, reinterpret_cast<const __nv_bfloat16*>(a.h),
                            a.topk_ids, a.topk_w, a.down, a.down_scale,
                            reinterpret_cast<__nv_bfloat16*>(a.out), a.error_flag, a.B, a.H, a.I,
                            a.E, a.K);
}

}  // namespace wd
