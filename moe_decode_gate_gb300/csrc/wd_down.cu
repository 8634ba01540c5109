// wd_down.cu - moe_down_3d_batched, the second of the two decode kernels.
//
// Cursor, "用 warp decode 实现更好的 MoE 模型推理", section 两个 kernel 如何工作
// (How the two kernels work), down paragraph: each warp owns one output
// dimension of one token, walks all top-k routed experts, streams each one's
// down-projection row against the intermediate activations h, and folds every
// expert's routing weight into ONE running FP32 accumulator; after the last
// expert a __shfl_xor_sync butterfly reduces the 32 lane partials and the
// warp writes one value.  The weighted top-k combine is part of the projection
// itself, not a separate epilogue.
//
// GB300 mapping:
//   - the K routed rows of one output dim form one virtual stream of K*I/32
//     MXFP8 blocks (192 for K=8, I=768: 6 per lane), so every lane is busy even
//     when I/32 is not a multiple of 32, and all of a warp's weight bytes are
//     in flight at once;
//   - a warp owns RPW consecutive output dims of one token and reuses each h
//     block RPW times from registers;
//   - the weight loads depend only on the call's inputs, so they are issued
//     BEFORE waiting on the first kernel (programmatic dependent launch): the
//     down rows stream in while the gate/up kernel finishes;
//   - warps are numbered output-dim-major, token-minor, so tokens that share
//     an expert read its rows while they are still in L2.
#include "wd_device.cuh"
#include "wd_launch.h"

namespace wd {

template <int RPW, int QPL>
__global__ void __launch_bounds__(256, 2) moe_down_3d_batched(
    const __nv_bfloat16* __restrict__ h, const int32_t* __restrict__ topk_ids,
    const float* __restrict__ topk_w, const uint8_t* __restrict__ down,
    const uint8_t* __restrict__ down_scale, __nv_bfloat16* __restrict__ out,
    uint32_t* __restrict__ error_flag, int B, int H, int I, int E, int K,
    unsigned long long ib_magic) {
  grid_launch_dependents();

  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long total = (long long)(H / RPW) * B;
  if (gw >= total) return;
  const int grp = (int)(gw / B);
  const int b = (int)(gw - (long long)grp * B);
  const int d0 = grp * RPW;
  const int ib = I >> 5;  // MXFP8 blocks per down row
  const int nq = K * ib;  // virtual blocks over all K routed rows
  const int32_t* ids = topk_ids + (size_t)b * K;
  const float* tw = topk_w + (size_t)b * K;
  const uint8_t* hb = reinterpret_cast<const uint8_t*>(h + (size_t)b * K * I);

  float acc[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) acc[r] = 0.0f;
  bool bad = false;

  for (int q0 = 0; q0 < nq; q0 += 32 * QPL) {
    U32x8 wd[RPW][QPL];
    uint32_t sd[RPW][QPL];
    float wk[QPL];
    int hoff[QPL];  // byte offset of the h block within this token's h
    bool ok[QPL];
#pragma unroll
    for (int j = 0; j < QPL; ++j) {
      const int q = q0 + lane + 32 * j;
      ok[j] = false;
      if (q < nq) {
        // k = q / ib without a division: ib_magic = ceil(2^32 / ib) is exact for
        // q * ib < 2^32 (q < K*ib <= 32768, ib <= 512)
        const int k = (int)(((unsigned long long)q * ib_magic) >> 32);
        const int blk = q - k * ib;
        const int e = __ldg(ids + k);
        if (e >= 0 && e < E) {
          ok[j] = true;
          wk[j] = __ldg(tw + k);
          hoff[j] = (k * I + blk * 32) * 2;
          const size_t row0 = (size_t)e * H + d0;
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            wd[r][j] = ld_weights_32B(down + (row0 + r) * I + (size_t)blk * 32);
            sd[r][j] = ld_scale(down_scale + (row0 + r) * ib + blk);
          }
        } else {
          bad = true;
        }
      }
    }
    // h is produced by the first kernel: wait for it (once; later calls return at once)
    const uint32_t wait_token = grid_dependency_wait();
#pragma unroll
    for (int j = 0; j < QPL; ++j) {
      if (ok[j]) {
        const U32x8 ha = ld_act_32B(hb + hoff[j] + wait_token);
        const U32x8 hc = ld_act_32B(hb + hoff[j] + wait_token + 32);
        float2 hf[16];
        unpack_act32(ha, hc, hf);
#pragma unroll
        for (int r = 0; r < RPW; ++r)
          acc[r] = fmaf(wk[j] * e8m0_to_f32(sd[r][j]), block_dot(wd[r][j], hf), acc[r]);
      }
    }
  }

  float y[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) y[r] = warp_sum(acc[r]);
#pragma unroll
  for (int r = 0; r < RPW; ++r)
    if (lane == r) out[(size_t)b * H + d0 + r] = __float2bfloat16_rn(y[r]);
  if (error_flag && __any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(error_flag, 1u);
}

template <int RPW, int QPL>
static cudaError_t launch_down_t(const DownArgs& a, cudaStream_t stream, bool pdl) {
  const long long warps = (long long)(a.H / RPW) * a.B;
  const long long blocks = (warps + 7) / 8;
  const unsigned long long ib = (unsigned long long)(a.I / 32);
  const unsigned long long ib_magic = ((1ull << 32) + ib - 1) / ib;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_3d_batched<RPW, QPL>,
                            reinterpret_cast<const __nv_bfloat16*>(a.h), a.topk_ids, a.topk_w,
                            a.down, a.down_scale, reinterpret_cast<__nv_bfloat16*>(a.out),
                            a.error_flag, a.B, a.H, a.I, a.E, a.K, ib_magic);
}

cudaError_t launch_down(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl) {
#define WD_DN_CASE(RPW, QPL) \
  if (p.rpw == RPW && p.qpl == QPL) return launch_down_t<RPW, QPL>(a, stream, pdl);
  WD_DN_CASE(1, 1)
  WD_DN_CASE(1, 2)
  WD_DN_CASE(1, 4)
  WD_DN_CASE(1, 6)
  WD_DN_CASE(2, 1)
  WD_DN_CASE(2, 2)
  WD_DN_CASE(2, 3)
  WD_DN_CASE(4, 1)
  WD_DN_CASE(4, 2)
#undef WD_DN_CASE
  return cudaErrorInvalidConfiguration;
}

}  // namespace wd
