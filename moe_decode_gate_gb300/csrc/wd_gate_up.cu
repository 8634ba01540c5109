// wd_gate_up.cu - moe_gate_up_3d_batched, the first of the two decode kernels.
//
// Cursor, "用 warp decode 实现更好的 MoE 模型推理", section 两个 kernel 如何工作
// (How the two kernels work), gate/up paragraph: CTAs of 8 warps; each warp
// owns the intermediate neuron(s) of one (token, routed expert) pair, loads the
// routed expert id, streams that neuron's gate row and up row with the MXFP8
// codes converted on the fly, dots both against the same activation vector x
// (read once, reused for both projections, no shared-memory staging), reduces
// across the warp, applies SiLU(gate) * up and writes one BF16 value.
//
// GB300 mapping:
//   - a warp owns NPW consecutive neurons of one (token, slot) pair, so it keeps
//     2*NPW rows in flight (bytes in flight per warp = 2*NPW*H) and reuses each
//     x element 2*NPW times from registers;
//   - lane l handles MXFP8 blocks l, l+32, ... of every row: one 256-bit load
//     per block, so a warp-wide load covers 1 KiB of a row contiguously;
//   - warps are numbered neuron-group-major, (token, slot)-minor: warps that run
//     together read row n of every routed expert at once, so tokens that share
//     an expert hit the same rows in L2 instead of re-reading them from HBM.
#include "wd_device.cuh"
#include "wd_launch.h"

namespace wd {

// One neuron per warp and one block per lane per pass fits in 64 registers:
// 4 CTAs (32 warps) per SM, so the B = 1..4 grids need fewer waves.
template <int NPW, int CPL>
__global__ void __launch_bounds__(256, (NPW == 1 && CPL == 1) ? 4 : 2) moe_gate_up_3d_batched(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const uint8_t* __restrict__ gate_up, const uint8_t* __restrict__ gate_up_scale,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K) {
  // x and topk_ids may come from the kernel before this one on the stream.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();

  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int BK = B * K;
  const long long total = (long long)(I / NPW) * BK;
  if (gw >= total) return;
  const int grp = (int)(gw / BK);
  const int bk = (int)(gw - (long long)grp * BK);
  const int b = bk / K;
  const int n0 = grp * NPW;

  const int e = __ldg(topk_ids + bk);
  __nv_bfloat16* hout = h + (size_t)bk * I + n0;
  if (e < 0 || e >= E) {  // bad id: contributes nothing, raise the flag
    if (lane < NPW) hout[lane] = __float2bfloat16_rn(0.0f);
    if (lane == 0 && error_flag) atomicOr(error_flag, 1u);
    return;
  }

  const int nblk = H >> 5;  // MXFP8 blocks per row
  const size_t gate_row0 = (size_t)e * 2 * I + n0;
  const size_t up_row0 = gate_row0 + I;
  const uint8_t* xrow = reinterpret_cast<const uint8_t*>(x + (size_t)b * H) + wait_token;

  float accg[NPW], accu[NPW];
#pragma unroll
  for (int r = 0; r < NPW; ++r) accg[r] = accu[r] = 0.0f;

  for (int blk0 = 0; blk0 < nblk; blk0 += 32 * CPL) {
    U32x8 wg[NPW][CPL], wu[NPW][CPL];
    uint32_t sg[NPW][CPL], su[NPW][CPL];
    U32x8 xa[CPL], xb[CPL];
    // issue every load of this pass before any arithmetic
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int blk = blk0 + lane + 32 * j;
      if (blk < nblk) {
#pragma unroll
        for (int r = 0; r < NPW; ++r) {
          wg[r][j] = ld_weights_32B(gate_up + (gate_row0 + r) * H + (size_t)blk * 32);
          wu[r][j] = ld_weights_32B(gate_up + (up_row0 + r) * H + (size_t)blk * 32);
          sg[r][j] = ld_scale(gate_up_scale + (gate_row0 + r) * nblk + blk);
          su[r][j] = ld_scale(gate_up_scale + (up_row0 + r) * nblk + blk);
        }
        xa[j] = ld_act_32B(xrow + (size_t)blk * 64);
        xb[j] = ld_act_32B(xrow + (size_t)blk * 64 + 32);
      }
    }
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int blk = blk0 + lane + 32 * j;
      if (blk < nblk) {
        float2 xf[16];
        unpack_act32(xa[j], xb[j], xf);
#pragma unroll
        for (int r = 0; r < NPW; ++r) {
          accg[r] = fmaf(e8m0_to_f32(sg[r][j]), block_dot(wg[r][j], xf), accg[r]);
          accu[r] = fmaf(e8m0_to_f32(su[r][j]), block_dot(wu[r][j], xf), accu[r]);
        }
      }
    }
  }

  float hv[NPW];
#pragma unroll
  for (int r = 0; r < NPW; ++r) {
    const float g = warp_sum(accg[r]);
    const float u = warp_sum(accu[r]);
    hv[r] = silu(g) * u;
  }
  // lane r stores neuron r (every lane holds every reduced value)
#pragma unroll
  for (int r = 0; r < NPW; ++r)
    if (lane == r) hout[r] = __float2bfloat16_rn(hv[r]);
}

template <int NPW, int CPL>
static cudaError_t launch_gate_up_t(const GateUpArgs& a, cudaStream_t stream, bool pdl) {
  const long long warps = (long long)(a.I / NPW) * a.B * a.K;
  const int threads = 256;
  const long long blocks = (warps + 7) / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_up_3d_batched<NPW, CPL>,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids, a.gate_up,
                            a.gate_up_scale, reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K);
}

cudaError_t launch_gate_up(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                           bool pdl) {
  if (p.variant == kGateUpRowShare) return launch_gate_up_rowshare(a, p, stream, pdl);
  if (p.variant == kGateUpPersist) return launch_gate_up_persist(a, p, stream, pdl);
  if (p.variant == kGateUpMma) return launch_gate_up_mma(a, p, stream, pdl);
#define WD_GU_CASE(NPW, CPL) \
  if (p.npw == NPW && p.cpl == CPL) return launch_gate_up_t<NPW, CPL>(a, stream, pdl);
  WD_GU_CASE(1, 1)
  WD_GU_CASE(1, 2)
  WD_GU_CASE(2, 1)
#undef WD_GU_CASE
  return cudaErrorInvalidConfiguration;
}

}  // namespace wd
