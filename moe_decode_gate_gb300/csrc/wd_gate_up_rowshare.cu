// wd_gate_up_rowshare.cu - moe_gate_up_rowshare: the gate/up kernel for batches
// in which tokens share experts.
//
// Same computation as moe_gate_up_3d_batched (Cursor, "用 warp decode 实现更好的
// MoE 模型推理", section 两个 kernel 如何工作, gate/up paragraph): every output
// h[b,k,n] is one warp's reduction of gate row n and up row I+n of expert
// ids[b,k] against x[b], followed by SiLU(gate) * up and one BF16 store.  What
// changes is how much work one warp does with a row once it has it: a warp owns
// NPW neurons of ONE routed expert and produces them for EVERY token routed to
// that expert, so each weight row is read from HBM and dequantised once per
// layer instead of once per (token, slot).  At B=32 with uniform routing that
// is 256 (token, slot) pairs over ~112 distinct experts.
//
// Which experts a CTA serves, and for which tokens, is read straight from the
// routing: the CTA scans the B*K ids into a shared-memory bitmap of routed
// experts, takes the u-th set bit (u = blockIdx.y) as its expert, and lists the
// (token, slot) pairs routed to it.  Nothing is padded, no activation is
// gathered or copied, and there is no combine: each warp still writes its own
// outputs directly, with no state shared between warps.
#include "wd_device.cuh"
#include "wd_launch.h"

namespace wd {

// Activation loads; `p` carries grid_dependency_wait()'s token (see wd_device.cuh).
__device__ __forceinline__ uint4 ld_act_16B(const void* p) {
  uint4 r;
  asm("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_act_8B(const void* p) {
  uint2 r;
  asm("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// Dot products of R weight rows (NPW gate rows then NPW up rows) with the
// activations of TC tokens.  Lane l handles MXFP8 blocks l, l+32, ...; each
// block is dequantised once (scale folded in), 4*SBW elements at a time, and
// used for all TC tokens.
template <int NPW, int TC, int SBW>
__device__ __forceinline__ void rowshare_tokens(const uint8_t* __restrict__ gate_up,
                                                const uint8_t* __restrict__ gate_up_scale,
                                                const uint8_t* __restrict__ xbytes,
                                                __nv_bfloat16* __restrict__ h,
                                                const int* __restrict__ slots, size_t gate_row0,
                                                int n0, int H, int I, int K) {
  constexpr int R = 2 * NPW;
  const int lane = threadIdx.x & 31;
  const int nblk = H >> 5;
  const size_t up_row0 = gate_row0 + I;
  uint32_t xoff[TC];  // byte offset of each token's x row (x is at most 128 MiB)
#pragma unroll
  for (int t = 0; t < TC; ++t) xoff[t] = (uint32_t)(slots[t] / K) * (uint32_t)H * 2u;

  float2 acc[TC][R];
#pragma unroll
  for (int t = 0; t < TC; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[t][r] = make_float2(0.f, 0.f);

  for (int blk = lane; blk < nblk; blk += 32) {
    U32x8 wv[R];
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const size_t row = (r < NPW) ? gate_row0 + r : up_row0 + (r - NPW);
      wv[r] = ld_weights_32B(gate_up + row * H + (size_t)blk * 32);
      sc[r] = e8m0_to_f32(ld_scale(gate_up_scale + row * nblk + blk));
    }
#pragma unroll
    for (int sb = 0; sb < 8 / SBW; ++sb) {  // 4*SBW elements per step
      float2 wf[R][2 * SBW];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int w = 0; w < SBW; ++w) {
          float2 lo, hi;
          e4m3x4_to_f32(wv[r].v[SBW * sb + w], lo, hi);
          const float2 s2 = make_float2(sc[r], sc[r]);
          wf[r][2 * w] = __fmul2_rn(lo, s2);
          wf[r][2 * w + 1] = __fmul2_rn(hi, s2);
        }
#pragma unroll
      for (int t = 0; t < TC; ++t) {
        float2 xf[2 * SBW];
        const uint8_t* xp = xbytes + xoff[t] + (size_t)blk * 64 + sb * 8 * SBW;
        if constexpr (SBW == 2) {
          const uint4 xv = ld_act_16B(xp);
          xf[0] = bf16x2_to_f32(xv.x);
          xf[1] = bf16x2_to_f32(xv.y);
          xf[2] = bf16x2_to_f32(xv.z);
          xf[3] = bf16x2_to_f32(xv.w);
        } else {
          const uint2 xv = ld_act_8B(xp);
          xf[0] = bf16x2_to_f32(xv.x);
          xf[1] = bf16x2_to_f32(xv.y);
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int w = 0; w < 2 * SBW; ++w) acc[t][r] = __ffma2_rn(wf[r][w], xf[w], acc[t][r]);
      }
    }
  }

#pragma unroll
  for (int t = 0; t < TC; ++t) {
    float hv[NPW];
#pragma unroll
    for (int r = 0; r < NPW; ++r) {
      const float g = warp_sum(acc[t][r].x + acc[t][r].y);
      const float u = warp_sum(acc[t][NPW + r].x + acc[t][NPW + r].y);
      hv[r] = silu(g) * u;
    }
#pragma unroll
    for (int r = 0; r < NPW; ++r)
      if (lane == t * NPW + r) h[(size_t)slots[t] * I + n0 + r] = __float2bfloat16_rn(hv[r]);
  }
}

template <int NPW, int SBW>
__global__ void __launch_bounds__(256, 2) moe_gate_up_rowshare(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const uint8_t* __restrict__ gate_up, const uint8_t* __restrict__ gate_up_scale,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K) {
  __shared__ uint32_t s_mask[kRowShareMaxExperts / 32];
  __shared__ int s_slot[kRowShareMaxSlots];
  __shared__ int s_count, s_expert, s_bad;

  // x and topk_ids may come from the kernel before this one on the stream.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BK = B * K;
  const int nwords = (E + 31) >> 5;
  const int n0 = (blockIdx.x * (blockDim.x >> 5) + warp) * NPW;

  // 1. bitmap of the experts this batch routes to
  for (int i = tid; i < nwords; i += blockDim.x) s_mask[i] = 0u;
  if (tid == 0) {
    s_count = 0;
    s_expert = -1;
    s_bad = 0;
  }
  __syncthreads();
  for (int s = tid; s < BK; s += blockDim.x) {
    const int e = __ldg(topk_ids + s);
    if (e >= 0 && e < E)
      atomicOr(&s_mask[e >> 5], 1u << (e & 31));
    else
      s_bad = 1;
  }
  __syncthreads();

  // out-of-range ids: their h entries are zero and the flag is raised (CTAs of
  // expert slot 0 cover every neuron block once)
  if (s_bad && blockIdx.y == 0) {
    for (int s = tid; s < BK; s += blockDim.x) {
      const int e = __ldg(topk_ids + s);
      if (e < 0 || e >= E)
        for (int n = blockIdx.x * (blockDim.x >> 5) * NPW; n < min(I, (int)(blockIdx.x + 1) * (int)(blockDim.x >> 5) * NPW); ++n)
          h[(size_t)s * I + n] = __float2bfloat16_rn(0.0f);
    }
    if (tid == 0 && blockIdx.x == 0 && error_flag) atomicOr(error_flag, 1u);
  }

  // 2. this CTA's expert: the blockIdx.y-th set bit of the bitmap (warp 0)
  if (warp == 0) {
    const int u = blockIdx.y;
    int base = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const uint32_t word = (w0 + lane < nwords) ? s_mask[w0 + lane] : 0u;
      const int c = __popc(word);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      const int first = base + incl - c;
      if (u >= first && u < first + c) {
        uint32_t wd = word;
        for (int i = first; i < u; ++i) wd &= wd - 1u;  // drop the lower set bits
        s_expert = (w0 + lane) * 32 + (__ffs(wd) - 1);
      }
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  __syncthreads();
  const int e = s_expert;
  if (e < 0) return;  // fewer distinct experts than expert slots: nothing to do

  // 3. the (token, slot) pairs routed to this expert
  for (int s = tid; s < BK; s += blockDim.x)
    if (__ldg(topk_ids + s) == e) s_slot[atomicAdd(&s_count, 1)] = s;
  __syncthreads();
  const int T = s_count;
  if (n0 >= I) return;

  const size_t gate_row0 = (size_t)e * 2 * I + n0;
  const uint8_t* xb = reinterpret_cast<const uint8_t*>(x) + wait_token;
  for (int c0 = 0; c0 < T; c0 += 4) {
    const int tc = min(4, T - c0);
    if (tc == 4)
      rowshare_tokens<NPW, 4, SBW>(gate_up, gate_up_scale, xb, h, s_slot + c0, gate_row0, n0, H, I, K);
    else if (tc == 3)
      rowshare_tokens<NPW, 3, SBW>(gate_up, gate_up_scale, xb, h, s_slot + c0, gate_row0, n0, H, I, K);
    else if (tc == 2)
      rowshare_tokens<NPW, 2, SBW>(gate_up, gate_up_scale, xb, h, s_slot + c0, gate_row0, n0, H, I, K);
    else
      rowshare_tokens<NPW, 1, SBW>(gate_up, gate_up_scale, xb, h, s_slot + c0, gate_row0, n0, H, I, K);
  }
}

template <int NPW, int SBW>
static cudaError_t launch_rowshare_t(const GateUpArgs& a, cudaStream_t stream, bool pdl) {
  const int warps_per_cta = 8;
  const int nb = (a.I + warps_per_cta * NPW - 1) / (warps_per_cta * NPW);
  const int slots = a.B * a.K < a.E ? a.B * a.K : a.E;  // at most this many distinct experts
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nb, (unsigned)slots);
  cfg.blockDim = dim3(32 * warps_per_cta);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_up_rowshare<NPW, SBW>,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids, a.gate_up,
                            a.gate_up_scale, reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K);
}

cudaError_t launch_gate_up_rowshare(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                    bool pdl) {
  if (a.B * a.K > kRowShareMaxSlots || a.E > kRowShareMaxExperts) return cudaErrorInvalidValue;
  // cpl selects the sub-block width for this variant: 1 -> 4 elements, 2 -> 8 elements per step
  if (p.npw == 1 && p.cpl == 2) return launch_rowshare_t<1, 2>(a, stream, pdl);
  if (p.npw == 1 && p.cpl == 1) return launch_rowshare_t<1, 1>(a, stream, pdl);
  if (p.npw == 2 && p.cpl == 1) return launch_rowshare_t<2, 1>(a, stream, pdl);
  if (p.npw == 2 && p.cpl == 2) return launch_rowshare_t<2, 2>(a, stream, pdl);
  return cudaErrorInvalidConfiguration;
}

}  // namespace wd
