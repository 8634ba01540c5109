// wd_gate_up_persist.cu - moe_gate_up_persist: the gate/up kernel as one wave
// of persistent CTAs over shared expert rows.
//
// Computes what moe_gate_up_3d_batched computes (Cursor, "用 warp decode 实现
// 更好的 MoE 模型推理", section 两个 kernel 如何工作, gate/up paragraph): for
// every (token, routed slot) and intermediate neuron n, the dot products of
// gate row n and up row I+n of the routed expert with x, then one BF16 value
// bf16(SiLU(g) * u).  Each output is still produced by exactly one warp, with
// no padding, no activation scatter and no combine pass.  What is organised
// differently, for batches in which tokens share experts:
//
//   - a warp owns NPW (1 or 2) neurons of one routed expert and produces them
//     for every token routed to that expert, so each weight row is read from
//     HBM and dequantised once per call;
//   - the grid is one wave of CTAs.  Each CTA builds the routing tables once
//     (routed experts ascending, their (token, slot) lists), then walks a
//     contiguous range of (expert, 8*NPW-neuron block) items.  Ranges are cut so
//     that every CTA gets the same estimated cost (items of an expert with T
//     tokens cost T + kItemBase units), so experts with many tokens do not
//     leave a tail;
//   - when a CTA moves to a new expert it stages that expert's tokens' x rows
//     in shared memory once, converted to FP32, each 32-element block padded
//     to 144 bytes so that the lanes of a warp (one MXFP8 block each) read them
//     without bank conflicts at immediate offsets.  The dot products then read
//     activations from shared memory with no conversion;
//   - the E8M0 block scale multiplies each 32-element partial sum rather than
//     every element (exact for a power of two barring FP32 over/underflow);
//   - the 4*TC partial sums of a chunk of TC tokens are reduced across the
//     warp by a transpose-reduction (each shuffle step halves the number of
//     values per lane), after which lane pairs hold gate and up of one output.
#include "wd_launch.h"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kItemBase = 3;                   // item cost = T + kItemBase
constexpr int kXMaxTokens = 8;                 // x rows staged at once (upper bound)
constexpr int kXBudget = 96 * 1024;            // shared-memory bytes for staged x

__host__ __device__ inline int persist_x_tokens(int H) {
  const int t = kXBudget / x_padded_row_bytes(H);
  return t < 1 ? 1 : (t > kXMaxTokens ? kXMaxTokens : t);
}

__host__ __device__ inline int persist_smem_bytes(int H) {
  return kXOffset + persist_x_tokens(H) * x_padded_row_bytes(H);
}

// One chunk of TC (<= 4) tokens for this warp's NPW neurons: dots of its
// 2*NPW rows (gate n0..n0+NPW-1, then up n0..n0+NPW-1) with the staged x of
// tokens t0..t0+TC-1, reduction, SiLU(g)*u, one BF16 store per output.
template <int NPW, int TC>
__device__ __forceinline__ void persist_chunk(const uint8_t* __restrict__ gate_up,
                                              const uint8_t* __restrict__ gate_up_scale,
                                              __nv_bfloat16* __restrict__ h, uint32_t xs,
                                              const int* __restrict__ slots, int t0,
                                              size_t gate_row0, int n0, int H, int I) {
  constexpr int R = 2 * NPW;
  constexpr int TCP = TC == 3 ? 4 : TC;
  const int lane = threadIdx.x & 31;
  const int nblk = H >> 5;
  const uint8_t* wbase = gate_up + gate_row0 * H;
  const uint8_t* sbase = gate_up_scale + gate_row0 * nblk;
  const size_t wup = (size_t)I * H;
  const int sup = I * nblk;
  const int row_bytes = x_padded_row_bytes(H);
  float acc[TCP][R];
#pragma unroll
  for (int t = 0; t < TCP; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[t][r] = 0.0f;

  for (int blk = lane; blk < nblk; blk += 32) {
    U32x8 wv[R];
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wv[r] = ld_weights_32B(wbase + (r / NPW) * wup + (r % NPW) * H + blk * 32);
      sc[r] = e8m0_to_f32(ld_scale(sbase + (r / NPW) * sup + (r % NPW) * nblk + blk));
    }
    float2 p[TC][R];
#pragma unroll
    for (int t = 0; t < TC; ++t)
#pragma unroll
      for (int r = 0; r < R; ++r) p[t][r] = make_float2(0.f, 0.f);
    // padded x layout: chunk c of this lane's block is at xt[t] + 16 c
    uint32_t xt[TC];
#pragma unroll
    for (int t = 0; t < TC; ++t)
      xt[t] = xs + (uint32_t)((t0 + t) * row_bytes + blk * kXPadBlockBytes);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float2 wf[R][2];
#pragma unroll
      for (int r = 0; r < R; ++r) e4m3x4_to_f32(wv[r].v[c], wf[r][0], wf[r][1]);
#pragma unroll
      for (int t = 0; t < TC; ++t) {
        const float4 xv = lds_f32x4(xt[t] + 16 * c);
        const float2 x01 = make_float2(xv.x, xv.y), x23 = make_float2(xv.z, xv.w);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          p[t][r] = __ffma2_rn(wf[r][0], x01, p[t][r]);
          p[t][r] = __ffma2_rn(wf[r][1], x23, p[t][r]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TC; ++t)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[t][r] = fmaf(p[t][r].x + p[t][r].y, sc[r], acc[t][r]);
  }

  store_chunk<NPW, TC, TCP>(acc, h, slots, n0, I);
}

}  // namespace

// PFD: items ahead whose rows lane 0 of each warp requests into L2
// (cp.async.bulk.prefetch) before computing the current one; 0 = none.
template <int NPW, int MINB, int PFD>
__global__ void __launch_bounds__(kPThreads, MINB) moe_gate_up_persist(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const uint8_t* __restrict__ gate_up, const uint8_t* __restrict__ gate_up_scale,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const uint32_t xs = smem_u32(smem + kXOffset);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K;
  const int xtok = persist_x_tokens(H);
  const int nblk = H >> 5;

  // x and topk_ids may come from the kernel before this one on the stream.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();
  build_routing_tables(rt, topk_ids, BK, E, 4, kPThreads);

  zero_bad_slots(rt, h, error_flag, BK, I, E);

  // cost-balanced contiguous range of (expert, neuron block) items for this CTA;
  // `coff` ([S + 1], unused here) holds the cost prefix
  const int U = rt.scalar[0];
  constexpr int kNeurons = kPWarps * NPW;  // neurons per item
  const int nb = (I + kNeurons - 1) / kNeurons;
  int* pc = rt.coff;
  expert_cost_prefix(rt, nb, kItemBase, pc);
  const long long total = pc[U];
  const int lo = (int)(total * blockIdx.x / gridDim.x);
  const int hi = (int)(total * (blockIdx.x + 1) / gridDim.x);
  if (lo >= hi) return;

  int u = first_expert(pc, U, lo);
  const uint8_t* xg = reinterpret_cast<const uint8_t*>(x) + wait_token;
  for (; u < U && pc[u] < hi; ++u) {
    const int T = rt.off[u + 1] - rt.off[u];
    const int cu = T + kItemBase;
    // items g of expert u whose cost start pc[u] + g*cu lies in [lo, hi)
    const int g0 = pc[u] >= lo ? 0 : (lo - pc[u] + cu - 1) / cu;
    const int g1 = min(nb, (hi - pc[u] + cu - 1) / cu);
    if (g0 >= g1) continue;
    const int* slots = rt.slots + rt.off[u];
    const size_t expert_row0 = (size_t)rt.expert[u] * 2 * I;
    for (int q0 = 0; q0 < T; q0 += xtok) {
      const int nq = min(xtok, T - q0);
      stage_x_padded(xs, xg, slots + q0, nq, H, K);
      // this warp's rows (NPW gate, NPW up; each group contiguous) of item gp, into L2
      auto prefetch_item = [&](int gp) {
        const int np = (gp * kPWarps + warp) * NPW;
        if (lane != 0 || gp >= g1 || np >= I) return;
        const size_t r0 = expert_row0 + np;
        prefetch_l2_bulk(gate_up + r0 * H, (uint32_t)(NPW * H));
        prefetch_l2_bulk(gate_up + (r0 + I) * H, (uint32_t)(NPW * H));
        prefetch_l2_bulk(gate_up_scale + r0 * nblk, (uint32_t)(NPW * nblk));
        prefetch_l2_bulk(gate_up_scale + (r0 + I) * nblk, (uint32_t)(NPW * nblk));
      };
#pragma unroll
      for (int k = 0; k < PFD; ++k) prefetch_item(g0 + k);
      for (int g = g0; g < g1; ++g) {
        if (PFD > 0) prefetch_item(g + PFD);
        const int n0 = (g * kPWarps + warp) * NPW;
        if (n0 >= I) continue;  // partial last block (I % (8*NPW) != 0)
        const size_t gate_row0 = expert_row0 + n0;
        for (int c0 = 0; c0 < nq; c0 += 4) {
          const int tc = min(4, nq - c0);
          const int* sl = slots + q0 + c0;
          if (tc == 4)
            persist_chunk<NPW, 4>(gate_up, gate_up_scale, h, xs, sl, c0, gate_row0, n0, H, I);
          else if (tc == 3)
            persist_chunk<NPW, 3>(gate_up, gate_up_scale, h, xs, sl, c0, gate_row0, n0, H, I);
          else if (tc == 2)
            persist_chunk<NPW, 2>(gate_up, gate_up_scale, h, xs, sl, c0, gate_row0, n0, H, I);
          else
            persist_chunk<NPW, 1>(gate_up, gate_up_scale, h, xs, sl, c0, gate_row0, n0, H, I);
        }
      }
    }
  }
}

bool gate_up_persist_supported(int B, int H, int I, int E, int K) {
  return B * K <= kStreamMaxSlots && E <= 4096 && H % 32 == 0 && I % 2 == 0 &&
         persist_smem_bytes(H) <= 113 * 1024;
}

template <int NPW, int MINB, int PFD>
static cudaError_t launch_persist_t(const GateUpArgs& a, cudaStream_t stream, bool pdl) {
  const int smem = persist_smem_bytes(a.H);
  {
    const cudaError_t e = ensure_dynamic_smem(
        reinterpret_cast<const void*>(moe_gate_up_persist<NPW, MINB, PFD>), smem);
    if (e != cudaSuccess) return e;
  }
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, moe_gate_up_persist<NPW, MINB, PFD>, kPThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(per_sm * sms));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_up_persist<NPW, MINB, PFD>,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids, a.gate_up,
                            a.gate_up_scale, reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K);
}

// p.npw: neurons per warp (1: 3 CTAs per SM, 2: 2 CTAs per SM); p.cpl: L2
// prefetch distance in items plus one (1: none, 2: one item ahead).
cudaError_t launch_gate_up_persist(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                   bool pdl) {
  if (!gate_up_persist_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  if (p.npw == 1) return p.cpl == 2 ? launch_persist_t<1, 3, 1>(a, stream, pdl)
                                    : launch_persist_t<1, 3, 0>(a, stream, pdl);
  return p.cpl == 2 ? launch_persist_t<2, 2, 1>(a, stream, pdl)
                    : launch_persist_t<2, 2, 0>(a, stream, pdl);
}

}  // namespace wd
