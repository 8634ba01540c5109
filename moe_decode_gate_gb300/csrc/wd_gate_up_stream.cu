// wd_gate_up_stream.cu - moe_gate_up_stream: the gate/up kernel with its weight
// rows and activations streamed through a shared-memory ring by bulk copies.
//
// Computes exactly what moe_gate_up_3d_batched computes (Cursor, "用 warp
// decode 实现更好的 MoE 模型推理", section 两个 kernel 如何工作, gate/up
// paragraph): for each (token, routed slot) and intermediate neuron n, one warp
// reduces gate row n and up row I+n of the routed expert against x, applies
// SiLU(gate) * up and writes one BF16 value.  The output-centric structure
// stays: every warp owns a fixed set of outputs and shares no state with other
// warps; there is no padding, no activation gather and no combine.
//
// What is GB300-specific is how the rows reach the warps:
//   - persistent CTAs walk a static list of work items; an item is (routed
//     expert, up to kTC of the tokens routed to it, NG = C*NPW neurons);
//   - one producer thread per CTA streams each item into a ring of shared-
//     memory stages with cp.async.bulk, armed on an mbarrier: the NG gate rows
//     and the NG up rows are each ONE contiguous copy (NG*H bytes), then the
//     two scale blocks and the item's tokens' x rows.  Large copies are what
//     keeps a GB300 at its streaming bandwidth (small ones are issue-bound);
//     weight rows use an evict-first L2 policy (read once per layer), x an
//     evict-last one (re-read by many CTAs);
//   - C consumer warps each own NPW neurons: they dequantise each 8-element
//     slice of their rows once and use it for every token of the item, reading
//     only shared memory, then release the stage.
// Which experts and tokens exist is read from the routing in the CTA prologue
// (bitmap of routed experts, token lists per expert, all in shared memory).
#include "wd_device.cuh"
#include "wd_launch.h"
#include "wd_pipeline.cuh"
#include "wd_routing.cuh"

namespace wd {

namespace {

constexpr int kTC = 4;  // tokens per work item (at most)

// Shared-memory layout (offsets in bytes), computed the same way on host and device.
struct StreamLayout {
  int ng;           // rows per matrix per stage
  int sw;           // scale bytes per row (H / 32)
  int x_off;        // x rows within a stage
  int stage_bytes;  // gate rows, up rows, gate scales, up scales, x rows
  int routing_off;  // routing tables
  int scale_off;    // per-consumer-warp decoded scales (FP32)
  int stage_off;    // first stage
  int total;        // bytes of dynamic shared memory
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline StreamLayout stream_layout(int H, int ng, int nst) {
  StreamLayout L;
  L.ng = ng;
  L.sw = H / 32;
  L.x_off = 2 * ng * H + 2 * ng * L.sw;
  L.stage_bytes = round_up(L.x_off + kTC * H * 2, 128);
  L.routing_off = round_up(2 * nst * 8, 128);
  L.scale_off = round_up(L.routing_off + routing_table_bytes(), 128);
  L.stage_off = round_up(L.scale_off + 2 * ng * L.sw * 4, 1024);  // 2*NPW rows per warp
  L.total = L.stage_off + nst * L.stage_bytes;
  return L;
}

// One item for one consumer warp: dot the warp's 2*NPW rows (full rows,
// staged) with the item's TC tokens' staged x rows.  Lane l handles the
// 8-element slices starting at columns 8*l + 256*i, i < NSL (H = 256*NSL), so
// every shared-memory access of the warp is contiguous.  `sc` holds the warp's
// rows' block scales, already decoded to FP32 (row-major, H/32 per row).
template <int NPW, int TC, int NSL>
__device__ __forceinline__ void consume_item(uint32_t sbuf, const StreamLayout& L, int H,
                                             const float* __restrict__ sc,
                                             float2 (&acc)[kTC][2 * NPW]) {
  constexpr int R = 2 * NPW;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint32_t rowp[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    rowp[r] = sbuf + (r < NPW ? 0u : (uint32_t)(L.ng * H)) + (uint32_t)((warp * NPW + r % NPW) * H);
  const uint32_t x_s = sbuf + L.x_off;
#pragma unroll
  for (int i = 0; i < NSL; ++i) {
    const int c = 8 * lane + 256 * i;
    float2 wf[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint2 q = lds_u32x2(rowp[r] + c);
      const float s = sc[r * (NSL * 8) + (c >> 5)];
      const float2 s2 = make_float2(s, s);
      float2 lo, hi;
      e4m3x4_to_f32(q.x, lo, hi);
      wf[r][0] = __fmul2_rn(lo, s2);
      wf[r][1] = __fmul2_rn(hi, s2);
      e4m3x4_to_f32(q.y, lo, hi);
      wf[r][2] = __fmul2_rn(lo, s2);
      wf[r][3] = __fmul2_rn(hi, s2);
    }
#pragma unroll
    for (int t = 0; t < TC; ++t) {
      uint4 xv;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                   : "r"(x_s + (uint32_t)(t * H + c) * 2u));
      const float2 x0 = bf16x2_to_f32(xv.x), x1 = bf16x2_to_f32(xv.y);
      const float2 x2 = bf16x2_to_f32(xv.z), x3 = bf16x2_to_f32(xv.w);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        acc[t][r] = __ffma2_rn(wf[r][0], x0, acc[t][r]);
        acc[t][r] = __ffma2_rn(wf[r][1], x1, acc[t][r]);
        acc[t][r] = __ffma2_rn(wf[r][2], x2, acc[t][r]);
        acc[t][r] = __ffma2_rn(wf[r][3], x3, acc[t][r]);
      }
    }
  }
}

// Reduce and store one item's outputs: tokens' h for the warp's NPW neurons.
template <int NPW, int TC>
__device__ __forceinline__ void store_item(const float2 (&acc)[kTC][2 * NPW],
                                           const int* __restrict__ slots,
                                           __nv_bfloat16* __restrict__ h, int n0, int I) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < TC; ++t) {
    const int slot = slots[t];
#pragma unroll
    for (int r = 0; r < NPW; ++r) {
      const float gs = warp_sum(acc[t][r].x + acc[t][r].y);
      const float us = warp_sum(acc[t][NPW + r].x + acc[t][NPW + r].y);
      if (lane == r) h[(size_t)slot * I + n0 + r] = __float2bfloat16_rn(silu(gs) * us);
    }
  }
}

template <int NPW, int TC, int NSL>
__device__ __forceinline__ void item_tc(uint32_t sbuf, const StreamLayout& L, int H,
                                        const float* sc, const int* slots,
                                        __nv_bfloat16* h, int n0, int I, uint32_t empty_bar) {
  float2 acc[kTC][2 * NPW];
#pragma unroll
  for (int t = 0; t < kTC; ++t)
#pragma unroll
    for (int r = 0; r < 2 * NPW; ++r) acc[t][r] = make_float2(0.f, 0.f);
  consume_item<NPW, TC, NSL>(sbuf, L, H, sc, acc);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);  // the stage is no longer read
  store_item<NPW, TC>(acc, slots, h, n0, I);
}

}  // namespace

template <int C, int NPW>
__global__ void __launch_bounds__(32 * (C + 1)) moe_gate_up_stream(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const uint8_t* __restrict__ gate_up, const uint8_t* __restrict__ gate_up_scale,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K, int nst) {
  constexpr int kThreads = 32 * (C + 1);
  constexpr int NG = C * NPW;
  extern __shared__ __align__(1024) uint8_t smem[];
  const StreamLayout L = stream_layout(H, NG, nst);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[nst], empty[nst]
  const RoutingTables rt = routing_tables_at(smem + L.routing_off);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BK = B * K;

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[nst + s]), C);
    }
    mbar_init_fence();
  }
  // x and topk_ids may come from the kernel before this one on the stream.
  grid_dependency_wait();
  grid_launch_dependents();
  build_routing_tables(rt, topk_ids, BK, E, kTC, kThreads);

  // out-of-range ids: zero their h rows (CTA 0) and raise the flag
  if (rt.scalar[2] && blockIdx.x == 0) {
    for (int s = 0; s < BK; ++s) {
      const int e = rt.ids[s];
      if (e < 0 || e >= E)
        for (int n = tid; n < I; n += kThreads) h[(size_t)s * I + n] = __float2bfloat16_rn(0.0f);
    }
    if (tid == 0 && error_flag) atomicOr(error_flag, 1u);
  }

  const int n_groups = I / NG;
  const int n_items = rt.scalar[1] * n_groups;

  if (warp == C) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    const uint64_t pol_w = l2_evict_first_policy();
    const uint64_t pol_x = l2_evict_last_policy();
    const uint8_t* xg = reinterpret_cast<const uint8_t*>(x);
    int j = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
      const int q = it / n_groups;
      const int g = it - q * n_groups;
      const int u = rt.chunk_u[q];
      const int first = rt.off[u] + (q - rt.coff[u]) * kTC;
      const int tc = min(kTC, rt.off[u + 1] - first);
      const size_t gate_row0 = (size_t)rt.expert[u] * 2 * I + (size_t)g * NG;
      const size_t up_row0 = gate_row0 + I;
      const int st = j % nst;
      const uint32_t full = smem_u32(&bars[st]), empty = smem_u32(&bars[nst + st]);
      if (!mbar_wait(empty, ((j / nst) & 1) ^ 1)) {
        if (error_flag) atomicOr(error_flag, 2u);
        // let the copies already issued land before the CTA can exit
        for (int k = (j > nst ? j - nst : 0); k < j; ++k)
          (void)mbar_wait(smem_u32(&bars[k % nst]), (k / nst) & 1);
        return;
      }
      const uint32_t sbuf = smem_u32(smem + L.stage_off + st * L.stage_bytes);
      mbar_arrive_expect_tx(full, (uint32_t)(L.x_off + tc * H * 2));
      bulk_g2s(sbuf, gate_up + gate_row0 * H, NG * H, full, pol_w);
      bulk_g2s(sbuf + NG * H, gate_up + up_row0 * H, NG * H, full, pol_w);
      bulk_g2s(sbuf + 2 * NG * H, gate_up_scale + gate_row0 * L.sw, NG * L.sw, full, pol_w);
      bulk_g2s(sbuf + 2 * NG * H + NG * L.sw, gate_up_scale + up_row0 * L.sw, NG * L.sw, full,
               pol_w);
      for (int t = 0; t < tc; ++t)
        bulk_g2s(sbuf + L.x_off + t * H * 2, xg + (size_t)(rt.slots[first + t] / K) * H * 2, H * 2,
                 full, pol_x);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  float* sc = reinterpret_cast<float*>(smem + L.scale_off) + warp * (2 * NPW) * L.sw;
  int j = 0;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
    const int q = it / n_groups;
    const int g = it - q * n_groups;
    const int u = rt.chunk_u[q];
    const int first = rt.off[u] + (q - rt.coff[u]) * kTC;
    const int tc = min(kTC, rt.off[u + 1] - first);
    const int st = j % nst;
    if (!mbar_wait(smem_u32(&bars[st]), (j / nst) & 1)) {
      if (error_flag && lane == 0) atomicOr(error_flag, 2u);
      return;
    }
    const uint32_t sbuf = smem_u32(smem + L.stage_off + st * L.stage_bytes);
    // this warp's rows' E8M0 block scales -> FP32, once per item
    for (int k = lane; k < 2 * NPW * L.sw; k += 32) {
      const int r = k / L.sw, b = k - r * L.sw;
      const uint32_t base = sbuf + 2 * NG * H + (r < NPW ? 0 : NG * L.sw);
      sc[k] = e8m0_to_f32(lds_u8(base + (warp * NPW + r % NPW) * L.sw + b));
    }
    __syncwarp();
    const int n0 = g * NG + warp * NPW;
    const int* slots = rt.slots + first;
    const uint32_t empty = smem_u32(&bars[nst + st]);
#define WD_ITEM(TCV, NSLV) item_tc<NPW, TCV, NSLV>(sbuf, L, H, sc, slots, h, n0, I, empty)
#define WD_ITEMS(NSLV)          \
  switch (tc) {                 \
    case 4: WD_ITEM(4, NSLV); break; \
    case 3: WD_ITEM(3, NSLV); break; \
    case 2: WD_ITEM(2, NSLV); break; \
    default: WD_ITEM(1, NSLV); break; \
  }
    switch (H >> 8) {
      case 2: WD_ITEMS(2); break;
      case 4: WD_ITEMS(4); break;
      case 8: WD_ITEMS(8); break;
      default: WD_ITEMS(16); break;
    }
#undef WD_ITEMS
#undef WD_ITEM
    __syncwarp();
  }
}

namespace {

// Stages: as many as fit one CTA (at least 2); CTAs per SM: as many as fit.
struct StreamShape {
  int nst, ctas_per_sm;
  StreamLayout L;
};

StreamShape stream_shape(int H, int ng, int nst_req) {
  constexpr int kSmem = 227 * 1024;
  StreamShape s;
  s.nst = nst_req > 0 ? nst_req : 2;
  while (s.nst > 2 && stream_layout(H, ng, s.nst).total > kSmem) --s.nst;
  s.L = stream_layout(H, ng, s.nst);
  s.ctas_per_sm = s.L.total <= kSmem / 2 - 1024 ? 2 : 1;
  return s;
}

// npw encodes (consumer warps, neurons per warp): 1 -> (8, 1), 2 -> (8, 2), 3 -> (4, 2)
int stream_ng(int npw) { return npw == 1 ? 8 : (npw == 2 ? 16 : (npw == 3 ? 8 : 0)); }

}  // namespace

template <int C, int NPW>
static cudaError_t launch_stream_t(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                   bool pdl) {
  const StreamShape sh = stream_shape(a.H, C * NPW, p.cpl);
  static int configured_bytes = 0;
  if (configured_bytes < sh.L.total) {
    const cudaError_t e = cudaFuncSetAttribute(moe_gate_up_stream<C, NPW>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               sh.L.total);
    if (e != cudaSuccess) return e;
    configured_bytes = sh.L.total;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sh.ctas_per_sm * sms));
  cfg.blockDim = dim3(32 * (C + 1));
  cfg.dynamicSmemBytes = (size_t)sh.L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_up_stream<C, NPW>,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids, a.gate_up,
                            a.gate_up_scale, reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K, sh.nst);
}

bool gate_up_stream_supported(int B, int H, int I, int E, int K, int npw) {
  const int ng = stream_ng(npw);
  const int nsl = H / 256;
  return ng > 0 && B * K <= kStreamMaxSlots && E <= 4096 && H % 512 == 0 && I % ng == 0 &&
         (nsl == 2 || nsl == 4 || nsl == 8 || nsl == 16) &&
         stream_layout(H, ng, 2).total <= 227 * 1024;
}

cudaError_t launch_gate_up_stream(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                  bool pdl) {
  if (!gate_up_stream_supported(a.B, a.H, a.I, a.E, a.K, p.npw)) return cudaErrorInvalidValue;
  if (p.npw == 1) return launch_stream_t<8, 1>(a, p, stream, pdl);
  if (p.npw == 2) return launch_stream_t<8, 2>(a, p, stream, pdl);
  if (p.npw == 3) return launch_stream_t<4, 2>(a, p, stream, pdl);
  return cudaErrorInvalidConfiguration;
}

}  // namespace wd
