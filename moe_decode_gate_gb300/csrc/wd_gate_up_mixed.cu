// wd_gate_up_mixed.cu - moe_gate_up_mixed: the streamed gate/up kernel with its
// dot products on mixed-precision FMAs (FP16 x FP16 -> FP32 accumulate).
//
// Computes exactly what moe_gate_up_3d_batched computes (Cursor, "用 warp
// decode 实现更好的 MoE 模型推理", section 两个 kernel 如何工作, gate/up
// paragraph): for each (token, routed slot) and intermediate neuron n, one warp
// reduces gate row n and up row I+n of the routed expert against x, applies
// SiLU(gate) * up and writes one BF16 value.  The output-centric structure
// stays: every warp owns a fixed set of outputs and shares no state with other
// warps; there is no padding, no activation gather and no combine.
//
// Arithmetic: every finite E4M3 value is an FP16 normal, so one hardware
// cvt.rn.f16x2.e4m3x2 per pair gives the weights exactly; x is converted once
// per CTA to FP16 in shared memory, token by token, and only where that is
// exact (every element zero or with a binary exponent in [-17, 15]); a token
// that does not fit keeps its BF16 values and takes the FP32 path.  Each
// product w * x is then exact inside fma.rn.f32.f16 and accumulates in FP32 with
// one rounding per term, as with FP32 operands, while skipping the FP16 -> FP32
// widening that otherwise dominates the FMA pipes.  The E8M0 block scale
// multiplies each 8-element partial sum.
//
// What is GB300-specific is how the rows reach the warps:
//   - persistent CTAs walk a static list of work items; an item is (routed
//     expert, up to kTC of the tokens routed to it, NG = C*NPW neurons);
//   - one producer thread per CTA streams each item into a ring of shared-
//     memory stages with cp.async.bulk, armed on an mbarrier: the NG gate rows
//     and the NG up rows are each ONE contiguous copy (NG*H bytes), then the
//     two scale blocks.  Large copies are what keeps a GB300 at its streaming
//     bandwidth (small ones are issue-bound); weight rows use an evict-first L2
//     policy (read once per layer);
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
  int stage_bytes;  // gate rows, up rows, gate scales, up scales
  int x_off;        // every token's x (FP16 where exact, else BF16), B * H * 2 bytes
  int flag_off;     // per-token: 1 if x stayed BF16
  int routing_off;  // routing tables
  int scale_off;    // per-consumer-warp decoded scales (FP32)
  int stage_off;    // first stage
  int total;        // bytes of dynamic shared memory
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline StreamLayout stream_layout(int B, int H, int ng, int nst) {
  StreamLayout L;
  L.ng = ng;
  L.sw = H / 32;
  L.stage_bytes = round_up(2 * ng * H + 2 * ng * L.sw, 128);
  L.routing_off = round_up(2 * nst * 8, 128);
  L.scale_off = round_up(L.routing_off + routing_table_bytes(), 128);
  L.flag_off = round_up(L.scale_off + 2 * ng * L.sw * 4, 128);  // 2*NPW rows per warp
  L.x_off = round_up(L.flag_off + 4 * B, 128);
  L.stage_off = round_up(L.x_off + B * H * 2, 1024);
  L.total = L.stage_off + nst * L.stage_bytes;
  return L;
}

__device__ __forceinline__ float mfma16(uint32_t a, uint32_t b, float c) {  // a.lo*b.lo + c
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %3;\n\t}"
      : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float mfma16_hi(uint32_t a, uint32_t b, float c) {  // a.hi*b.hi + c
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %3;\n\t}"
      : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// Two E4M3 codes (low 16 bits / high 16 bits of w) -> FP16 pair, exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& h01, uint32_t& h23) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(h01), "=r"(h23) : "r"(w));
}

// 1 if the BF16 value with these bits is exactly representable in FP16.
__device__ __forceinline__ bool bf16_fits_f16(uint32_t bits16) {
  const uint32_t e = (bits16 >> 7) & 0xFFu;
  return (e == 0u && (bits16 & 0x7Fu) == 0u) || (e >= 110u && e <= 142u);
}

// One item for one consumer warp: dot the warp's 2*NPW rows (full rows,
// staged) with the item's TC tokens' x (shared memory).  Lane l handles the
// 8-element slices starting at columns 8*l + 256*i, i < NSL (H = 256*NSL), so
// every shared-memory access of the warp is contiguous.  `sc` holds the warp's
// rows' block scales decoded to FP32; `xrow[t]` is token t's x in shared
// memory, FP16 if `slow[t]` is 0 and BF16 otherwise.
template <int NPW, int TC, int NSL>
__device__ __forceinline__ void consume_item(uint32_t sbuf, const StreamLayout& L, int H,
                                             const float* __restrict__ sc,
                                             const uint32_t (&xrow)[kTC], const int (&slow)[kTC],
                                             float (&acc)[kTC][2 * NPW]) {
  constexpr int R = 2 * NPW;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint32_t rowp[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    rowp[r] = sbuf + (r < NPW ? 0u : (uint32_t)(L.ng * H)) + (uint32_t)((warp * NPW + r % NPW) * H);
#pragma unroll
  for (int i = 0; i < NSL; ++i) {
    const int c = 8 * lane + 256 * i;
    uint32_t wh[R][4];  // FP16 pairs: elements (0,1) (2,3) (4,5) (6,7) of the slice
    float s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint2 q = lds_u32x2(rowp[r] + c);
      e4m3x4_to_f16x2x2(q.x, wh[r][0], wh[r][1]);
      e4m3x4_to_f16x2x2(q.y, wh[r][2], wh[r][3]);
      s[r] = sc[r * (NSL * 8) + (c >> 5)];
    }
#pragma unroll
    for (int t = 0; t < TC; ++t) {
      uint4 xv;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                   : "r"(xrow[t] + (uint32_t)c * 2u));
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      if (!slow[t]) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float p = 0.0f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            p = mfma16(wh[r][k], xw[k], p);
            p = mfma16_hi(wh[r][k], xw[k], p);
          }
          acc[t][r] = fmaf(s[r], p, acc[t][r]);
        }
      } else {  // BF16 activations that FP16 cannot hold: FP32 products
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float2 p2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            p2 = __ffma2_rn(__half22float2(*reinterpret_cast<const __half2*>(&wh[r][k])),
                            bf16x2_to_f32(xw[k]), p2);
          acc[t][r] = fmaf(s[r], p2.x + p2.y, acc[t][r]);
        }
      }
    }
  }
}

// Reduce and store one item's outputs: tokens' h for the warp's NPW neurons.
template <int NPW, int TC>
__device__ __forceinline__ void store_item(const float (&acc)[kTC][2 * NPW],
                                           const int* __restrict__ slots,
                                           __nv_bfloat16* __restrict__ h, int n0, int I) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < TC; ++t) {
    const int slot = slots[t];
#pragma unroll
    for (int r = 0; r < NPW; ++r) {
      const float gs = warp_sum(acc[t][r]);
      const float us = warp_sum(acc[t][NPW + r]);
      if (lane == r) h[(size_t)slot * I + n0 + r] = __float2bfloat16_rn(silu(gs) * us);
    }
  }
}

template <int NPW, int TC, int NSL>
__device__ __forceinline__ void item_tc(uint32_t sbuf, const StreamLayout& L, int H,
                                        const float* sc, const int* slots, const int* xslow,
                                        uint32_t x_s, int K, __nv_bfloat16* h, int n0, int I,
                                        uint32_t empty_bar) {
  float acc[kTC][2 * NPW];
  uint32_t xrow[kTC];
  int slow[kTC];
#pragma unroll
  for (int t = 0; t < kTC; ++t) {
    const int b = (t < TC) ? slots[t] / K : 0;
    xrow[t] = x_s + (uint32_t)(b * H) * 2u;
    slow[t] = (t < TC) ? xslow[b] : 0;
#pragma unroll
    for (int r = 0; r < 2 * NPW; ++r) acc[t][r] = 0.0f;
  }
  consume_item<NPW, TC, NSL>(sbuf, L, H, sc, xrow, slow, acc);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);  // the stage is no longer read
  store_item<NPW, TC>(acc, slots, h, n0, I);
}

}  // namespace

template <int C, int NPW>
__global__ void __launch_bounds__(32 * (C + 1)) moe_gate_up_mixed(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const uint8_t* __restrict__ gate_up, const uint8_t* __restrict__ gate_up_scale,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K, int nst) {
  constexpr int kThreads = 32 * (C + 1);
  constexpr int NG = C * NPW;
  extern __shared__ __align__(1024) uint8_t smem[];
  const StreamLayout L = stream_layout(B, H, NG, nst);
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
  int* xslow = reinterpret_cast<int*>(smem + L.flag_off);
  const uint32_t x_s = smem_u32(smem + L.x_off);

  if (warp == C) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;  // (the consumers convert x meanwhile)
    const uint64_t pol_w = l2_evict_first_policy();
    int j = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
      const int q = it / n_groups;
      const int g = it - q * n_groups;
      const int u = rt.chunk_u[q];
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
      mbar_arrive_expect_tx(full, (uint32_t)(2 * NG * H + 2 * NG * L.sw));
      bulk_g2s(sbuf, gate_up + gate_row0 * H, NG * H, full, pol_w);
      bulk_g2s(sbuf + NG * H, gate_up + up_row0 * H, NG * H, full, pol_w);
      bulk_g2s(sbuf + 2 * NG * H, gate_up_scale + gate_row0 * L.sw, NG * L.sw, full, pol_w);
      bulk_g2s(sbuf + 2 * NG * H + NG * L.sw, gate_up_scale + up_row0 * L.sw, NG * L.sw, full,
               pol_w);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  // every token's x into shared memory once: FP16 where exact, BF16 otherwise
  {
    constexpr int kCons = 32 * C;
    for (int b = tid; b < B; b += kCons) xslow[b] = 0;
    named_barrier_sync(1, kCons);
    const uint32_t* xg = reinterpret_cast<const uint32_t*>(x);
    const int words = B * H / 2;
    for (int k = tid; k < words; k += kCons) {
      const uint32_t v = __ldg(xg + k);
      if (!bf16_fits_f16(v & 0xFFFFu) || !bf16_fits_f16(v >> 16)) xslow[k / (H / 2)] = 1;
    }
    named_barrier_sync(1, kCons);
    for (int k = tid; k < words; k += kCons) {
      const uint32_t v = __ldg(xg + k);
      uint32_t o = v;
      if (!xslow[k / (H / 2)]) {
        const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(hi), "f"(lo));
      }
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(x_s + 4u * k), "r"(o) : "memory");
    }
    named_barrier_sync(1, kCons);
  }
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
#define WD_ITEM(TCV, NSLV) \
  item_tc<NPW, TCV, NSLV>(sbuf, L, H, sc, slots, xslow, x_s, K, h, n0, I, empty)
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

StreamShape stream_shape(int B, int H, int ng, int nst_req) {
  constexpr int kSmem = 227 * 1024;
  StreamShape s;
  s.nst = nst_req > 0 ? nst_req : 2;
  while (s.nst > 2 && stream_layout(B, H, ng, s.nst).total > kSmem) --s.nst;
  s.L = stream_layout(B, H, ng, s.nst);
  s.ctas_per_sm = s.L.total <= kSmem / 2 - 1024 ? 2 : 1;
  return s;
}

// npw encodes (consumer warps, neurons per warp): 1 -> (8, 1), 2 -> (8, 2), 3 -> (4, 2)
int mixed_ng(int npw) { return npw == 1 ? 8 : (npw == 2 ? 16 : (npw == 3 ? 8 : 0)); }

}  // namespace

template <int C, int NPW>
static cudaError_t launch_mixed_t(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                  bool pdl) {
  const StreamShape sh = stream_shape(a.B, a.H, C * NPW, p.cpl);
  static int configured_bytes = 0;
  if (configured_bytes < sh.L.total) {
    const cudaError_t e = cudaFuncSetAttribute(moe_gate_up_mixed<C, NPW>,
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
  return cudaLaunchKernelEx(&cfg, moe_gate_up_mixed<C, NPW>,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids, a.gate_up,
                            a.gate_up_scale, reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K, sh.nst);
}

bool gate_up_mixed_supported(int B, int H, int I, int E, int K, int npw) {
  const int ng = mixed_ng(npw);
  const int nsl = H / 256;
  return ng > 0 && B * K <= kStreamMaxSlots && E <= 4096 && H % 512 == 0 && I % ng == 0 &&
         (nsl == 2 || nsl == 4 || nsl == 8 || nsl == 16) &&
         stream_layout(B, H, ng, 2).total <= 227 * 1024;
}

cudaError_t launch_gate_up_mixed(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                 bool pdl) {
  if (!gate_up_mixed_supported(a.B, a.H, a.I, a.E, a.K, p.npw)) return cudaErrorInvalidValue;
  if (p.npw == 1) return launch_mixed_t<8, 1>(a, p, stream, pdl);
  if (p.npw == 2) return launch_mixed_t<8, 2>(a, p, stream, pdl);
  if (p.npw == 3) return launch_mixed_t<4, 2>(a, p, stream, pdl);
  return cudaErrorInvalidConfiguration;
}

}  // namespace wd
