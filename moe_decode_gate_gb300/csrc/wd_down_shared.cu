// wd_down_shared.cu - moe_down_shared: the down projection over shared expert
// rows, for batches in which tokens share experts.
//
// Computes what moe_down_3d_batched computes (Cursor, "用 warp decode 实现更好
// 的 MoE 模型推理", section 两个 kernel 如何工作, down paragraph):
// out[b,d] = bf16( sum_k w[b,k] * (Wd[e_k][d,:] . h[b,k,:]) ), with the routing
// weight folded into the projection and no separate combine kernel.  The
// pages give each (token, output dim) its own warp, so a down row shared by T
// tokens is streamed and dequantised T times.  Here the unit of ownership is
// an output-dim group instead:
//
//   - a CTA owns RPW output dims d0..d0+RPW-1 for every token of the call and
//     writes each of those outputs exactly once;
//   - its 8 warps split the routed experts into contiguous ranges of equal
//     estimated cost (an expert with T tokens costs T + kDnBase); a warp
//     streams the RPW rows of each of its experts once, dequantises them once
//     (E8M0 scale folded into the FP32 weights) and applies them to every
//     (token, slot) routed to that expert, reading h directly (8 elements per
//     lane per load, lanes on consecutive octets of the row);
//   - the TC*RPW lane partials of a chunk of TC tokens are summed across the
//     warp by a transpose-reduction; the lanes holding the sums multiply by the
//     routing weight and add into the warp's row of a shared-memory table
//     y[warp][b][r] (one lane per entry, warps in a fixed expert order);
//   - after a barrier the CTA adds the 8 warps' tables in warp order and stores
//     BF16.  Every sum is FP32, on chip, in an order fixed by the routing.
#include "wd_device.cuh"
#include "wd_launch.h"
#include "wd_pipeline.cuh"
#include "wd_routing.cuh"

namespace wd {

namespace {

constexpr int kDnWarps = 8;
constexpr int kDnThreads = 32 * kDnWarps;
constexpr int kDnBase = 2;          // expert cost = T + kDnBase
constexpr int kDnMaxB = 256;        // table rows (tokens)

__host__ __device__ inline int dn_table_offset() { return (routing_table_bytes() + 127) / 128 * 128; }

template <int RPW>
__host__ __device__ inline int dn_smem_bytes(int B) {
  return dn_table_offset() + kDnWarps * B * RPW * 4;
}

__device__ __forceinline__ uint2 ld_weights_8B(const void* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_act_16B(const void* p) {
  uint4 r;
  asm("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Warp sum of V values per lane by transpose-reduction (V a power of two,
// 2 <= V <= 32): lane l ends with the sum of value index l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float dn_transpose_reduce(float (&v)[V]) {
  constexpr int L = V == 2 ? 1 : (V == 4 ? 2 : (V == 8 ? 3 : (V == 16 ? 4 : 5)));
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < L; ++k) {
    const int off = 16 >> k;
    const int n = V >> k;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
  float s = v[0];
#pragma unroll
  for (int off = 16 >> L; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  return s;
}

// One chunk of TC (<= 4) (token, slot) pairs of one expert for this warp's RPW
// rows; adds w * dot into the warp's table rows of those tokens.
template <int RPW, int TC>
__device__ __forceinline__ void dn_chunk(const uint8_t* __restrict__ wrow0,
                                         const uint8_t* __restrict__ srow0,
                                         const uint8_t* __restrict__ hb,
                                         const float* __restrict__ topk_w,
                                         const int* __restrict__ slots, float* __restrict__ ytab,
                                         int I, int K) {
  constexpr int TCP = TC == 3 ? 4 : TC;
  const int lane = threadIdx.x & 31;
  const int noct = I >> 3;  // 8-element octets per row
  const int ib = I >> 5;
  float2 acc[TCP][RPW];
#pragma unroll
  for (int t = 0; t < TCP; ++t)
#pragma unroll
    for (int r = 0; r < RPW; ++r) acc[t][r] = make_float2(0.f, 0.f);
  uint32_t hoff[TC];
#pragma unroll
  for (int t = 0; t < TC; ++t) hoff[t] = (uint32_t)slots[t] * (uint32_t)I * 2u;

  for (int o = lane; o < noct; o += 32) {
    float2 wf[RPW][4];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const uint2 q = ld_weights_8B(wrow0 + (size_t)r * I + o * 8);
      const float s = e8m0_to_f32(ld_scale(srow0 + (size_t)r * ib + (o >> 2)));
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
      const uint4 hv = ld_act_16B(hb + hoff[t] + (uint32_t)o * 16u);
      const float2 h0 = bf16x2_to_f32(hv.x), h1 = bf16x2_to_f32(hv.y);
      const float2 h2 = bf16x2_to_f32(hv.z), h3 = bf16x2_to_f32(hv.w);
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        acc[t][r] = __ffma2_rn(wf[r][0], h0, acc[t][r]);
        acc[t][r] = __ffma2_rn(wf[r][1], h1, acc[t][r]);
        acc[t][r] = __ffma2_rn(wf[r][2], h2, acc[t][r]);
        acc[t][r] = __ffma2_rn(wf[r][3], h3, acc[t][r]);
      }
    }
  }

  constexpr int V = TCP * RPW;
  constexpr int L = V == 2 ? 1 : (V == 4 ? 2 : (V == 8 ? 3 : (V == 16 ? 4 : 5)));
  float v[V];
#pragma unroll
  for (int t = 0; t < TCP; ++t)
#pragma unroll
    for (int r = 0; r < RPW; ++r) v[t * RPW + r] = acc[t][r].x + acc[t][r].y;
  const float sum = dn_transpose_reduce<V>(v);
  const int idx = lane >> (5 - L);
  const int t = idx / RPW, r = idx - t * RPW;
  const bool holder = (lane & ((1 << (5 - L)) - 1)) == 0;
  // one token of the chunk at a time: two slots of one token (a repeated
  // expert id) update the same table entry
#pragma unroll
  for (int tt = 0; tt < TC; ++tt) {
    if (holder && t == tt) {
      const int s = slots[t];
      const int b = s / K;
      ytab[b * RPW + r] = fmaf(__ldg(topk_w + s), sum, ytab[b * RPW + r]);
    }
    __syncwarp();
  }
}

}  // namespace

template <int RPW>
__global__ void __launch_bounds__(kDnThreads, 2) moe_down_shared(
    const __nv_bfloat16* __restrict__ h, const int32_t* __restrict__ topk_ids,
    const float* __restrict__ topk_w, const uint8_t* __restrict__ down,
    const uint8_t* __restrict__ down_scale, __nv_bfloat16* __restrict__ out,
    uint32_t* __restrict__ error_flag, int B, int H, int I, int E, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  float* ytab_all = reinterpret_cast<float*>(smem + dn_table_offset());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BK = B * K;
  const int d0 = blockIdx.x * RPW;
  grid_launch_dependents();

  // the routing comes from before the first kernel: read it before waiting
  build_routing_tables(rt, topk_ids, BK, E, 4, kDnThreads);
  for (int i = tid; i < kDnWarps * B * RPW; i += kDnThreads) ytab_all[i] = 0.0f;
  if (rt.scalar[2] && blockIdx.x == 0 && tid == 0 && error_flag) atomicOr(error_flag, 1u);

  // this warp's experts: contiguous range of equal estimated cost
  const int U = rt.scalar[0];
  int* pc = rt.coff;  // [U + 1] cost prefix (coff is not used by this kernel)
  if (warp == 0) {
    int base = 0;
    for (int u0 = 0; u0 < U; u0 += 32) {
      const int u = u0 + lane;
      const int c = u < U ? rt.off[u + 1] - rt.off[u] + kDnBase : 0;
      int excl, total;
      warp_exclusive_scan(c, excl, total);
      if (u < U) pc[u] = base + excl;
      base += total;
    }
    if (lane == 0) pc[U] = base;
  }
  __syncthreads();
  const long long total = pc[U];
  const int lo = (int)(total * warp / kDnWarps);
  const int hi = (int)(total * (warp + 1) / kDnWarps);
  // experts u whose cost start pc[u] lies in [lo, hi)
  int u_begin = 0;
  while (u_begin < U && pc[u_begin] < lo) ++u_begin;
  int u_end = u_begin;
  while (u_end < U && pc[u_end] < hi) ++u_end;

  const int ib = I >> 5;
  if (lane == 0 && u_begin < u_end) {
    const size_t row0 = (size_t)rt.expert[u_begin] * H + d0;
    prefetch_l2_bulk(down + row0 * I, (uint32_t)(RPW * I));
    prefetch_l2_bulk(down_scale + row0 * ib, (uint32_t)(RPW * ib));
  }

  // h is written by the first kernel
  const uint32_t wait_token = grid_dependency_wait();
  const uint8_t* hb = reinterpret_cast<const uint8_t*>(h) + wait_token;
  float* ytab = ytab_all + warp * B * RPW;

  for (int u = u_begin; u < u_end; ++u) {
    if (lane == 0 && u + 1 < u_end) {
      const size_t nrow0 = (size_t)rt.expert[u + 1] * H + d0;
      prefetch_l2_bulk(down + nrow0 * I, (uint32_t)(RPW * I));
      prefetch_l2_bulk(down_scale + nrow0 * ib, (uint32_t)(RPW * ib));
    }
    const size_t row0 = (size_t)rt.expert[u] * H + d0;
    const uint8_t* wrow0 = down + row0 * I;
    const uint8_t* srow0 = down_scale + row0 * ib;
    const int first = rt.off[u];
    const int T = rt.off[u + 1] - first;
    for (int c0 = 0; c0 < T; c0 += 4) {
      const int tc = min(4, T - c0);
      const int* sl = rt.slots + first + c0;
      if (tc == 4)
        dn_chunk<RPW, 4>(wrow0, srow0, hb, topk_w, sl, ytab, I, K);
      else if (tc == 3)
        dn_chunk<RPW, 3>(wrow0, srow0, hb, topk_w, sl, ytab, I, K);
      else if (tc == 2)
        dn_chunk<RPW, 2>(wrow0, srow0, hb, topk_w, sl, ytab, I, K);
      else
        dn_chunk<RPW, 1>(wrow0, srow0, hb, topk_w, sl, ytab, I, K);
      __syncwarp();
    }
  }
  __syncthreads();

  // sum the warps' tables in warp order; one BF16 store per output
  for (int i = tid; i < B * RPW; i += kDnThreads) {
    float y = 0.0f;
#pragma unroll
    for (int w = 0; w < kDnWarps; ++w) y += ytab_all[w * B * RPW + i];
    const int b = i / RPW, r = i - b * RPW;
    out[(size_t)b * H + d0 + r] = __float2bfloat16_rn(y);
  }
}

bool down_shared_supported(int B, int H, int I, int E, int K, int rpw) {
  (void)I;
  return (rpw == 2 || rpw == 4) && B * K <= kStreamMaxSlots && B <= kDnMaxB && E <= 4096 &&
         H % rpw == 0;
}

template <int RPW>
static cudaError_t launch_down_shared_t(const DownArgs& a, cudaStream_t stream, bool pdl) {
  const int smem = dn_smem_bytes<RPW>(a.B);
  static int configured = 0;
  if (configured < smem) {
    const cudaError_t e = cudaFuncSetAttribute(moe_down_shared<RPW>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.H / RPW));
  cfg.blockDim = dim3(kDnThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_shared<RPW>,
                            reinterpret_cast<const __nv_bfloat16*>(a.h), a.topk_ids, a.topk_w,
                            a.down, a.down_scale, reinterpret_cast<__nv_bfloat16*>(a.out),
                            a.error_flag, a.B, a.H, a.I, a.E, a.K);
}

cudaError_t launch_down_shared(const DownArgs& a, const DownPlan& p, cudaStream_t stream,
                               bool pdl) {
  if (!down_shared_supported(a.B, a.H, a.I, a.E, a.K, p.rpw)) return cudaErrorInvalidValue;
  if (p.rpw == 4) return launch_down_shared_t<4>(a, stream, pdl);
  return launch_down_shared_t<2>(a, stream, pdl);
}

}  // namespace wd
