// wd_down_stream.cu - moe_down_stream: the down kernel with its weight rows and
// activations streamed through a shared-memory ring by bulk async copies.
//
// Computes exactly what moe_down_3d_batched computes (Cursor, "用 warp decode
// 实现更好的 MoE 模型推理", section 两个 kernel 如何工作, down paragraph):
// out[b,d] = bf16( sum_k w[b,k] * (down[e_k][d,:] . h[b,k,:]) ), every routed
// expert's weighted contribution folded into ONE FP32 register accumulator per
// output, lane partials reduced with __shfl_xor_sync, one store per output.
//
// GB300 mapping (B <= 32):
//   - a CTA owns 8 consecutive output dims d0..d0+7 for all tokens; each of its
//     8 consumer warps owns one of them, and lane b of that warp holds the
//     accumulator of token b;
//   - one producer thread streams, per stage, the 8 contiguous down rows
//     e*H+d0.. of one routed expert e, their scales, and the h rows of up to 8
//     (token, slot) pairs routed to e, with cp.async.bulk into a ring of
//     shared-memory stages.  The weight rows do not depend on the gate/up
//     kernel, so the first stages' rows are requested before the programmatic-
//     dependent-launch wait and only the h rows after it;
//   - a warp dequantises its row once per stage, dots it with each staged h
//     row (shared memory only), reduces the 8 slot partials across the warp in
//     one recursive-halving pass (9 shuffles instead of 8 butterflies), and
//     lane b adds w[b,k] times its token's sums to its accumulator.
#include "wd_device.cuh"
#include "wd_launch.h"
#include "wd_pipeline.cuh"
#include "wd_routing.cuh"

namespace wd {

namespace {

constexpr int kDnConsumers = 8;  // consumer warps per CTA, one output dim each
constexpr int kDnThreads = 32 * (kDnConsumers + 1);
constexpr int kDnNd = kDnConsumers;  // output dims per CTA
constexpr int kDnSlots = 8;          // (token, slot) h rows per stage

struct DownLayout {
  int nst, stage_bytes, routing_off, stage_off, total;
};

__host__ __device__ inline int dn_round_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline DownLayout down_layout(int I, int nst) {
  DownLayout L;
  L.nst = nst;
  L.stage_bytes = dn_round_up(kDnNd * I + kDnNd * (I / 32) + kDnSlots * I * 2, 128);
  L.routing_off = dn_round_up(2 * nst * 8, 128);
  L.stage_off = dn_round_up(L.routing_off + routing_table_bytes(), 1024);
  L.total = L.stage_off + nst * L.stage_bytes;
  return L;
}

// Sum each of 8 per-lane values over the 32 lanes in one pass: after it, lane
// 4j holds the total of value j (and lanes 4j+1..4j+3 hold it too).
__device__ __forceinline__ float reduce8_to_lane4j(float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  bool hi = (lane & 16) != 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = hi ? v[i + 4] : v[i], send = hi ? v[i] : v[i + 4];
    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
  }
  hi = (lane & 8) != 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = hi ? v[i + 2] : v[i], send = hi ? v[i] : v[i + 2];
    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
  }
  hi = (lane & 4) != 0;
  {
    const float keep = hi ? v[1] : v[0], send = hi ? v[0] : v[1];
    v[0] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
  }
  v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 2);
  v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
  return v[0];
}

}  // namespace

template <int NS>
__global__ void __launch_bounds__(kDnThreads, 2) moe_down_stream(
    const __nv_bfloat16* __restrict__ h, const int32_t* __restrict__ topk_ids,
    const float* __restrict__ topk_w, const uint8_t* __restrict__ down,
    const uint8_t* __restrict__ down_scale, __nv_bfloat16* __restrict__ out,
    uint32_t* __restrict__ error_flag, int B, int H, int I, int E, int K, int nst) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const DownLayout L = down_layout(I, nst);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  const RoutingTables rt = routing_tables_at(smem + L.routing_off);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BK = B * K;
  const int d0 = blockIdx.x * kDnNd;
  const int ib = I >> 5;
  const uint32_t row_bytes = (uint32_t)(kDnNd * I), sc_bytes = (uint32_t)(kDnNd * ib);

  grid_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[nst + s]), kDnConsumers);
    }
    mbar_init_fence();
  }
  // The routing is an input of the call (complete before the gate/up kernel
  // started), so it is read before waiting on that kernel.
  build_routing_tables(rt, topk_ids, BK, E, kDnSlots, kDnThreads);
  const int nq = rt.scalar[1];  // chunks of <= kDnSlots slots, one stage each
  if (rt.scalar[2] && blockIdx.x == 0 && tid == 0 && error_flag) atomicOr(error_flag, 1u);

  if (warp == kDnConsumers) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    const uint64_t pol_w = l2_evict_first_policy();
    const uint64_t pol_h = l2_evict_last_policy();
    const uint8_t* hb = reinterpret_cast<const uint8_t*>(h);
    auto chunk = [&](int q, int& first, int& tc) {
      const int u = rt.chunk_u[q];
      first = rt.off[u] + (q - rt.coff[u]) * kDnSlots;
      tc = min(kDnSlots, rt.off[u + 1] - first);
      return u;
    };
    auto issue_weights = [&](int q, int st, int tc, int u) {
      const uint32_t full = smem_u32(&bars[st]);
      const size_t row0 = (size_t)rt.expert[u] * H + d0;
      const uint32_t sbuf = smem_u32(smem + L.stage_off + st * L.stage_bytes);
      mbar_arrive_expect_tx(full, row_bytes + sc_bytes + (uint32_t)(tc * I * 2));
      bulk_g2s(sbuf, down + row0 * I, row_bytes, full, pol_w);
      bulk_g2s(sbuf + row_bytes, down_scale + row0 * ib, sc_bytes, full, pol_w);
    };
    auto issue_h = [&](int st, int first, int tc) {
      const uint32_t full = smem_u32(&bars[st]);
      const uint32_t hs = smem_u32(smem + L.stage_off + st * L.stage_bytes) + row_bytes + sc_bytes;
      for (int t = 0; t < tc; ++t)
        bulk_g2s(hs + t * I * 2, hb + (size_t)rt.slots[first + t] * I * 2, I * 2, full, pol_h);
    };
    // the first stages: weight rows now, h rows once the gate/up kernel is done
    const int pre = min(nst, nq);
    for (int q = 0; q < pre; ++q) {
      int first, tc;
      const int u = chunk(q, first, tc);
      issue_weights(q, q, tc, u);
    }
    grid_dependency_wait();
    for (int q = 0; q < pre; ++q) {
      int first, tc;
      chunk(q, first, tc);
      issue_h(q, first, tc);
    }
    for (int q = pre; q < nq; ++q) {
      const int st = q % nst;
      if (!mbar_wait(smem_u32(&bars[nst + st]), ((q / nst) & 1) ^ 1)) {
        if (error_flag) atomicOr(error_flag, 2u);
        for (int k = q - nst; k < q; ++k) (void)mbar_wait(smem_u32(&bars[k % nst]), (k / nst) & 1);
        return;
      }
      int first, tc;
      const int u = chunk(q, first, tc);
      issue_weights(q, st, tc, u);
      issue_h(st, first, tc);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  float acc = 0.0f;  // lane b: out[b, d0 + warp]
  for (int q = 0; q < nq; ++q) {
    const int st = q % nst;
    if (!mbar_wait(smem_u32(&bars[st]), (q / nst) & 1)) {
      if (error_flag && lane == 0) atomicOr(error_flag, 2u);
      return;
    }
    const int u = rt.chunk_u[q];
    const int first = rt.off[u] + (q - rt.coff[u]) * kDnSlots;
    const int tc = min(kDnSlots, rt.off[u + 1] - first);
    const uint32_t sbuf = smem_u32(smem + L.stage_off + st * L.stage_bytes);
    const uint32_t hs = sbuf + row_bytes + sc_bytes;

    float2 wf[NS][4];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int c = 8 * (lane + 32 * i);
      if (c < I) {
        const uint2 qv = lds_u32x2(sbuf + warp * I + c);
        const float s = e8m0_to_f32(lds_u8(sbuf + row_bytes + warp * ib + (c >> 5)));
        const float2 s2 = make_float2(s, s);
        float2 lo, hi;
        e4m3x4_to_f32(qv.x, lo, hi);
        wf[i][0] = __fmul2_rn(lo, s2);
        wf[i][1] = __fmul2_rn(hi, s2);
        e4m3x4_to_f32(qv.y, lo, hi);
        wf[i][2] = __fmul2_rn(lo, s2);
        wf[i][3] = __fmul2_rn(hi, s2);
      }
    }
    float p[kDnSlots];
#pragma unroll
    for (int t = 0; t < kDnSlots; ++t) {
      p[t] = 0.0f;
      if (t < tc) {
        float2 pp = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          const int c = 8 * (lane + 32 * i);
          if (c < I) {
            uint4 hv;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(hv.x), "=r"(hv.y), "=r"(hv.z), "=r"(hv.w)
                         : "r"(hs + (uint32_t)(t * I + c) * 2u));
            pp = __ffma2_rn(wf[i][0], bf16x2_to_f32(hv.x), pp);
            pp = __ffma2_rn(wf[i][1], bf16x2_to_f32(hv.y), pp);
            pp = __ffma2_rn(wf[i][2], bf16x2_to_f32(hv.z), pp);
            pp = __ffma2_rn(wf[i][3], bf16x2_to_f32(hv.w), pp);
          }
        }
        p[t] = pp.x + pp.y;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[nst + st]));  // stage fully read

    const float total = reduce8_to_lane4j(p);
#pragma unroll
    for (int t = 0; t < kDnSlots; ++t) {
      if (t < tc) {
        const float v = __shfl_sync(0xFFFFFFFFu, total, 4 * t);
        const int s = rt.slots[first + t];
        if (lane == s / K) acc = fmaf(__ldg(topk_w + s), v, acc);
      }
    }
  }
  if (lane < B) out[(size_t)lane * H + d0 + warp] = __float2bfloat16_rn(acc);
}

bool down_stream_supported(int B, int H, int I, int E, int K) {
  return B <= 32 && B * K <= kStreamMaxSlots && E <= 4096 && I % 64 == 0 && I <= 1024 &&
         H % kDnNd == 0;
}

template <int NS>
static cudaError_t launch_down_stream_t(const DownArgs& a, int nst, cudaStream_t stream, bool pdl) {
  const DownLayout L = down_layout(a.I, nst);
  static int configured_bytes[5] = {0, 0, 0, 0, 0};
  if (configured_bytes[NS] < L.total) {
    const cudaError_t e = cudaFuncSetAttribute(moe_down_stream<NS>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    configured_bytes[NS] = L.total;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.H / kDnNd));
  cfg.blockDim = dim3(kDnThreads);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_stream<NS>, reinterpret_cast<const __nv_bfloat16*>(a.h),
                            a.topk_ids, a.topk_w, a.down, a.down_scale,
                            reinterpret_cast<__nv_bfloat16*>(a.out), a.error_flag, a.B, a.H, a.I,
                            a.E, a.K, nst);
}

cudaError_t launch_down_stream(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl) {
  if (!down_stream_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  int nst = p.qpl > 0 ? p.qpl : 4;
  while (nst > 2 && down_layout(a.I, nst).total > 227 * 1024) --nst;  // fit one CTA's smem
  switch ((a.I + 255) / 256) {
    case 1: return launch_down_stream_t<1>(a, nst, stream, pdl);
    case 2: return launch_down_stream_t<2>(a, nst, stream, pdl);
    case 3: return launch_down_stream_t<3>(a, nst, stream, pdl);
    case 4: return launch_down_stream_t<4>(a, nst, stream, pdl);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace wd
