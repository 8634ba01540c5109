// wd_gate_up_ring.cu - moe_gate_up_ring: moe_gate_up_persist with each warp's
// weight rows streamed through its own shared-memory ring by bulk copies.
//
// Same outputs and the same organisation as moe_gate_up_persist (Cursor, "用
// warp decode 实现更好的 MoE 模型推理", section 两个 kernel 如何工作, gate/up
// paragraph, re-organised so that every token routed to an expert is served
// from one read of its rows): persistent CTAs, routing tables built once,
// cost-balanced contiguous (expert, 16-neuron block) items, the expert's
// tokens' x staged as swizzled FP32, block scales on 32-element partials, a
// transpose-reduction epilogue.
//
// What changes is how weight bytes reach a warp.  In moe_gate_up_persist each
// lane loads its 32-byte blocks into registers and waits for them before it
// computes, so a warp has 4 KiB in flight only between its compute phases.
// Here a warp's work is a sequence of steps, one step = the 32 blocks (one per
// lane) of the warp's 4 rows = 4 x 1 KiB of codes + 4 x 32 scale bytes.  Lane 0
// issues each step as 8 cp.async.bulk copies into a stage of the warp's S-stage
// ring, completing on that stage's mbarrier, S steps ahead of the step the
// warp computes; the lanes read their block from shared memory.  The bytes in
// flight are therefore held by shared memory, not registers, and never stop
// while the warp computes.  Each warp is its own producer and consumer: after
// computing a step the warp synchronises and lane 0 refills the same stage.
//
// Every mbarrier wait is bounded (wd_pipeline.cuh).  A warp whose wait runs out
// raises bit 1 of the error flag, stops issuing, computes nothing more and
// only follows the CTA's barriers; at the end it waits (bounded) for the copies
// it had issued, so none is in flight when the CTA exits.
#include "wd_launch.h"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kRItemBase = 3;       // item cost = T + kRItemBase
constexpr int kRStep = 1024;        // bytes of one row per step (32 blocks)
constexpr int kRStageBytes = 4 * kRStep + 4 * 32;  // 4 rows of codes + their scale bytes
constexpr int kRXMaxTokens = 4;     // x rows staged at once (upper bound)
constexpr int kRXBudget = 32 * 1024;
static_assert(kRStageBytes % 128 == 0, "stage alignment");

__host__ __device__ inline int ring_x_tokens(int H) {
  const int t = kRXBudget / (H * 4);
  return t < 1 ? 1 : (t > kRXMaxTokens ? kRXMaxTokens : t);
}

__host__ __device__ inline int ring_offset(int H) {
  return (kXOffset + ring_x_tokens(H) * H * 4 + 127) / 128 * 128;
}

__host__ __device__ inline int ring_smem_bytes(int H, int S) {
  return ring_offset(H) + kPWarps * S * (kRStageBytes + 8);
}

// Bulk copy without an L2 cache hint (rows re-read by a later token group
// should stay in L2 like any other line).
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Position of a warp in its sequence of steps within one (expert, token group):
// item g (neuron block), token chunk c0, block step bs.
struct StepPos {
  int g, c0, bs;
};

__device__ __forceinline__ void step_advance(StepPos& p, int nsteps, int nq) {
  if (++p.bs == nsteps) {
    p.bs = 0;
    p.c0 += 4;
    if (p.c0 >= nq) {
      p.c0 = 0;
      ++p.g;
    }
  }
}

// Lane 0: copy step `p` of this warp's rows into ring stage `slot`.
__device__ __forceinline__ void issue_step(const StepPos& p, uint32_t stage, uint32_t bar,
                                           const uint8_t* __restrict__ gate_up,
                                           const uint8_t* __restrict__ gate_up_scale,
                                           size_t expert_row0, int warp, int H, int I) {
  const int nblk = H >> 5;
  const size_t gate_row0 = expert_row0 + (size_t)(p.g * kPWarps + warp) * 2;
  mbar_arrive_expect_tx(bar, (uint32_t)kRStageBytes);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const size_t row = gate_row0 + (r >> 1) * (size_t)I + (r & 1);
    bulk_g2s_plain(stage + r * kRStep, gate_up + row * H + (size_t)p.bs * kRStep, kRStep, bar);
    bulk_g2s_plain(stage + 4 * kRStep + r * 32, gate_up_scale + row * nblk + (size_t)p.bs * 32, 32,
                   bar);
  }
}

// One step of one chunk of TC tokens: lane's block blk = bs*32 + lane of the 4
// staged rows, against staged x of tokens t0..t0+TC-1, into acc.
template <int TC, int TCP>
__device__ __forceinline__ void ring_step(uint32_t stage, uint32_t xs, int t0, int bs, int H,
                                          float (&acc)[TCP][4]) {
  const int lane = threadIdx.x & 31;
  const int blk = bs * 32 + lane;
  // Lanes of odd quads read the two 16-byte halves of their 32 bytes in the
  // other order, so the 8 lanes of a quarter-warp hit 8 different bank groups;
  // register word m then holds physical word m ^ 4q.
  const int q = (lane >> 2) & 1;
  uint32_t w[4][8];
  float sc[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t rb = stage + r * kRStep + lane * 32;
    const uint4 a = lds_u32x4(rb + 16 * q);
    const uint4 b = lds_u32x4(rb + 16 * (1 - q));
    w[r][0] = a.x; w[r][1] = a.y; w[r][2] = a.z; w[r][3] = a.w;
    w[r][4] = b.x; w[r][5] = b.y; w[r][6] = b.z; w[r][7] = b.w;
    sc[r] = e8m0_to_f32(lds_u8(stage + 4 * kRStep + r * 32 + lane));
  }
  float2 p[TC][4];
#pragma unroll
  for (int t = 0; t < TC; ++t)
#pragma unroll
    for (int r = 0; r < 4; ++r) p[t][r] = make_float2(0.f, 0.f);
  const uint32_t xb = xs + (uint32_t)(t0 * H + blk * 32) * 4u;
  const int swq = (blk & 3) ^ (4 * q);  // x staged with swizzle mask 3 (xs_chunk)
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float2 wf[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) e4m3x4_to_f32(w[r][m], wf[r][0], wf[r][1]);
    const uint32_t xc = xb + (uint32_t)((m ^ swq) << 4);
#pragma unroll
    for (int t = 0; t < TC; ++t) {
      const float4 xv = lds_f32x4(xc + (uint32_t)(t * H * 4));
      const float2 x01 = make_float2(xv.x, xv.y), x23 = make_float2(xv.z, xv.w);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        p[t][r] = __ffma2_rn(wf[r][0], x01, p[t][r]);
        p[t][r] = __ffma2_rn(wf[r][1], x23, p[t][r]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TC; ++t)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[t][r] = fmaf(p[t][r].x + p[t][r].y, sc[r], acc[t][r]);
}

// Per-warp ring state (all lanes hold the same values).
struct Ring {
  uint32_t stages;  // shared address of stage 0
  uint32_t bars;    // shared address of the S mbarriers
  uint32_t consumed, issued;
  uint32_t dead_from, dead_to;  // copies left in flight when a wait ran out
  bool dead;
};

// One chunk of TC tokens of the current item: its steps, then the epilogue.
template <int S, int TC>
__device__ __forceinline__ void ring_chunk(Ring& ring, StepPos& pp, int g1, int nsteps, int nq,
                                           uint32_t xs, int t0, const int* slots, int n0,
                                           __nv_bfloat16* __restrict__ h,
                                           const uint8_t* __restrict__ gate_up,
                                           const uint8_t* __restrict__ gate_up_scale,
                                           size_t expert_row0, uint32_t* error_flag, int H,
                                           int I) {
  constexpr int TCP = TC == 3 ? 4 : TC;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[TCP][4];
#pragma unroll
  for (int t = 0; t < TCP; ++t)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[t][r] = 0.0f;
  for (int bs = 0; bs < nsteps; ++bs) {
    const uint32_t s = ring.consumed % S;
    const uint32_t stage = ring.stages + s * kRStageBytes;
    if (!ring.dead) {
      if (!mbar_wait(ring.bars + 8 * s, (ring.consumed / S) & 1)) {
        ring.dead = true;
        ring.dead_from = ring.consumed;  // this step's copies have not been seen to land
        ring.dead_to = ring.issued;
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
      }
    }
    if (!ring.dead) ring_step<TC, TCP>(stage, xs, t0, bs, H, acc);
    __syncwarp();  // every lane is done with the stage before it is refilled
    ++ring.consumed;
    if (!ring.dead && pp.g < g1) {
      if (lane == 0)
        issue_step(pp, stage, ring.bars + 8 * s, gate_up, gate_up_scale, expert_row0, warp, H, I);
      ++ring.issued;
      step_advance(pp, nsteps, nq);
    }
  }
  if (!ring.dead) store_chunk<2, TC, TCP>(acc, h, slots, n0, I);
}

}  // namespace

template <int S>
__global__ void __launch_bounds__(kPThreads, 2) moe_gate_up_ring(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const uint8_t* __restrict__ gate_up, const uint8_t* __restrict__ gate_up_scale,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K) {
  extern __shared__ __align__(128) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const uint32_t xs = smem_u32(smem + kXOffset);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K;
  const int xtok = ring_x_tokens(H);
  const int nsteps = H / kRStep;

  Ring ring;
  ring.stages = smem_u32(smem + ring_offset(H)) + warp * S * kRStageBytes;
  ring.bars = smem_u32(smem + ring_offset(H) + kPWarps * S * kRStageBytes) + warp * S * 8;
  ring.consumed = ring.issued = ring.dead_from = ring.dead_to = 0;
  ring.dead = false;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(ring.bars + 8 * s, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // x and topk_ids may come from the kernel before this one on the stream.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();
  build_routing_tables(rt, topk_ids, BK, E, 4, kPThreads);
  zero_bad_slots(rt, h, error_flag, BK, I, E);

  const int U = rt.scalar[0];
  const int nb = I / 16;  // items per expert (I % 16 == 0 here)
  int* pc = rt.coff;
  expert_cost_prefix(rt, nb, kRItemBase, pc);
  const long long total = pc[U];
  const int lo = (int)(total * blockIdx.x / gridDim.x);
  const int hi = (int)(total * (blockIdx.x + 1) / gridDim.x);

  if (lo < hi) {
    const uint8_t* xg = reinterpret_cast<const uint8_t*>(x) + wait_token;
    for (int u = first_expert(pc, U, lo); u < U && pc[u] < hi; ++u) {
      const int T = rt.off[u + 1] - rt.off[u];
      const int cu = T + kRItemBase;
      const int g0 = pc[u] >= lo ? 0 : (lo - pc[u] + cu - 1) / cu;
      const int g1 = min(nb, (hi - pc[u] + cu - 1) / cu);
      if (g0 >= g1) continue;
      const int* slots = rt.slots + rt.off[u];
      const size_t expert_row0 = (size_t)rt.expert[u] * 2 * I;
      for (int q0 = 0; q0 < T; q0 += xtok) {
        const int nq = min(xtok, T - q0);
        // the first S steps of this group go out before x is staged
        StepPos pp{g0, 0, 0};
        for (int k = 0; k < S && pp.g < g1 && !ring.dead; ++k) {
          const uint32_t s = ring.issued % S;
          if (lane == 0)
            issue_step(pp, ring.stages + s * kRStageBytes, ring.bars + 8 * s, gate_up,
                       gate_up_scale, expert_row0, warp, H, I);
          ++ring.issued;
          step_advance(pp, nsteps, nq);
        }
        stage_x(xs, xg, slots + q0, nq, H, K, 3);
        for (int g = g0; g < g1; ++g) {
          const int n0 = (g * kPWarps + warp) * 2;
          for (int c0 = 0; c0 < nq; c0 += 4) {
            const int tc = min(4, nq - c0);
            const int* sl = slots + q0 + c0;
#define WD_RING_CHUNK(TCV)                                                                    \
  ring_chunk<S, TCV>(ring, pp, g1, nsteps, nq, xs, c0, sl, n0, h, gate_up, gate_up_scale, \
                     expert_row0, error_flag, H, I)
            if (tc == 4) WD_RING_CHUNK(4);
            else if (tc == 3) WD_RING_CHUNK(3);
            else if (tc == 2) WD_RING_CHUNK(2);
            else WD_RING_CHUNK(1);
#undef WD_RING_CHUNK
          }
        }
      }
    }
  }
  // a warp whose wait ran out lets the copies it had issued land before exiting
  if (ring.dead)
    for (uint32_t k = ring.dead_from; k < ring.dead_to; ++k)
      (void)mbar_wait(ring.bars + 8 * (k % S), (k / S) & 1);
}

bool gate_up_ring_supported(int B, int H, int I, int E, int K, int stages) {
  return (stages == 2 || stages == 3) && B * K <= kStreamMaxSlots && E <= 4096 &&
         H % kRStep == 0 && I % 16 == 0 && ring_smem_bytes(H, stages) <= 113 * 1024;
}

template <int S>
static cudaError_t launch_ring_t(const GateUpArgs& a, cudaStream_t stream, bool pdl) {
  const int smem = ring_smem_bytes(a.H, S);
  static int configured = 0;
  if (configured < smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(moe_gate_up_ring<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_gate_up_ring<S>, kPThreads, smem);
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
  return cudaLaunchKernelEx(&cfg, moe_gate_up_ring<S>, reinterpret_cast<const __nv_bfloat16*>(a.x),
                            a.topk_ids, a.gate_up, a.gate_up_scale,
                            reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag, a.B, a.H, a.I,
                            a.E, a.K);
}

// p.npw = ring stages per warp (2 or 3).
cudaError_t launch_gate_up_ring(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                bool pdl) {
  if (!gate_up_ring_supported(a.B, a.H, a.I, a.E, a.K, p.npw)) return cudaErrorInvalidValue;
  if (p.npw == 3) return launch_ring_t<3>(a, stream, pdl);
  return launch_ring_t<2>(a, stream, pdl);
}

}  // namespace wd
