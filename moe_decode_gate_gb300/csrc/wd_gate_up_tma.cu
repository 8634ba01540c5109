// wd_gate_up_tma.cu - moe_gate_up_tma: the shared-row gate/up kernel fed by
// tensor-memory-accelerator copies into a CTA-wide shared-memory ring.
//
// Same outputs as moe_gate_up_3d_batched (Cursor, "用 warp decode 实现更好的
// MoE 模型推理", section 两个 kernel 如何工作, gate/up paragraph): every
// h[b,k,n] = bf16(SiLU(g) * u) from gate row n and up row I+n of the routed
// expert, produced by exactly one warp, with no padding, gather or combine.
// It is organised like moe_gate_up_persist (a warp owns 2 neurons of one
// routed expert for all tokens routed to it; persistent CTAs walk
// cost-balanced contiguous (expert, neuron block) items; the expert's tokens'
// x is staged once as swizzled FP32; block scales multiply 32-element
// partials; transpose-reduction epilogue) but the weight bytes arrive
// differently:
//
//   - one CTA per SM: 12 consumer warps (24 neurons per item) and one producer
//     lane;
//   - a step is one 1024-column slab of the item's 48 rows (24 gate rows, 24
//     up rows, each group contiguous in [E][2I][H]) plus their 32 scale bytes
//     per row: 8 two-dimensional TMA boxes of 256 B x 24 rows and 2 boxes of
//     32 B x 24 rows, 50,688 bytes, landing in one stage of a 3-stage ring
//     and completing on the stage's "full" mbarrier;
//   - the producer refills a stage as soon as all 12 consumer warps have
//     arrived on its "empty" mbarrier, so up to 3 steps (~150 KB) are in
//     flight or resident per SM at any time, independent of registers.
//
// Shared memory per CTA (H = 2048): routing tables 8.3 KB, staged x 64 KB,
// ring 150 KB.  Every mbarrier wait is bounded (wd_pipeline.cuh); a wait that
// runs out raises bit 1 of the error flag and the thread stops computing but
// keeps arriving, so no other thread waits on it forever, and a consumer that
// gave up waits (bounded) for the copies into the stage it abandoned.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "wd_launch.h"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kTWarps = 12;                   // consumer warps
constexpr int kTThreads = 32 * (kTWarps + 1);  // + producer warp
constexpr int kTConsumers = 32 * kTWarps;
constexpr int kTRows = 2 * kTWarps;           // gate (or up) rows per item
constexpr int kTBoxCols = 256;                // inner box extent (bytes)
constexpr int kTStepCols = 1024;              // columns per step (one block per lane)
constexpr int kTBoxBytes = kTBoxCols * kTRows;                   // 6144
constexpr int kTScaleBytes = 32 * kTRows;                        // 768
constexpr int kTStageData = 2 * 4 * kTBoxBytes + 2 * kTScaleBytes;  // 50,688
constexpr int kTStageStride = 51200;          // 1024-aligned stages
constexpr int kTItemBase = 3;
constexpr int kTXMaxTokens = 8;
constexpr int kTXBudget = 64 * 1024;
constexpr int kTSmemLimit = 227 * 1024;
static_assert(kTStageData <= kTStageStride && kTStageStride % 1024 == 0, "stage layout");

__host__ __device__ inline int tma_x_tokens(int H) {
  const int t = kTXBudget / (H * 4);
  return t < 1 ? 1 : (t > kTXMaxTokens ? kTXMaxTokens : t);
}
__host__ __device__ inline int tma_ring_offset(int H) {
  return (kXOffset + tma_x_tokens(H) * H * 4 + 1023) / 1024 * 1024;
}
__host__ __device__ inline int tma_smem_bytes(int H, int S) {
  return tma_ring_offset(H) + S * kTStageStride + 2 * S * 8;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// One consumer step: this warp's 4 rows (gate 2w, 2w+1; up 2w, 2w+1 of the
// item's boxes), lane's block bs*32 + lane, against staged x of TC tokens.
template <int TC, int TCP>
__device__ __forceinline__ void tma_step(uint32_t stage, uint32_t xs, int t0, int bs, int H,
                                         float (&acc)[TCP][4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int blk = bs * 32 + lane;
  // lanes of odd quads read their two 16-byte halves in the other order (the
  // 8 lanes of a quarter-warp then touch 8 different bank groups); register
  // word m holds physical word m ^ 4q
  const int q = (lane >> 2) & 1;
  uint32_t w[4][8];
  float sc[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 2 * warp + (r & 1);
    const uint32_t rb = stage + (r >> 1) * (4 * kTBoxBytes) + (lane >> 3) * kTBoxBytes +
                        row * kTBoxCols + (lane & 7) * 32;
    const uint4 a = lds_u32x4(rb + 16 * q);
    const uint4 b = lds_u32x4(rb + 16 * (1 - q));
    w[r][0] = a.x; w[r][1] = a.y; w[r][2] = a.z; w[r][3] = a.w;
    w[r][4] = b.x; w[r][5] = b.y; w[r][6] = b.z; w[r][7] = b.w;
    sc[r] = e8m0_to_f32(
        lds_u8(stage + 8 * kTBoxBytes + (r >> 1) * kTScaleBytes + row * 32 + lane));
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

// Consumer-side ring state (all lanes of a warp hold the same values).
struct TmaConsumer {
  uint32_t stages, full, empty;  // shared addresses: stage 0, full[0], empty[0]
  uint32_t step;                 // steps consumed
  bool dead;
};

template <int S, int TC>
__device__ __forceinline__ void tma_chunk(TmaConsumer& c, int nsteps, uint32_t xs, int t0,
                                          const int* slots, int n0, __nv_bfloat16* h,
                                          uint32_t* error_flag, int H, int I) {
  constexpr int TCP = TC == 3 ? 4 : TC;
  const int lane = threadIdx.x & 31;
  float acc[TCP][4];
#pragma unroll
  for (int t = 0; t < TCP; ++t)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[t][r] = 0.0f;
  for (int bs = 0; bs < nsteps; ++bs) {
    const uint32_t s = c.step % S;
    if (!c.dead && !mbar_wait(c.full + 8 * s, (c.step / S) & 1)) {
      c.dead = true;
      if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
      // let the copies into this stage land before anything else happens
      (void)mbar_wait(c.full + 8 * s, (c.step / S) & 1);
    }
    if (!c.dead && n0 < I) tma_step<TC, TCP>(c.stages + s * kTStageStride, xs, t0, bs, H, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(c.empty + 8 * s);
    ++c.step;
  }
  if (!c.dead && n0 < I) store_chunk<2, TC, TCP>(acc, h, slots, n0, I);
}

}  // namespace

template <int S>
__global__ void __maxnreg__(128) moe_gate_up_tma(
    const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I, int E,
    int K) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const uint32_t xs = smem_u32(smem + kXOffset);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K;
  const int xtok = tma_x_tokens(H);
  const int nsteps = H / kTStepCols;
  const uint32_t stages = smem_u32(smem + tma_ring_offset(H));
  const uint32_t full = stages + S * kTStageStride;
  const uint32_t empty = full + 8 * S;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, kTWarps);
    }
    mbar_init_fence();
  }
  // x and topk_ids may come from the kernel before this one on the stream.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();
  build_routing_tables(rt, topk_ids, BK, E, 4, kTThreads);  // ends with a barrier
  zero_bad_slots(rt, h, error_flag, BK, I, E);

  const int U = rt.scalar[0];
  const int nb = (I + kTRows - 1) / kTRows;  // items per expert
  int* pc = rt.coff;
  expert_cost_prefix(rt, nb, kTItemBase, pc);
  const long long total = pc[U];
  const int lo = (int)(total * blockIdx.x / gridDim.x);
  const int hi = (int)(total * (blockIdx.x + 1) / gridDim.x);
  if (lo >= hi) return;
  const int u_first = first_expert(pc, U, lo);

  if (warp == kTWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    uint32_t step = 0;
    bool dead = false;
    for (int u = u_first; u < U && pc[u] < hi && !dead; ++u) {
      const int T = rt.off[u + 1] - rt.off[u];
      const int cu = T + kTItemBase;
      const int g0 = pc[u] >= lo ? 0 : (lo - pc[u] + cu - 1) / cu;
      const int g1 = min(nb, (hi - pc[u] + cu - 1) / cu);
      const int row0 = rt.expert[u] * 2 * I;
      for (int q0 = 0; q0 < T && !dead; q0 += xtok) {
        const int nq = min(xtok, T - q0);
        for (int g = g0; g < g1 && !dead; ++g)
          for (int c0 = 0; c0 < nq && !dead; c0 += 4)
            for (int bs = 0; bs < nsteps; ++bs, ++step) {
              const uint32_t s = step % S;
              if (!mbar_wait(empty + 8 * s, ((step / S) & 1) ^ 1)) {
                dead = true;
                if (error_flag) atomicOr(error_flag, 2u);
                break;
              }
              const uint32_t st = stages + s * kTStageStride;
              const uint32_t bar = full + 8 * s;
              mbar_arrive_expect_tx(bar, (uint32_t)kTStageData);
              const int rg = row0 + g * kTRows, ru = rg + I;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                tma_load_2d(st + k * kTBoxBytes, &tmap_w, bs * kTStepCols + k * kTBoxCols, rg, bar);
                tma_load_2d(st + (4 + k) * kTBoxBytes, &tmap_w, bs * kTStepCols + k * kTBoxCols,
                            ru, bar);
              }
              tma_load_2d(st + 8 * kTBoxBytes, &tmap_s, bs * 32, rg, bar);
              tma_load_2d(st + 8 * kTBoxBytes + kTScaleBytes, &tmap_s, bs * 32, ru, bar);
            }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  TmaConsumer c{stages, full, empty, 0u, false};
  const uint8_t* xg = reinterpret_cast<const uint8_t*>(x) + wait_token;
  for (int u = u_first; u < U && pc[u] < hi; ++u) {
    const int T = rt.off[u + 1] - rt.off[u];
    const int cu = T + kTItemBase;
    const int g0 = pc[u] >= lo ? 0 : (lo - pc[u] + cu - 1) / cu;
    const int g1 = min(nb, (hi - pc[u] + cu - 1) / cu);
    const int* slots = rt.slots + rt.off[u];
    for (int q0 = 0; q0 < T; q0 += xtok) {
      const int nq = min(xtok, T - q0);
      if (g0 < g1) stage_x_consumers(xs, xg, slots + q0, nq, H, K, kTConsumers, 1, 3);
      for (int g = g0; g < g1; ++g) {
        const int n0 = g * kTRows + 2 * warp;
        for (int c0 = 0; c0 < nq; c0 += 4) {
          const int tc = min(4, nq - c0);
          const int* sl = slots + q0 + c0;
          if (tc == 4) tma_chunk<S, 4>(c, nsteps, xs, c0, sl, n0, h, error_flag, H, I);
          else if (tc == 3) tma_chunk<S, 3>(c, nsteps, xs, c0, sl, n0, h, error_flag, H, I);
          else if (tc == 2) tma_chunk<S, 2>(c, nsteps, xs, c0, sl, n0, h, error_flag, H, I);
          else tma_chunk<S, 1>(c, nsteps, xs, c0, sl, n0, h, error_flag, H, I);
        }
      }
    }
  }
}

bool gate_up_tma_supported(int B, int H, int I, int E, int K) {
  return B * K <= kStreamMaxSlots && E <= 4096 && H % kTStepCols == 0 && H <= 16384 &&
         tma_smem_bytes(H, 3) <= kTSmemLimit;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D byte tensor [rows][cols] (row stride = cols) with boxes of box_cols x box_rows.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int S>
cudaError_t launch_tma_t(const GateUpArgs& a, cudaStream_t stream, bool pdl) {
  const int smem = tma_smem_bytes(a.H, S);
  static int configured = 0;
  if (configured < smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(moe_gate_up_tma<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  CUtensorMap mw, ms;
  const uint64_t rows = (uint64_t)a.E * 2 * a.I;
  if (!encode_2d(&mw, a.gate_up, (uint64_t)a.H, rows, kTBoxCols, kTRows) ||
      !encode_2d(&ms, a.gate_up_scale, (uint64_t)(a.H / 32), rows, 32, kTRows))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_up_tma<S>, mw, ms,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids,
                            reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag, a.B, a.H, a.I,
                            a.E, a.K);
}

}  // namespace

cudaError_t launch_gate_up_tma(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                               bool pdl) {
  (void)p;
  if (!gate_up_tma_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  return launch_tma_t<3>(a, stream, pdl);
}

}  // namespace wd
