// wd_down_mma.cu - moe_down_mma: the down kernel for batches whose tokens share
// experts, with the products of the dequantised down rows and h done by
// warp-level tensor-core MMAs.
//
// Computes what moe_down_3d_batched computes (Cursor, "用 warp decode 实现
// 更好的 MoE 模型推理", section 两个 kernel 如何工作, down paragraph): for every
// token b and output dim d, y = sum_k w[b,k] * (down row d of expert e_k) .
// h[b,k,:], then out[b,d] = bf16(y).  The kernel stays organised around
// outputs: one CTA owns 16 output dims for every token, accumulates all of
// their contributions on chip and writes each of its outputs once; nothing is
// padded, scattered to expert-major buffers or combined by a later pass.
//
// Organisation:
//   - grid: one CTA per 16 output dims (H / 16 CTAs); each builds the routing
//     tables and walks every routed expert in ascending order, in groups of up
//     to 4 of its (token, slot) pairs; a step is (expert, pair group);
//   - a producer warp streams each step into an S-stage ring: the 16 down rows
//     (16 x I bytes, one 3-D tensor-map copy, 128-byte swizzled so the MMA
//     fragment reads of 8 rows hit different banks), and, one lane per copy,
//     the pairs' BF16 h rows and the rows' scale codes (bulk copies);
//   - one converter warp per ring stage then finishes that stage, step after
//     step: the block scales decoded to FP32, and each pair's h row re-encoded
//     as FP16 scaled by a power of two 2^k so that its largest magnitude lies
//     in [2^14, 2^15) (exact for every BF16 value within 2^31 of that
//     magnitude; smaller ones are rounded to a 2^-38 grid of it, below the
//     FP32 accumulation's own rounding), with the pair's routing weight and k;
//   - 8 consumer warps split I: warp w owns the 32-column blocks w, w+8, ...
//     For each block two k16 MMAs (E4M3 -> FP16 straight into A fragments,
//     exact) give a 16 dims x 8 pairs tile that is multiplied by the block's
//     scale into the warp's FP32 sums;
//   - after a step each lane adds its sums, times w * 2^-k, into the warp's own
//     FP32 table [16 dims][B tokens] in shared memory (one table per warp, so
//     the only concurrent adds to one entry are two slots of one token on one
//     expert, which the shared-memory atomic add serialises);
//   - at the end the 8 tables are summed and each output written once as BF16.
//
// Every mbarrier wait is bounded (wd_pipeline.cuh); a warp whose wait runs out
// raises bit 1 of the error flag, stops computing or issuing and keeps
// following the consumers' final barrier; the producer waits (bounded) for its
// last copies before exiting.
#include "wd_launch.h"
#include "wd_mma.cuh"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kDWarps = 8;                      // consumer warps
constexpr int kDConv = 7;                       // converter warps (one per ring stage)
constexpr int kDThreads = 32 * (kDWarps + 1 + kDConv);
constexpr int kDRows = 16;                      // output dims per CTA
constexpr int kDPairs = 4;                      // (token, slot) pairs per step (<= 8)
constexpr int kDMaxB = 64;                      // tokens (per-warp tables)
constexpr int kDMaxStages = kDConv;
constexpr int kDSmemCap = 227 * 1024;

__host__ __device__ constexpr int d_round(int v, int a) { return (v + a - 1) / a * a; }

// Stage: [0, 16 I) swizzled down rows; FP32 scales [16 rows][I/32 blocks];
// FP16 h rows [kDPairs][hpitch]; pair info [8] x {float w, int k, int token,
// 0} (read for all 8 MMA columns, filled for the step's pairs); then what the
// copies bring for the converter: the pairs' BF16 h rows [kDPairs][2 I] and the
// rows' scale codes [16][I/32].
struct DownLayout {
  int scales, hrows, hpitch, info, hraw, sraw, stage;
  int bars, ring, tables, total;
};

__host__ __device__ inline DownLayout down_layout(int I, int B, int S) {
  DownLayout L;
  L.scales = kDRows * I;
  L.hrows = L.scales + kDRows * (I / 32) * 4;
  // FP16 row rounded up to 128 bytes, plus 64: the two pair rows read by one
  // quarter-warp fall in different halves of the 32 banks
  L.hpitch = d_round(2 * I, 128) + 64;
  L.info = L.hrows + kDPairs * L.hpitch;
  L.hraw = L.info + 8 * 16;  // info is read for 8 columns
  L.sraw = L.hraw + kDPairs * 2 * I;
  L.stage = d_round(L.sraw + kDRows * (I / 32), 1024);
  L.bars = kXOffset;  // full, empty, raw (kDMaxStages each)
  L.ring = d_round(kXOffset + 24 * kDMaxStages, 1024);
  L.tables = L.ring + S * L.stage;
  L.total = L.tables + kDWarps * kDRows * B * 4;
  return L;
}

__device__ __forceinline__ void red_add_shared(uint32_t addr, float v) {
  asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// The step sequence shared by every role of the CTA: routed expert u, pair
// group q (pairs q*8 .. of u's list).
struct DownCursor {
  int u, q;
};

__device__ __forceinline__ bool down_advance(const RoutingTables& rt, DownCursor& c) {
  if ((c.q + 1) * kDPairs < rt.off[c.u + 1] - rt.off[c.u]) {
    ++c.q;
    return true;
  }
  c.q = 0;
  return ++c.u < rt.scalar[0];
}

}  // namespace

// Threads: kDWarps consumer warps, one producer warp, kDConv converter warps.
// `tmap`: the down codes as a 3-D byte tensor {128, E * H, I / 128} with
// strides {I, 128}, boxes {128, 16, I / 128}, 128-byte swizzle.
__global__ void __launch_bounds__(kDThreads, 1) moe_down_mma(
    const __grid_constant__ CUtensorMap tmap, const __nv_bfloat16* __restrict__ h,
    const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_w,
    const uint8_t* __restrict__ down_scale, __nv_bfloat16* __restrict__ out,
    uint32_t* __restrict__ error_flag, int B, int H, int I, int E, int K, int S) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const DownLayout L = down_layout(I, B, S);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K, nbi = I >> 5;
  const int d0 = blockIdx.x * kDRows;
  const uint32_t base = smem_u32(smem);
  const uint32_t full = base + L.bars, empty = full + 8 * kDMaxStages, raw = empty + 8 * kDMaxStages;
  const uint32_t ring = base + L.ring;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + 8 * s, 2);  // the row copy's arrive and the stage's converter warp
      mbar_init(empty + 8 * s, kDWarps);
      mbar_init(raw + 8 * s, 1);
    }
    mbar_init_fence();
  }
  // the consumers' token tables start at zero
  for (int i = tid; i < kDWarps * kDRows * B; i += blockDim.x)
    reinterpret_cast<float*>(smem + L.tables)[i] = 0.0f;
  // h, topk_ids and topk_w may come from the kernel before this one.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();
  build_routing_tables(rt, topk_ids, BK, E, kDPairs, blockDim.x);  // ends with a CTA barrier
  if (rt.scalar[2] && blockIdx.x == 0 && tid == 0 && error_flag) atomicOr(error_flag, 1u);
  const int U = rt.scalar[0];

  if (warp == kDWarps) {  // producer: every copy of a step, one lane per copy
    if (U == 0) return;
    DownCursor c{0, 0};
    uint32_t i = 0;
    bool ok = true;
    const uint8_t* hg = reinterpret_cast<const uint8_t*>(h) + wait_token;
    for (; ok; ++i, ok = down_advance(rt, c)) {
      const uint32_t s = i % S, r = i / S;
      bool free = true;
      if (lane == 0 && r > 0) free = mbar_wait(empty + 8 * s, (r - 1) & 1);
      if (!__shfl_sync(0xFFFFFFFFu, free ? 1 : 0, 0)) {
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
        break;
      }
      const uint32_t st = ring + s * L.stage;
      const int T = rt.off[c.u + 1] - rt.off[c.u];
      const int* sl = rt.slots + rt.off[c.u] + c.q * kDPairs;
      const int nq = min(kDPairs, T - c.q * kDPairs);
      const size_t row0 = (size_t)rt.expert[c.u] * H + d0;
      if (lane == 0) {
        mbar_arrive_expect_tx(full + 8 * s, (uint32_t)(kDRows * I));
        tma_load_3d(st, &tmap, 0, (int)row0, 0, full + 8 * s);
        mbar_arrive_expect_tx(raw + 8 * s, (uint32_t)(nq * 2 * I + kDRows * nbi));
      }
      __syncwarp();
      if (lane < nq)  // pair `lane`'s BF16 h row
        bulk_g2s_nohint(st + L.hraw + lane * 2 * I, hg + (size_t)sl[lane] * I * 2,
                        (uint32_t)(2 * I), raw + 8 * s);
      if (lane == 31)  // the 16 rows' scale codes
        bulk_g2s_nohint(st + L.sraw, down_scale + row0 * nbi, (uint32_t)(kDRows * nbi),
                        raw + 8 * s);
    }
    if (lane == 0)  // the copies issued last land before the CTA exits
      for (uint32_t k = i > (uint32_t)S ? i - S : 0u; k < i; ++k) {
        (void)mbar_wait(full + 8 * (k % S), (k / S) & 1);
        (void)mbar_wait(raw + 8 * (k % S), (k / S) & 1);
      }
    return;
  }

  if (warp > kDWarps) {  // converters: warp cw fills every step of ring stage cw
    const int cw = warp - kDWarps - 1;
    if (U == 0 || cw >= S) return;
    DownCursor c{0, 0};
    uint32_t i = 0;
    bool ok = true;
    for (; ok; ++i, ok = down_advance(rt, c)) {
      // one converter per stage, so its waits on the stage's barriers always
      // target the phase right after the one it last saw complete
      if ((int)(i % S) != cw) continue;
      const uint32_t s = i % S;
      if (!mbar_wait(raw + 8 * s, (i / S) & 1)) {
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
        break;
      }
      const uint32_t st = ring + s * L.stage;
      const int T = rt.off[c.u + 1] - rt.off[c.u];
      const int* sl = rt.slots + rt.off[c.u] + c.q * kDPairs;
      const int nq = min(kDPairs, T - c.q * kDPairs);
      // scale codes -> FP32 [row][block], 16 codes per lane per pass
      for (int q16 = lane; q16 < nbi; q16 += 32) {
        const uint4 v = lds_u32x4(st + L.sraw + q16 * 16);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(st + L.scales + (q16 * 16 + 4 * q) * 4),
                       "f"(e8m0_to_f32(wv[q] & 0xFFu)), "f"(e8m0_to_f32((wv[q] >> 8) & 0xFFu)),
                       "f"(e8m0_to_f32((wv[q] >> 16) & 0xFFu)), "f"(e8m0_to_f32(wv[q] >> 24))
                       : "memory");
      }
      // each pair's h row: largest magnitude, then FP16 times 2^k
      const int nch = I >> 3;  // 16-byte chunks of 8 BF16 values
      for (int p = 0; p < nq; ++p) {
        const uint32_t src = st + L.hraw + p * 2 * I;
        uint32_t mx = 0u;
        for (int ch = lane; ch < nch; ch += 32) {
          const uint4 w = lds_u32x4(src + ch * 16);
          mx = max(mx, max(max(max_abs_bf16x2(w.x), max_abs_bf16x2(w.y)),
                           max(max_abs_bf16x2(w.z), max_abs_bf16x2(w.w))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        const int k = fp16_row_exponent(mx);
        const float f1 = exp2_int(k >> 1), f2 = exp2_int(k - (k >> 1));
        for (int ch = lane; ch < nch; ch += 32) {
          const uint4 w = lds_u32x4(src + ch * 16);
          const uint32_t in[4] = {w.x, w.y, w.z, w.w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = bf16x2_to_f32(in[q]);
            const __half2 hv = __floats2half2_rn((f.x * f1) * f2, (f.y * f1) * f2);
            o[q] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(st + L.hrows + p * L.hpitch + ch * 16),
                       "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
        if (lane == 0)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(st + L.info + p * 16),
                       "f"(__ldg(topk_w + sl[p])), "r"(k), "r"(sl[p] / K), "r"(0)
                       : "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full + 8 * s);
    }
    return;
  }

  // consumers
  const int g = lane >> 2, tig = lane & 3;
  const int pg = slab_row(g);  // the down row (output dim) of tile rows g and g + 8
  const uint32_t table = base + L.tables + warp * kDRows * B * 4;
  bool dead = false;
  if (U > 0) {
    DownCursor c{0, 0};
    uint32_t i = 0;
    bool ok = true;
    for (; ok; ++i, ok = down_advance(rt, c)) {
      const uint32_t s = i % S;
      const uint32_t st = ring + s * L.stage;
      const int T = rt.off[c.u + 1] - rt.off[c.u];
      const int nq = min(kDPairs, T - c.q * kDPairs);
      if (!dead && !mbar_wait(full + 8 * s, (i / S) & 1)) {
        dead = true;
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
      }
      if (dead) continue;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t brow = st + L.hrows + (g < nq ? g : 0) * L.hpitch + tig * 16;
      for (int j = warp; j < nbi; j += kDWarps) {
        const int col = j * 32 + tig * 8;
        const uint2 w0 = lds_u32x2(st + slab_offset(pg, col));
        const uint2 w1 = lds_u32x2(st + slab_offset(pg + 8, col));
        const uint4 b = lds_u32x4(brow + j * 64);
        // columns 8 tig + 0..3 (first k16 step) and 8 tig + 4..7 (second)
        float cc[4];
        mma_f16_zero(cc, e4m3x2_lo_to_f16x2(w0.x), e4m3x2_lo_to_f16x2(w1.x),
                     e4m3x2_hi_to_f16x2(w0.x), e4m3x2_hi_to_f16x2(w1.x), b.x, b.y);
        mma_f16_acc(cc, e4m3x2_lo_to_f16x2(w0.y), e4m3x2_lo_to_f16x2(w1.y),
                    e4m3x2_hi_to_f16x2(w0.y), e4m3x2_hi_to_f16x2(w1.y), b.z, b.w);
        const float s0 = lds_f32(st + L.scales + (pg * nbi + j) * 4);
        const float s1 = lds_f32(st + L.scales + ((pg + 8) * nbi + j) * 4);
        acc[0] = fmaf(cc[0], s0, acc[0]);
        acc[1] = fmaf(cc[1], s0, acc[1]);
        acc[2] = fmaf(cc[2], s1, acc[2]);
        acc[3] = fmaf(cc[3], s1, acc[3]);
      }
      // this lane's pairs 2 tig, 2 tig + 1: routing weight, exponent, token
      uint4 info[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) info[q] = lds_u32x4(st + L.info + (2 * tig + q) * 16);
      __syncwarp();  // every lane is done with the stage
      if (lane == 0) mbar_arrive(empty + 8 * s);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (2 * tig + q >= nq) continue;
        const float wv = __uint_as_float(info[q].x);
        const int k = (int)info[q].y, tok = (int)info[q].z;
        const float f1 = exp2_int(-(k >> 1)), f2 = exp2_int(-(k - (k >> 1)));
        red_add_shared(table + (uint32_t)((pg * B + tok) * 4), ((acc[q] * wv) * f1) * f2);
        red_add_shared(table + (uint32_t)(((pg + 8) * B + tok) * 4), ((acc[2 + q] * wv) * f1) * f2);
      }
    }
  }
  // all consumer warps' tables are complete: sum them, one BF16 store per output
  named_barrier_sync(1, kDWarps * 32);
  const float* tabs = reinterpret_cast<const float*>(smem + L.tables);
  for (int idx = tid; idx < kDRows * B; idx += kDWarps * 32) {
    float y = 0.0f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) y += tabs[w * kDRows * B + idx];
    const int row = idx / B, b = idx - row * B;
    out[(size_t)b * H + d0 + row] = __float2bfloat16_rn(y);
  }
}

namespace {

int down_mma_stages(int I, int B) {
  for (int S = kDMaxStages; S >= 2; --S)
    if (down_layout(I, B, S).total <= kDSmemCap) return S;
  return 0;
}

}  // namespace

bool down_mma_supported(int B, int H, int I, int E, int K) {
  return B <= kDMaxB && B * K <= kStreamMaxSlots && E <= 4096 && H % kDRows == 0 &&
         I % 128 == 0 && I / 128 <= 256 && (long long)E * H < (1ll << 31) &&
         down_mma_stages(I, B) >= 2;
}

cudaError_t launch_down_mma(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl) {
  if (!down_mma_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  int S = down_mma_stages(a.I, a.B);
  if (p.qpl >= 2 && p.qpl < S) S = p.qpl;
  const int smem = down_layout(a.I, a.B, S).total;
  static int configured = 0;
  if (configured < smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(moe_down_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  CUtensorMap map;
  if (!encode_row_slab_map(&map, a.down, (uint64_t)a.E * a.H, a.I)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.H / kDRows));
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_mma, map, reinterpret_cast<const __nv_bfloat16*>(a.h),
                            a.topk_ids, a.topk_w, a.down_scale,
                            reinterpret_cast<__nv_bfloat16*>(a.out), a.error_flag, a.B, a.H,
                            a.I, a.E, a.K, S);
}

}  // namespace wd
