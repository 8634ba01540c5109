// wd_down_expert_mma.cu - moe_down_expert_mma: the down kernel for batches
// whose tokens share experts, one warp per routed expert (and group of up to
// 4 of its pairs) with the products on the tensor cores.
//
// Computes what moe_down_3d_batched computes (Cursor, "用 warp decode 实现
// 更好的 MoE 模型推理", section 两个 kernel 如何工作, down paragraph): for every
// token b and output dim d, y = sum_k w[b,k] * (down row d of expert e_k) .
// h[b,k,:], then out[b,d] = bf16(y).  One CTA owns 16 output dims for every
// token, accumulates all of their contributions on chip and writes each of its
// outputs once: nothing is padded, scattered to expert-major buffers or
// combined by a later pass.
//
// Organisation:
//   - grid: one CTA per 16 output dims (H / 16 CTAs).  Each builds the routing
//     tables and walks the routed experts in ascending order, in groups of up
//     to 4 of their (token, slot) pairs, and splits I into nh parts (1, or 2
//     when I / 128 is even); a step is (expert, pair group, part);
//   - one producer warp streams every step into an S-stage ring: the part of
//     the 16 down rows (16 x I / nh bytes, one 3-D tensor-map copy, 128-byte
//     swizzled so that
//     the MMA fragment reads of 8 rows hit different banks), the rows' scale
//     codes and the part of the pairs' BF16 h rows (bulk copies, one lane per
//     copy).  The weights of the first S steps are requested before the kernel
//     waits for the grid that writes h.  S >= 8, the number of consumer warps:
//     no warp can then wait on a stage whose previous step has not landed yet,
//     which the mbarrier phase parity could not tell apart;
//   - consumer warp w takes steps w, w + 8, ... whole: it decodes the step's
//     scale codes into its own FP32 table, re-encodes each pair's part of h in
//     place as FP16 scaled by a power of two 2^k (largest magnitude in
//     [2^14, 2^15): exact for every BF16 value within 2^31 of that magnitude,
//     smaller ones rounded to a 2^-38 grid of it, below the FP32 accumulation's
//     own rounding), then runs over the part's blocks: two k16 MMAs (E4M3 ->
//     FP16 straight into A fragments, exact) give a 16 dims x 8 pair-columns
//     tile, multiplied by the block's scale into FP32 sums;
//   - after a step each lane adds its sums, times w * 2^-k, into the warp's
//     own FP32 table [16 dims][B tokens] (shared-memory atomic add: the only
//     concurrent adds to one entry are two slots of one token on one expert);
//   - at the end the 8 tables are summed in warp order and each output is
//     written once as BF16.
//
// Every mbarrier wait is bounded (wd_pipeline.cuh); a warp whose wait runs out
// raises bit 1 of the error flag and stops computing or issuing; the producer
// waits (bounded) for its last copies before exiting.
#include "wd_launch.h"
#include "wd_mma.cuh"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kEWarps = 8;                  // consumer warps
constexpr int kEThreads = 32 * (kEWarps + 1);
constexpr int kERows = 16;                  // output dims per CTA
constexpr int kEPairs = 4;                  // (token, slot) pairs per step (<= 8)
constexpr int kEMaxB = 64;                  // tokens (per-warp tables)
constexpr int kEMaxStages = 16;
constexpr int kESmemCap = 227 * 1024;

__host__ __device__ constexpr int e_round(int v, int a) { return (v + a - 1) / a * a; }

// Parts of I per step: 1, or 2 when I / 128 is even (each part whole
// 128-column slabs).
__host__ __device__ inline bool edown_parts_ok(int I, int nh) {
  return nh == 1 || (nh == 2 && (I / 128) % 2 == 0);
}

// Stage: [0, 16 Ip) swizzled down rows of the part (Ip = I / nh columns);
// the 16 rows' scale codes [16][I/32] (all parts); the pairs' h parts
// [kEPairs][hpitch] (BF16 as copied, FP16 once re-encoded).  After the ring:
// per-warp FP32 scale tables [16][Ip/32], per-warp token tables [16][B] and
// the call's routing weights [B*K].
struct EDownLayout {
  int ip, sraw, hrows, hpitch, stage, bars, ring, scl, tables, wtab, total;
};

__host__ __device__ inline EDownLayout edown_layout(int I, int B, int S, int nh) {
  EDownLayout L;
  const int nbi = I / 32;
  L.ip = I / nh;
  L.sraw = kERows * L.ip;
  L.hrows = e_round(L.sraw + kERows * nbi, 16);
  // row rounded up to 128 bytes, plus 64: the two pair rows read by one
  // quarter-warp fall in different halves of the 32 banks
  L.hpitch = e_round(2 * L.ip, 128) + 64;
  L.stage = e_round(L.hrows + kEPairs * L.hpitch, 1024);
  L.bars = kXOffset;  // full, empty (kEMaxStages each)
  L.ring = e_round(kXOffset + 16 * kEMaxStages, 1024);
  L.scl = L.ring + S * L.stage;
  L.tables = L.scl + kEWarps * kERows * (L.ip / 32) * 4;
  L.wtab = L.tables + kEWarps * kERows * B * 4;
  L.total = L.wtab + kStreamMaxSlots * 4;
  return L;
}

__device__ __forceinline__ void red_add_shared_f32(uint32_t addr, float v) {
  asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Step sequence shared by every role of the CTA: routed expert u, pair group
// q (pairs kEPairs q .. of u's list), part p of I (nh parts).
struct ECursor {
  int u, q, p;
};

__device__ __forceinline__ bool e_advance(const RoutingTables& rt, ECursor& c, int nh) {
  if (++c.p < nh) return true;
  c.p = 0;
  if ((c.q + 1) * kEPairs < rt.off[c.u + 1] - rt.off[c.u]) {
    ++c.q;
    return true;
  }
  c.q = 0;
  return ++c.u < rt.scalar[0];
}

__device__ __forceinline__ int e_pairs(const RoutingTables& rt, const ECursor& c) {
  return min(kEPairs, rt.off[c.u + 1] - rt.off[c.u] - c.q * kEPairs);
}

// Re-encode the BF16 row at `row` (n values) in place as FP16 times 2^k; all
// 32 lanes take part.  Returns k.
__device__ __forceinline__ int h_row_to_f16(uint32_t row, int n) {
  const int lane = threadIdx.x & 31;
  const int nch = n >> 3;  // 16-byte chunks of 8 values
  uint32_t mx = 0u;
  for (int ch = lane; ch < nch; ch += 32) {
    const uint4 w = lds_u32x4(row + ch * 16);
    mx = max(mx, max(max(max_abs_bf16x2(w.x), max_abs_bf16x2(w.y)),
                     max(max_abs_bf16x2(w.z), max_abs_bf16x2(w.w))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  const int k = fp16_row_exponent(mx);
  // one multiply while 2^k is a normal FP32 value, else two (both exact)
  const bool one = k >= -126 && k <= 127;
  const float f1 = one ? exp2_int(k) : exp2_int(k >> 1);
  const float f2 = one ? 1.0f : exp2_int(k - (k >> 1));
  for (int ch = lane; ch < nch; ch += 32) {
    const uint4 w = lds_u32x4(row + ch * 16);
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = bf16x2_to_f32(in[q]);
      const __half2 hv = one ? __floats2half2_rn(f.x * f1, f.y * f1)
                             : __floats2half2_rn((f.x * f1) * f2, (f.y * f1) * f2);
      o[q] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + ch * 16), "r"(o[0]),
                 "r"(o[1]), "r"(o[2]), "r"(o[3])
                 : "memory");
  }
  return k;
}

}  // namespace

// Threads: kEWarps consumer warps, then one producer warp.  `tmap`: the down
// codes as a 3-D byte tensor {128, E * H, I / 128} with strides {I, 128},
// boxes {128, 16, I / (128 nh)}, 128-byte swizzle.
__global__ void __launch_bounds__(kEThreads, 1) moe_down_expert_mma(
    const __grid_constant__ CUtensorMap tmap, const __nv_bfloat16* __restrict__ h,
    const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_w,
    const uint8_t* __restrict__ down_scale, __nv_bfloat16* __restrict__ out,
    uint32_t* __restrict__ error_flag, int B, int H, int I, int E, int K, int S, int nh) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const EDownLayout L = edown_layout(I, B, S, nh);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K, nbi = I >> 5;
  const int ip = L.ip, nbp = ip >> 5;  // columns and blocks per part
  const int d0 = blockIdx.x * kERows;
  const uint32_t base = smem_u32(smem);
  const uint32_t full = base + L.bars, empty = full + 8 * kEMaxStages;
  const uint32_t ring = base + L.ring;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + 8 * s, 1);   // the producer's arrive (with the step's bytes)
      mbar_init(empty + 8 * s, 1);  // the step's consumer warp
    }
    mbar_init_fence();
  }
  // the consumers' token tables start at zero; the routing weights
  for (int i = tid; i < kEWarps * kERows * B; i += blockDim.x)
    reinterpret_cast<float*>(smem + L.tables)[i] = 0.0f;
  float* wtab = reinterpret_cast<float*>(smem + L.wtab);
  for (int i = tid; i < BK; i += blockDim.x) wtab[i] = __ldg(topk_w + i);
  // The routing and the weights are the call's inputs; h is written by the
  // kernel before this one, and only the h copies wait for it.
  build_routing_tables(rt, topk_ids, BK, E, kEPairs, blockDim.x);  // ends with a CTA barrier
  if (rt.scalar[2] && blockIdx.x == 0 && tid == 0 && error_flag) atomicOr(error_flag, 1u);
  const int U = rt.scalar[0];

  if (warp == kEWarps) {  // producer
    if (U == 0) return;
    const uint32_t wbytes = (uint32_t)(kERows * ip + kERows * nbi);
    // lane 0: the stage's byte count, the part of the 16 rows and the rows'
    // scale codes
    auto issue_weights = [&](uint32_t s, const ECursor& c) {
      const uint32_t st = ring + s * L.stage;
      const int nq = e_pairs(rt, c);
      const int row0 = rt.expert[c.u] * H + d0;  // < 2^31 (checked on launch)
      mbar_arrive_expect_tx(full + 8 * s, wbytes + (uint32_t)(nq * 2 * ip));
      tma_load_3d(st, &tmap, 0, row0, c.p * (ip / 128), full + 8 * s);
      bulk_g2s_nohint(st + L.sraw, down_scale + (size_t)row0 * nbi, (uint32_t)(kERows * nbi),
                      full + 8 * s);
    };
    const uint8_t* hg = nullptr;
    // lane t < pairs: the part of pair t's BF16 h row
    auto issue_h = [&](uint32_t s, const ECursor& c) {
      const uint32_t st = ring + s * L.stage;
      const int nq = e_pairs(rt, c);
      const int* sl = rt.slots + rt.off[c.u] + c.q * kEPairs;
      if (lane < nq)
        bulk_g2s_nohint(st + L.hrows + lane * L.hpitch,
                        hg + (size_t)sl[lane] * I * 2 + (size_t)c.p * ip * 2, (uint32_t)(2 * ip),
                        full + 8 * s);
    };
    ECursor c{0, 0, 0};
    uint32_t i = 0;
    bool ok = true;
    // the first S steps' weights go out before waiting for the grid that writes h
    for (; ok && i < (uint32_t)S; ++i, ok = e_advance(rt, c, nh))
      if (lane == 0) issue_weights(i, c);
    const uint32_t npre = i;
    hg = reinterpret_cast<const uint8_t*>(h) + grid_dependency_wait();
    grid_launch_dependents();
    __syncwarp();
    {
      ECursor c2{0, 0, 0};
      for (uint32_t k = 0; k < npre; ++k, (void)e_advance(rt, c2, nh)) issue_h(k, c2);
    }
    for (; ok; ++i, ok = e_advance(rt, c, nh)) {
      const uint32_t s = i % S, r = i / S;  // r >= 1 here
      bool free = true;
      if (lane == 0) free = mbar_wait(empty + 8 * s, (r - 1) & 1);
      if (!__shfl_sync(0xFFFFFFFFu, free ? 1 : 0, 0)) {
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
        break;
      }
      if (lane == 0) issue_weights(s, c);
      __syncwarp();
      issue_h(s, c);
    }
    if (lane == 0)  // the copies issued last land before the CTA exits
      for (uint32_t k = i > (uint32_t)S ? i - S : 0u; k < i; ++k)
        (void)mbar_wait(full + 8 * (k % S), (k / S) & 1);
    return;
  }

  // consumers
  (void)grid_dependency_wait();  // the writes of `out` below follow the previous grid
  const int g = lane >> 2, tig = lane & 3;
  const int pg = slab_row(g);  // the down row (output dim) of tile rows g and g + 8
  const uint32_t table = base + L.tables + warp * kERows * B * 4;
  const uint32_t scl = base + L.scl + warp * kERows * nbp * 4;
  bool dead = false;
  if (U > 0) {
    ECursor c{0, 0, 0};
    uint32_t i = 0;
    bool ok = true;
    for (; ok; ++i, ok = e_advance(rt, c, nh)) {
      if ((int)(i % kEWarps) != warp) continue;
      const uint32_t s = i % S;
      const uint32_t st = ring + s * L.stage;
      const int nq = e_pairs(rt, c);
      const int* sl = rt.slots + rt.off[c.u] + c.q * kEPairs;
      if (!dead && !mbar_wait(full + 8 * s, (i / S) & 1)) {
        dead = true;
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
      }
      if (dead) continue;
      // the part's scale codes -> FP32 [row][block]; codes 1..254 decode as
      // code << 23, a word holding a 0 (2^-127) or 255 (NaN) takes the general
      // rule.  Word wi: row wi / (nbp / 4), blocks 4 (wi % (nbp / 4)) + 0..3.
      const int wpr = nbp >> 2;
      for (int wi = lane; wi < 4 * nbp; wi += 32) {
        const int row = wi / wpr;
        const uint32_t code = lds_u32(st + L.sraw + row * nbi + c.p * nbp + 4 * (wi - row * wpr));
        float f[4];
        if (!e8m0x4_any_special(code)) {
#pragma unroll
          for (int t = 0; t < 4; ++t) f[t] = __uint_as_float(((code >> (8 * t)) & 0xFFu) << 23);
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t) f[t] = e8m0_to_f32((code >> (8 * t)) & 0xFFu);
        }
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(scl + 16 * wi), "f"(f[0]),
                     "f"(f[1]), "f"(f[2]), "f"(f[3])
                     : "memory");
      }
      // the part of the pairs' h rows, FP16 times 2^k
      int kp[kEPairs];
#pragma unroll
      for (int t = 0; t < kEPairs; ++t) kp[t] = t < nq ? h_row_to_f16(st + L.hrows + t * L.hpitch, ip) : 0;
      __syncwarp();  // the tables and rows are complete
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t brow = st + L.hrows + (g < nq ? g : 0) * L.hpitch + tig * 16;
      const uint32_t s0row = scl + pg * nbp * 4, s1row = scl + (pg + 8) * nbp * 4;
      for (int j4 = 0; j4 < nbp; j4 += 4) {
        const float4 sa = lds_f32x4(s0row + 4 * j4), sb = lds_f32x4(s1row + 4 * j4);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = j4 + jj;
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
          const float s0 = jj == 0 ? sa.x : jj == 1 ? sa.y : jj == 2 ? sa.z : sa.w;
          const float s1 = jj == 0 ? sb.x : jj == 1 ? sb.y : jj == 2 ? sb.z : sb.w;
          acc[0] = fmaf(cc[0], s0, acc[0]);
          acc[1] = fmaf(cc[1], s0, acc[1]);
          acc[2] = fmaf(cc[2], s1, acc[2]);
          acc[3] = fmaf(cc[3], s1, acc[3]);
        }
      }
      __syncwarp();  // every lane is done with the stage
      if (lane == 0) mbar_arrive(empty + 8 * s);
      // this lane's pair columns 2 tig, 2 tig + 1
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int pc = 2 * tig + q;
        if (pc >= nq) continue;
        const int k = pc == 0 ? kp[0] : pc == 1 ? kp[1] : pc == 2 ? kp[2] : kp[3];
        const int slot = sl[pc];
        const int tok = slot / K;
        const float wv = wtab[slot];
        const float f1 = exp2_int(-(k >> 1)), f2 = exp2_int(-(k - (k >> 1)));
        red_add_shared_f32(table + (uint32_t)((pg * B + tok) * 4), ((acc[q] * wv) * f1) * f2);
        red_add_shared_f32(table + (uint32_t)(((pg + 8) * B + tok) * 4),
                           ((acc[2 + q] * wv) * f1) * f2);
      }
    }
  }
  // all consumer warps' tables are complete: sum them, one BF16 store per output
  named_barrier_sync(1, kEWarps * 32);
  const float* tabs = reinterpret_cast<const float*>(smem + L.tables);
  for (int idx = tid; idx < kERows * B; idx += kEWarps * 32) {
    float y = 0.0f;
#pragma unroll
    for (int w = 0; w < kEWarps; ++w) y += tabs[w * kERows * B + idx];
    const int row = idx / B, b = idx - row * B;
    out[(size_t)b * H + d0 + row] = __float2bfloat16_rn(y);
  }
}

namespace {

// Ring depth: the deepest (up to kEMaxStages) that fits; at least kEWarps
// (a consumer warp must never wait on a stage whose previous step it could
// mistake for its own), else 0 (unsupported).
int edown_stages(int I, int B, int nh) {
  for (int S = kEMaxStages; S >= kEWarps; --S)
    if (edown_layout(I, B, S, nh).total <= kESmemCap) return S;
  return 0;
}

}  // namespace

bool down_expert_mma_supported(int B, int H, int I, int E, int K) {
  return B <= kEMaxB && B * K <= kStreamMaxSlots && E <= 4096 && H % kERows == 0 &&
         I % 128 == 0 && I / 128 <= 256 && (long long)E * H < (1ll << 31) &&
         edown_stages(I, B, 1) >= kEWarps;
}

// p.qpl: ring stages (0: the deepest that fits; at least kEWarps); p.rpw:
// parts of I per step (2 if it applies and fits, else 1).
cudaError_t launch_down_expert_mma(const DownArgs& a, const DownPlan& p, cudaStream_t stream,
                                   bool pdl) {
  if (!down_expert_mma_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  const int nh = (p.rpw == 2 && edown_parts_ok(a.I, 2) && edown_stages(a.I, a.B, 2) > 0) ? 2 : 1;
  int S = edown_stages(a.I, a.B, nh);
  if (p.qpl >= kEWarps && p.qpl < S) S = p.qpl;
  const int smem = edown_layout(a.I, a.B, S, nh).total;
  static int configured = 0;
  if (configured < smem) {
    const cudaError_t e = cudaFuncSetAttribute(moe_down_expert_mma,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  CUtensorMap map;
  if (!encode_row_slab_map(&map, a.down, (uint64_t)a.E * a.H, a.I, a.I / nh))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.H / kERows));
  cfg.blockDim = dim3(kEThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_expert_mma, map,
                            reinterpret_cast<const __nv_bfloat16*>(a.h), a.topk_ids, a.topk_w,
                            a.down_scale, reinterpret_cast<__nv_bfloat16*>(a.out), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K, S, nh);
}

}  // namespace wd
