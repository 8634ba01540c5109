// wd_gate_up_mma.cu - moe_gate_up_mma: the gate/up kernel for batches whose
// tokens share experts, with the multiply-accumulate of the dequantised rows
// and the activations done by warp-level tensor-core MMAs.
//
// Computes what moe_gate_up_3d_batched computes (Cursor, "用 warp decode 实现
// 更好的 MoE 模型推理", section 两个 kernel 如何工作, gate/up paragraph): for
// every (token, routed slot) and intermediate neuron n, the dot products of
// gate row n and up row I+n of the routed expert with x, then one BF16 value
// bf16(SiLU(g) * u), written once, with no padding, scatter or combine pass.
//
// Why tensor cores here.  Once the tokens routed to one expert are grouped
// (as moe_gate_up_persist does), the work of that expert is a small dense
// product [2I x H] . [H x T] with T tokens.  On CUDA cores the dequantisation
// (E4M3 -> FP16 -> FP32) and the T FP32 multiply-adds per weight cost ~4.8
// warp instructions per weight element at B = 32, which bounds that kernel by
// instruction issue, not by HBM.  Here each weight element costs one half of a
// cvt (E4M3x2 -> F16x2, exact) and its share of one mma.sync.m16n8k16 per 256
// elements, whatever T is (up to 8 tokens per MMA column tile).
//
// Organisation:
//   - an item is (routed expert, 16 neurons): gate rows n0..n0+15 and up rows
//     I+n0..I+n0+15, computed as two 16-row MMA tiles; tile r has gate rows
//     n0+8r..n0+8r+7 as rows 0..7 and the matching up rows as rows 8..15, so
//     the lane holding gate(n, t) in the accumulator also holds up(n, t);
//   - one CTA per SM walks a contiguous, cost-balanced range of items (after
//     building the routing tables once).  A producer thread streams each item
//     into an S-stage shared-memory ring with four copies that complete on the
//     stage's mbarrier: the 16 gate rows and the 16 up rows (each one 3-D
//     tensor-map copy, 16 x H bytes, 128-byte swizzled so that the MMA fragment
//     reads of 8 rows hit different banks) and their scale bytes (two 3-D
//     tensor-map copies of 16 x H/32 bytes, stored as [H/512][16 rows][16] so
//     that the 8 or 4 codes a lane reads for its row and chunk sit 16 bytes
//     from the next row's, not H/32).  The bytes in flight are held by shared
//     memory (two items, 130 KiB per SM at H = 2048), not by registers;
//   - the consumer warps (8, or 16 on request) split H: at H = 2048 each owns
//     one 256-column (128-column) chunk of every item.  They write their
//     partial tiles into one of two shared-memory buffers guarded by mbarriers
//     and go on; an epilogue warp sums each buffer and stores the item's
//     bf16(SiLU(g) * u) values (gate and up of one output sit in one lane).
//     The consumers meet at a named barrier only when the staged activations
//     change;
//   - MMA tile row g reads slab row 2 (g % 4) + g / 4, which keeps every
//     half-warp's fragment loads on 8 distinct swizzled 16-byte chunks;
//   - MXFP8 block scales: the two k16 MMAs of one 32-column block accumulate
//     into a fresh tile, which is then multiplied by the block's power-of-two
//     scale into the running FP32 sum (exact barring FP32 over/underflow);
//   - the k index inside a block is permuted (lane quad tig takes columns
//     8 tig .. 8 tig + 7, i.e. 8 contiguous bytes of each of its rows), and
//     the activations are staged with the same permutation, which for this
//     fragment layout is the natural column order;
//   - activations: when the CTA enters an expert its consumer warps stage the
//     x rows of its tokens (up to 8 at a time) in shared memory as FP16, each
//     token scaled by a power of two 2^k_t so that its largest magnitude falls
//     in [2^14, 2^15).  Power-of-two scaling is exact, and every BF16 value
//     within 2^31 of the token's largest magnitude is an FP16 value after it,
//     so the re-encoding is exact for those; smaller values are rounded to a
//     grid of 2^-38 of that largest magnitude, below the rounding of the FP32
//     accumulation itself.  The accumulators are multiplied by 2^-k_t in the
//     epilogue.  FP16 x FP16 products are exact in FP32; the MMA accumulates in
//     FP32.  An expert with more than 8 tokens is computed in groups of 8,
//     each reading the item's rows again (from L2).
//
// Every mbarrier wait is bounded (wd_pipeline.cuh).  A consumer whose wait
// runs out raises bit 1 of the error flag and computes nothing more but keeps
// following the consumers' barriers; the epilogue warp stops at its first wait
// that runs out; the producer stops issuing when its wait runs out, and before
// exiting waits (bounded) for the copies it issued last.
#include "wd_launch.h"
#include "wd_mma.cuh"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kMMaxWarps = 16;            // consumer warps (8 or 16; 2048 / 16 = 128 columns each)
constexpr int kMTokens = 8;                // tokens staged at once: one MMA column tile
constexpr int kMNeurons = 16;              // neurons per item: two 16-row MMA tiles
constexpr int kMItemBase = 8;              // item cost = groups * kMItemBase + 1
// partial sums [2 parities][warps][2 tiles][32 lanes] float4, and per-warp FP32
// scale tables [32 rows][blocks per chunk]: 32 KiB + 8 KiB for either warp count
constexpr int kMRedBytes = 2 * kMMaxWarps * 2 * 32 * 16;
constexpr int kMScaleBytes = 8 * 1024;
constexpr int kMSmemCap = 227 * 1024;
constexpr int kMMaxStages = 4;

__host__ __device__ constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory layout for a given H and ring depth S.  A stage holds the
// gate slab (16 rows, as [H/128][16][128] swizzled bytes), the up slab (same),
// then the 16 gate rows' scale bytes and the 16 up rows' (16 * H/32 each).
struct MmaLayout {
  int slab;     // bytes of one slab (16 * H)
  int stage;    // bytes of one stage, a multiple of 1024
  int bars;     // full[kMMaxStages], then empty[kMMaxStages] (8 bytes each)
  int ring;     // S stages, 1024-byte aligned
  int xs;       // staged FP16 activations, `xtok` rows of `xstride` bytes
  int xstride;
  int xtok;
  int ktok;     // per staged token exponent k_t (int[kMTokens]), then the
                // exponents of each partial-sum buffer's item (int[2][kMTokens])
  int red;      // partial sums
  int scl;      // per-warp scale tables
  int total;
};

__host__ __device__ inline MmaLayout mma_layout(int H, int S) {
  MmaLayout L;
  L.slab = 16 * H;
  L.stage = round_up(2 * L.slab + 2 * 16 * (H / 32), 1024);
  L.bars = kXOffset;
  L.ring = round_up(kXOffset + 128, 1024);  // full, empty [kMMaxStages]; rfull, rempty [2]
  L.xs = L.ring + S * L.stage;
  // FP16 row rounded up to 128 bytes, plus 64, so that the two token rows
  // read by one quarter-warp fall in different halves of the 32 banks
  L.xstride = round_up(2 * H, 128) + 64;
  const int fixed = L.xs + 128 + kMRedBytes + kMScaleBytes;
  const int t = (kMSmemCap - fixed) / L.xstride;
  L.xtok = t > kMTokens ? kMTokens : (t < 0 ? 0 : t);
  L.ktok = L.xs + L.xtok * L.xstride;
  L.red = L.ktok + 128;
  L.scl = L.red + kMRedBytes;
  L.total = L.scl + kMScaleBytes;
  return L;
}

// Stage the x rows of tokens slots[0..nq) (token b = slot / K) in shared
// memory as FP16 scaled by 2^k_t, row t at xs + t * stride, and k_t in
// ktok[t].  Warp w converts tokens w, w + 8, ...; no barrier.
__device__ __forceinline__ void stage_x_f16(uint32_t xs, int stride, int* ktok, const uint8_t* xg,
                                            const int* slots, int nq, int H, int K, int nwarps) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = H >> 3;  // 16-byte chunks of 8 BF16 values
  for (int t = warp; t < nq; t += nwarps) {
    const uint8_t* row = xg + (size_t)(slots[t] / K) * H * 2;
    uint32_t mx = 0u;
    for (int i = lane; i < nch; i += 32) {
      const uint4 v = ld_act_16B(row + i * 16);
      mx = max(mx, max(max(max_abs_bf16x2(v.x), max_abs_bf16x2(v.y)),
                       max(max_abs_bf16x2(v.z), max_abs_bf16x2(v.w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    const int k = fp16_row_exponent(mx);
    const int k1 = k >> 1, k2 = k - k1;  // each within [-57, 74]
    const float f1 = exp2_int(k1), f2 = exp2_int(k2);
    for (int i = lane; i < nch; i += 32) {
      const uint4 v = ld_act_16B(row + i * 16);
      const uint32_t in[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = bf16x2_to_f32(in[q]);
        const __half2 hv = __floats2half2_rn((f.x * f1) * f2, (f.y * f1) * f2);
        o[q] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(xs + (uint32_t)(t * stride + i * 16)),
                   "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                   : "memory");
    }
    if (lane == 0) ktok[t] = k;
  }
}

__device__ __forceinline__ int mma_item_cost(int T, int xtok) {
  return ((T + xtok - 1) / xtok) * (kMItemBase + 1);
}

// pc[u] = cost of the items of routed experts before u (nb items each); warp
// 0 computes it, then a CTA barrier.
__device__ __forceinline__ void mma_cost_prefix(const RoutingTables& rt, int nb, int xtok, int* pc) {
  const int U = rt.scalar[0];
  if ((threadIdx.x >> 5) == 0) {
    const int lane = threadIdx.x & 31;
    int acc = 0;
    for (int u0 = 0; u0 < U; u0 += 32) {
      const int u = u0 + lane;
      const int c = u < U ? nb * mma_item_cost(rt.off[u + 1] - rt.off[u], xtok) : 0;
      int excl, total;
      warp_exclusive_scan(c, excl, total);
      if (u < U) pc[u] = acc + excl;
      acc += total;
    }
    if (lane == 0) pc[U] = acc;
  }
  __syncthreads();
}

// acc[r] += the contribution of chunk c (CB blocks of 32 columns) of the item
// held in ring stage `st`, for row tile r = 0, 1.  `xrow` is the shared-memory
// address of this lane's staged activation row (token g of the group) at
// column 0 of the chunk plus 16 * tig.  `scl` is this warp's table, into which
// the chunk's 32 x CB scale codes are decoded first (FP32 [32 rows][CB]).
template <int CB>
__device__ __forceinline__ void mma_chunk(uint32_t st, int H, int c, float (&acc)[2][4],
                                          uint32_t xrow, uint32_t scl) {
  static_assert(CB == 4 || CB == 8, "4 or 8 blocks per chunk");
  const int lane = threadIdx.x & 31, g = slab_row(lane >> 2), tig = lane & 3;
  const int nblk = H >> 5;
  const uint32_t gate = st, up = st + 16 * H, sc = st + 32 * H;
  // lane l decodes table row l (gate rows 0..15, then up rows 0..15), blocks
  // CB c .. CB c + CB - 1: codes [16-block group][row][16] per 16-row half
  const int o = c * CB;
  const uint32_t src = sc + (uint32_t)((lane >> 4) * 16 * nblk + (o >> 4) * 256 + (lane & 15) * 16 + (o & 15));
  uint32_t code[CB / 4];
  if (CB == 8) {
    const uint2 v = lds_u32x2(src);
    code[0] = v.x;
    code[CB / 4 - 1] = v.y;
  } else {
    code[0] = lds_u32(src);
  }
  __syncwarp();  // the previous chunk's scale reads are done
  // codes 1..254 decode as code << 23; a lane holding a 0 (2^-127) or 255
  // (NaN) takes the general rule
  bool special = false;
#pragma unroll
  for (int q = 0; q < CB / 4; ++q) special |= e8m0x4_any_special(code[q]);
#pragma unroll
  for (int q = 0; q < CB / 4; ++q) {
    float f[4];
    if (!special) {
#pragma unroll
      for (int t = 0; t < 4; ++t) f[t] = __uint_as_float(((code[q] >> (8 * t)) & 0xFFu) << 23);
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t) f[t] = e8m0_to_f32((code[q] >> (8 * t)) & 0xFFu);
    }
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(scl + 4 * CB * lane + 16 * q),
                 "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3])
                 : "memory");
  }
  __syncwarp();
  float4 sg4[2], su4[2];
#pragma unroll
  for (int j = 0; j < CB; ++j) {
    if ((j & 3) == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sg4[r] = lds_f32x4(scl + 4 * CB * (8 * r + g) + 4 * j);
        su4[r] = lds_f32x4(scl + 4 * CB * (16 + 8 * r + g) + 4 * j);
      }
    }
    const uint4 b = lds_u32x4(xrow + 64 * j);
    const int col = c * 32 * CB + j * 32 + tig * 8;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float sg = (j & 3) == 0 ? sg4[r].x : (j & 3) == 1 ? sg4[r].y : (j & 3) == 2 ? sg4[r].z : sg4[r].w;
      const float su = (j & 3) == 0 ? su4[r].x : (j & 3) == 1 ? su4[r].y : (j & 3) == 2 ? su4[r].z : su4[r].w;
      const uint32_t off = slab_offset(8 * r + g, col);
      const uint2 wg = lds_u32x2(gate + off), wu = lds_u32x2(up + off);
      // columns 8 tig + 0..3 (first k16 step) and 8 tig + 4..7 (second)
      const uint32_t a00 = e4m3x2_lo_to_f16x2(wg.x), a02 = e4m3x2_hi_to_f16x2(wg.x);
      const uint32_t a01 = e4m3x2_lo_to_f16x2(wu.x), a03 = e4m3x2_hi_to_f16x2(wu.x);
      const uint32_t a10 = e4m3x2_lo_to_f16x2(wg.y), a12 = e4m3x2_hi_to_f16x2(wg.y);
      const uint32_t a11 = e4m3x2_lo_to_f16x2(wu.y), a13 = e4m3x2_hi_to_f16x2(wu.y);
      float cc[4];
      mma_f16_zero(cc, a00, a01, a02, a03, b.x, b.y);
      mma_f16_acc(cc, a10, a11, a12, a13, b.z, b.w);
      acc[r][0] = fmaf(cc[0], sg, acc[r][0]);
      acc[r][1] = fmaf(cc[1], sg, acc[r][1]);
      acc[r][2] = fmaf(cc[2], su, acc[r][2]);
      acc[r][3] = fmaf(cc[3], su, acc[r][3]);
    }
  }
}

// Position in a CTA's walk: routed expert u, token group q (xtok tokens each),
// item g in [g0, g1) (the items of u in this CTA's range).
struct MmaCursor {
  int u, q, g, g0, g1;
};

}  // namespace

// Threads: NW consumer warps (each owns chunks of 2048 / NW columns of an
// item: 8 warps x 256 or 16 warps x 128 at H = 2048), then one producer warp.
// `S`: ring stages.  `tmap`: the gate/up codes as a 3-D byte tensor
// {128, E * 2I, H / 128} with strides {H, 128}, boxes {128, 16, H / 128},
// 128-byte swizzle.  `smap`: their scale codes as a 3-D byte tensor
// {16, E * 2I, H / 512} with strides {H / 32, 16}, boxes {16, 16, H / 512}.
template <int NW>
__global__ void __launch_bounds__(32 * NW + 64, 1) moe_gate_up_mma(
    const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap smap,
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_ids,
    __nv_bfloat16* __restrict__ h, uint32_t* __restrict__ error_flag, int B, int H, int I, int E,
    int K, int S) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const MmaLayout L = mma_layout(H, S);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int CB = 64 / NW;  // blocks of 32 columns per chunk
  const int BK = B * K, nblk = H >> 5, nchunk = nblk / CB;
  const uint32_t base = smem_u32(smem);
  const uint32_t full = base + L.bars, empty = full + 8 * kMMaxStages;
  const uint32_t rfull = empty + 8 * kMMaxStages, rempty = rfull + 16;  // [2] each
  const uint32_t ring = base + L.ring;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, NW);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(rfull + 8 * p, NW);  // each consumer warp's partial sums are in
      mbar_init(rempty + 8 * p, 1);  // the epilogue warp is done with them
    }
    mbar_init_fence();
  }
  // x and topk_ids may come from the kernel before this one on the stream.
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();
  build_routing_tables(rt, topk_ids, BK, E, 4, blockDim.x);  // ends with a CTA barrier
  zero_bad_slots(rt, h, error_flag, BK, I, E);

  // cost-balanced contiguous range of (expert, 16-neuron) items for this CTA
  const int U = rt.scalar[0];
  const int nb = I / kMNeurons;
  const int xtok = L.xtok;
  int* pc = rt.coff;
  mma_cost_prefix(rt, nb, xtok, pc);
  const int total = pc[U];
  const int lo = (int)((long long)total * blockIdx.x / gridDim.x);
  const int hi = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  if (lo >= hi) return;

  // first item of routed expert u or later that lies in [lo, hi)
  auto enter = [&](MmaCursor& c, int u) -> bool {
    for (; u < U && pc[u] < hi; ++u) {
      const int cu = mma_item_cost(rt.off[u + 1] - rt.off[u], xtok);
      const int g0 = pc[u] >= lo ? 0 : (lo - pc[u] + cu - 1) / cu;
      const int g1 = min(nb, (hi - pc[u] + cu - 1) / cu);
      if (g0 < g1) {
        c = MmaCursor{u, 0, g0, g0, g1};
        return true;
      }
    }
    return false;
  };
  // order: expert, token group, item
  auto advance = [&](MmaCursor& c) -> bool {
    if (++c.g < c.g1) return true;
    if ((c.q + 1) * xtok < rt.off[c.u + 1] - rt.off[c.u]) {
      ++c.q;
      c.g = c.g0;
      return true;
    }
    return enter(c, c.u + 1);
  };

  MmaCursor c;
  bool ok = enter(c, first_expert(pc, U, lo));
  uint32_t i = 0;

  if (warp == NW) {  // producer
    if (lane != 0) return;
    const uint32_t bytes = (uint32_t)(2 * L.slab + 32 * nblk);
    for (; ok; ++i, ok = advance(c)) {
      const uint32_t s = i % S, r = i / S;
      if (r > 0 && !mbar_wait(empty + 8 * s, (r - 1) & 1)) {
        if (error_flag) atomicOr(error_flag, 2u);
        break;
      }
      const uint32_t st = ring + s * L.stage;
      mbar_arrive_expect_tx(full + 8 * s, bytes);
      const int row0 = rt.expert[c.u] * 2 * I + c.g * kMNeurons;  // < 2^31 (checked on launch)
      tma_load_3d(st, &tmap, 0, row0, 0, full + 8 * s);
      tma_load_3d(st + L.slab, &tmap, 0, row0 + I, 0, full + 8 * s);
      tma_load_3d(st + 2 * L.slab, &smap, 0, row0, 0, full + 8 * s);
      tma_load_3d(st + 2 * L.slab + 16 * nblk, &smap, 0, row0 + I, 0, full + 8 * s);
    }
    // the copies issued last land before the CTA exits
    for (uint32_t k = i > (uint32_t)S ? i - S : 0u; k < i; ++k)
      (void)mbar_wait(full + 8 * (k % S), (k / S) & 1);
    return;
  }

  const uint32_t red = base + L.red;
  int* ktok = reinterpret_cast<int*>(smem + L.ktok);  // [kMTokens], then rk [2][kMTokens]
  int* rk = ktok + kMTokens;

  if (warp == NW + 1) {  // epilogue: sums of the consumers' partials, bf16(SiLU(g) * u)
    const int g = lane >> 2, tig = lane & 3, t0 = 2 * tig;
    for (; ok; ++i, ok = advance(c)) {
      const uint32_t p = i & 1;
      if (!mbar_wait(rfull + 8 * p, (i >> 1) & 1)) {
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
        break;
      }
      const int T = rt.off[c.u + 1] - rt.off[c.u];
      const int* sl = rt.slots + rt.off[c.u] + c.q * xtok;
      const int nq = min(xtok, T - c.q * xtok);
      const int k0 = t0 < nq ? rk[p * kMTokens + t0] : 0;
      const int k1 = t0 + 1 < nq ? rk[p * kMTokens + t0 + 1] : 0;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float4 v = lds_f32x4(red + (uint32_t)((((p * NW + w) * 2 + r) * 32 + lane) * 16));
          sum[0] += v.x;
          sum[1] += v.y;
          sum[2] += v.z;
          sum[3] += v.w;
        }
        const int n = c.g * kMNeurons + 8 * r + slab_row(g);
        if (t0 < nq) {
          const float f = exp2_int(-(k0 >> 1)), f2 = exp2_int(-(k0 - (k0 >> 1)));
          const float gv = (sum[0] * f) * f2, uv = (sum[2] * f) * f2;
          h[(size_t)sl[t0] * I + n] = __float2bfloat16_rn(silu(gv) * uv);
        }
        if (t0 + 1 < nq) {
          const float f = exp2_int(-(k1 >> 1)), f2 = exp2_int(-(k1 - (k1 >> 1)));
          const float gv = (sum[1] * f) * f2, uv = (sum[3] * f) * f2;
          h[(size_t)sl[t0 + 1] * I + n] = __float2bfloat16_rn(silu(gv) * uv);
        }
      }
      __syncwarp();  // every lane is done with the buffer
      if (lane == 0) mbar_arrive(rempty + 8 * p);
    }
    return;
  }

  // consumers
  const int g = lane >> 2, tig = lane & 3;
  const uint32_t xs = base + L.xs, scl = base + L.scl + 128 * CB * warp;
  const uint8_t* xg = reinterpret_cast<const uint8_t*>(x) + wait_token;
  int staged_u = -1, staged_q = -1;
  bool dead = false;
  for (; ok; ++i, ok = advance(c)) {
    const uint32_t s = i % S, p = i & 1;
    const uint32_t st = ring + s * L.stage;
    const int T = rt.off[c.u + 1] - rt.off[c.u];
    const int* sl = rt.slots + rt.off[c.u] + c.q * xtok;
    const int nq = min(xtok, T - c.q * xtok);
    if (c.u != staged_u || c.q != staged_q) {
      // no consumer still reads the previous group's staged x (or its ktok)
      named_barrier_sync(1, 32 * NW);
      stage_x_f16(xs, L.xstride, ktok, xg, sl, nq, H, K, NW);
      named_barrier_sync(1, 32 * NW);
      staged_u = c.u;
      staged_q = c.q;
    }
    if (!dead && !mbar_wait(full + 8 * s, (i / S) & 1)) {
      dead = true;
      if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
    }
    float acc[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[r][k] = 0.0f;
    if (!dead) {
      const uint32_t xrow = xs + (uint32_t)((g < nq ? g : 0) * L.xstride + tig * 16);
      for (int ch = warp; ch < nchunk; ch += NW)
        mma_chunk<CB>(st, H, ch, acc, xrow + (uint32_t)(ch * 64 * CB), scl);
      __syncwarp();  // every lane is done with the stage
      if (lane == 0) mbar_arrive(empty + 8 * s);
    }
    // partial sums into buffer p, once the epilogue warp is done with it
    if (!dead && i >= 2 && !mbar_wait(rempty + 8 * p, ((i >> 1) - 1) & 1)) {
      dead = true;
      if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
    }
    if (dead) continue;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t a = red + (uint32_t)((((p * NW + warp) * 2 + r) * 32 + lane) * 16);
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(acc[r][0]),
                   "f"(acc[r][1]), "f"(acc[r][2]), "f"(acc[r][3])
                   : "memory");
    }
    if (warp == 0 && lane < nq) rk[p * kMTokens + lane] = ktok[lane];
    __syncwarp();
    if (lane == 0) mbar_arrive(rfull + 8 * p);
  }
}

namespace {

// Ring depth for H: the deepest (up to kMMaxStages) that stages 8 tokens,
// else 0 (unsupported).
int mma_stages(int H) {
  for (int S = kMMaxStages; S >= 2; --S)
    if (mma_layout(H, S).xtok >= kMTokens) return S;
  return 0;
}

}  // namespace

bool gate_up_mma_supported(int B, int H, int I, int E, int K) {
  return B * K <= kStreamMaxSlots && E <= 4096 && H % 512 == 0 && H <= 2048 &&
         I % kMNeurons == 0 && (long long)E * 2 * I < (1ll << 31) && mma_stages(H) >= 2;
}

template <int NW>
static cudaError_t launch_mma_t(const GateUpArgs& a, int S, cudaStream_t stream, bool pdl) {
  const int smem = mma_layout(a.H, S).total;
  {
    const cudaError_t e =
        ensure_dynamic_smem(reinterpret_cast<const void*>(moe_gate_up_mma<NW>), smem);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap map, smap;
  if (!encode_row_slab_map(&map, a.gate_up, (uint64_t)a.E * 2 * a.I, a.H) ||
      !encode_scale_group_map(&smap, a.gate_up_scale, (uint64_t)a.E * 2 * a.I, a.H / 32))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(32 * NW + 64);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_up_mma<NW>, map, smap,
                            reinterpret_cast<const __nv_bfloat16*>(a.x), a.topk_ids,
                            reinterpret_cast<__nv_bfloat16*>(a.h), a.error_flag,
                            a.B, a.H, a.I, a.E, a.K, S);
}

// p.cpl: ring stages (0: the deepest that fits); p.npw: consumer warps (8 or 16).
cudaError_t launch_gate_up_mma(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                               bool pdl) {
  if (!gate_up_mma_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  int S = mma_stages(a.H);
  if (p.cpl >= 2 && p.cpl < S) S = p.cpl;
  return p.npw == 16 ? launch_mma_t<16>(a, S, stream, pdl) : launch_mma_t<8>(a, S, stream, pdl);
}

}  // namespace wd
