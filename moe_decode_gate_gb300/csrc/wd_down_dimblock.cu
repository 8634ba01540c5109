// wd_down_dimblock.cu - the down projection for batches whose tokens share
// experts: moe_h_encode (the intermediate h re-encoded once per call) and
// moe_down_dimblock (one CTA per 16 output dims over every routed expert, the
// products on the tensor cores).
//
// Computes what moe_down_3d_batched computes (Cursor, "用 warp decode 实现更好的
// MoE 模型推理", section 两个 kernel 如何工作, down paragraph): for every token
// b and output dim d, y = sum_k w[b,k] * (down row d of expert e_k) . h[b,k,:],
// folded over k = 0..K-1 in that order, out[b,d] = bf16(y), each output
// written once by the one CTA that owns it, with no padding, no scatter into
// expert-major buffers and no combine pass.
//
// Why a different organisation at B >= 8.  The pages' mapping (one warp per
// (token, output dim)) re-reads and re-dequantises a routed row for every
// (token, slot) that uses it: at B = 32 about 2.3 times per row, which makes
// that kernel bound by instruction issue and L2, not HBM.  Here each routed
// row is read from HBM and dequantised once per call, and the products of one
// row with all (token, slot) pairs routed to its expert are one m16n8k16 MMA
// column tile.
//
// moe_h_encode: one warp per (token, slot) row of h: the row's largest
// magnitude fixes a power of two 2^k that puts it in [2^14, 2^15); the row is
// written as FP16 h * 2^k next to k.  Power-of-two scaling is exact and every
// BF16 value within 2^31 of the row's largest magnitude is an FP16 value after
// it; smaller ones are rounded to a 2^-38 grid of that magnitude, below the
// rounding of the FP32 accumulation.  Done once per call instead of once per
// (CTA, step): the down kernel's operands are then plain copies.
//
// moe_down_dimblock organisation:
//   - grid: one CTA per 16 output dims (H / 16 CTAs); each builds the routing
//     tables (routed experts ascending, each with its (token, slot) list) and
//     walks every routed expert in steps of up to P pairs, so every CTA does
//     the same amount of work.  CTA c starts its walk at its own point of the
//     step list (c / gridDim of the way in) and wraps around, so the CTAs read
//     different experts' rows at any moment;
//   - two producer warps (even and odd stages: a step's copies cost the
//     issuing thread a few hundred cycles) stream each step into the ring: the
//     expert's 16 down rows (one 3-D tensor-map copy, 128-byte swizzled so
//     that the MMA fragment reads of 8 rows hit 8 different 16-byte bank
//     groups), their scale codes (one bulk copy of 16 x I/32 bytes) and the
//     pairs' FP16 h rows (one bulk copy per pair, issued by as many lanes).
//     The first S steps' weights are requested before the kernel waits for
//     the grid that writes h, so the ring fills while the previous kernels
//     drain;
//   - NW consumer warps; warp w takes the steps w, w + NW, ... whole and owns
//     the S / NW stages they use (built-in: 4 warps, 2 stages each, up to 6
//     pairs per step).  Per 32-column block: two k16 MMAs
//     (E4M3 -> FP16 straight into the A fragments, exact) from a zero tile,
//     then the tile times the rows' power-of-two block scales (decoded through
//     a 256-entry table) into FP32 sums.  A step is I / 32 independent block
//     chains, enough work in flight for one warp per scheduler;
//   - a step's sums are final for its pairs: each lane stores them, unscaled,
//     into the per-slot result table [B*K][16] (one writer per entry, plain
//     stores);
//   - at the end every output is y = sum over k = 0..K-1 of the slot's result
//     times w * 2^-k (the routing weight and the slot's re-encoding exponent),
//     then one BF16 store.
//
// A stage is refilled only after its consumer warp released it and every
// stage is used by one consumer warp (NW divides S) and one producer warp, in
// step order, so no wait can be more than one phase behind: the mbarrier
// phase parity is unambiguous.  Every wait is bounded
// (wd_pipeline.cuh); a warp whose wait runs out raises bit 1 of the error flag
// and stops; the producers wait (bounded) for their last copies before
// exiting.
#include "wd_launch.h"
#include "wd_mma.cuh"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kDMaxStages = 16;    // ring stages (stages per consumer warp x consumer warps)
constexpr int kDMaxWarps = 8;      // consumer warps
constexpr int kDProducers = 2;     // producer warps (alternate stages)
constexpr int kDRows = 16;         // output dims per CTA
constexpr int kDMaxPairs = 8;      // (token, slot) pairs per step: one 8-column MMA tile
constexpr int kDMaxB = 64;         // tokens
constexpr int kDSmemCap = 227 * 1024;
constexpr int kDMaxSteps = kStreamMaxSlots;  // every step holds at least one pair

__host__ __device__ constexpr int d_round(int v, int a) { return (v + a - 1) / a * a; }

// Stage: [0, 16 I) the 16 down rows as [I/128][16][128] swizzled bytes;
// [16 I, 16 I + 16 I/32) their scale codes [16][I/32]; from `hoff` the pairs'
// FP16 h rows (up to P of them), `hpitch` apart.  Before the ring: the barriers, the E8M0 decode
// table (256 FP32), the step list (int4 per step: first down row, first pair
// in the slot lists, pairs) and the per-slot results [B*K][16] FP32.
struct DimLayout {
  int hoff, hpitch, stage, bars, dec, steps, res, ring, total;
};

__host__ __device__ inline DimLayout dim_layout(int I, int S, int P) {
  DimLayout L;
  L.hoff = d_round(kDRows * I + kDRows * (I / 32), 16);
  // FP16 row rounded up to 128 bytes, plus 64: the two pair rows read by one
  // quarter-warp fall in different halves of the 32 banks
  L.hpitch = d_round(2 * I, 128) + 64;
  L.stage = d_round(L.hoff + P * L.hpitch, 1024);
  L.bars = kXOffset;  // full, empty [kDMaxStages] (8 bytes each)
  L.dec = L.bars + 16 * kDMaxStages;
  L.steps = L.dec + 256 * 4;
  L.res = L.steps + kDMaxSteps * 16;
  L.ring = d_round(L.res + kStreamMaxSlots * kDRows * 4, 1024);
  L.total = L.ring + S * L.stage;
  return L;
}

}  // namespace

// One warp per row r < rows of h (BF16 [rows][I]): h16[r] = FP16(h[r] * 2^k),
// hk[r] = k (largest magnitude of the row in [2^14, 2^15); 0 for a row that is
// all zero or holds Inf or NaN).  Rows of up to 2048 values are held in
// registers between the two passes; longer ones are read twice.
__global__ void __launch_bounds__(64) moe_h_encode(const __nv_bfloat16* __restrict__ h,
                                                   __half* __restrict__ h16,
                                                   int32_t* __restrict__ hk, int rows, int I) {
  // h is written by the kernel before this one on the stream
  const uint32_t wait_token = grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(h) + (size_t)r * I * 2 + wait_token;
  uint8_t* dst = reinterpret_cast<uint8_t*>(h16) + (size_t)r * I * 2;
  const int nch = I >> 3;  // 16-byte chunks of 8 values
  constexpr int kHeld = 8;  // chunks per lane kept in registers (I <= 2048)
  uint4 held[kHeld];
  uint32_t mx = 0u;
#pragma unroll
  for (int q = 0; q < kHeld; ++q) {
    const int ch = lane + 32 * q;
    held[q] = ch < nch ? ld_act_16B(src + ch * 16) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 w = held[q];
    mx = max(mx, max(max(max_abs_bf16x2(w.x), max_abs_bf16x2(w.y)),
                     max(max_abs_bf16x2(w.z), max_abs_bf16x2(w.w))));
  }
  for (int ch = lane + 32 * kHeld; ch < nch; ch += 32) {
    const uint4 w = ld_act_16B(src + ch * 16);
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
  auto encode = [&](const uint4& w) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = bf16x2_to_f32(in[q]);
      const __half2 hv = __floats2half2_rn((f.x * f1) * f2, (f.y * f1) * f2);
      o[q] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
#pragma unroll
  for (int q = 0; q < kHeld; ++q) {
    const int ch = lane + 32 * q;
    if (ch < nch) *reinterpret_cast<uint4*>(dst + ch * 16) = encode(held[q]);
  }
  for (int ch = lane + 32 * kHeld; ch < nch; ch += 32)
    *reinterpret_cast<uint4*>(dst + ch * 16) = encode(ld_act_16B(src + ch * 16));
  if (lane == 0) hk[r] = k;
}

// Threads: NW consumer warps (each owning S / NW stages), then kDProducers
// producer warps.  P: pairs per step (<= 8).
// `tmap`: the down codes as a 3-D byte tensor {128, E * H, I / 128} with
// strides {I, 128}, boxes {128, 16, I / 128}, 128-byte swizzle.  h16 / hk:
// moe_h_encode's output for the B * K rows of h.
__global__ void __launch_bounds__(32 * (kDMaxWarps + kDProducers), 1) moe_down_dimblock(
    const __grid_constant__ CUtensorMap tmap, const __half* __restrict__ h16,
    const int32_t* __restrict__ hk, const int32_t* __restrict__ topk_ids,
    const float* __restrict__ topk_w, const uint8_t* __restrict__ down_scale,
    __nv_bfloat16* __restrict__ out, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K, int S, int NW, int P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const DimLayout L = dim_layout(I, S, P);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K, nblk = I >> 5;
  const int d0 = blockIdx.x * kDRows;
  const uint32_t base = smem_u32(smem);
  const uint32_t full = base + L.bars, empty = full + 8 * kDMaxStages;
  const uint32_t ring = base + L.ring;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + 8 * s, 1);   // the producer's arrive (with the step's bytes)
      mbar_init(empty + 8 * s, 1);  // the stage's consumer warp
    }
    mbar_init_fence();
  }
  for (int c = tid; c < 256; c += blockDim.x)
    reinterpret_cast<float*>(smem + L.dec)[c] = e8m0_to_f32((uint32_t)c);
  // The routing is the call's input; h16 and hk are written by the kernel
  // before this one, and only their reads wait for it.
  build_routing_tables(rt, topk_ids, BK, E, P, blockDim.x);  // ends with a CTA barrier
  if (rt.scalar[2] && blockIdx.x == 0 && tid == 0 && error_flag) atomicOr(error_flag, 1u);
  // step c: chunk c of the routing tables (up to P pairs of one routed expert)
  const int nsteps = rt.scalar[1];
  for (int c = tid; c < nsteps; c += blockDim.x) {
    const int u = rt.chunk_u[c];
    const int first = rt.off[u] + (c - rt.coff[u]) * P;
    reinterpret_cast<int4*>(smem + L.steps)[c] =
        make_int4(rt.expert[u] * H + d0, first, min(P, rt.off[u + 1] - first), 0);
  }
  __syncthreads();
  const int4* step_tab = reinterpret_cast<const int4*>(smem + L.steps);
  // CTA c walks the steps from step c * nsteps / gridDim on, wrapping around
  const int rot = (int)(((long long)blockIdx.x * nsteps) / gridDim.x);
  auto step_at = [&](int i) -> int { const int t = i + rot; return t < nsteps ? t : t - nsteps; };

  if (warp >= NW) {  // producers: warp NW + p issues the steps whose stage s has s % 2 == p
    if (nsteps == 0) return;
    const int p = warp - NW;
    auto mine = [&](int i) { return (i % S) % kDProducers == p; };
    const uint32_t wbytes = (uint32_t)(kDRows * I + kDRows * nblk);
    const uint8_t* hg = nullptr;
    // lane 0: the stage's byte count, the 16 rows and their scale codes
    auto issue_weights = [&](uint32_t s, const int4& st_info) {
      const uint32_t st = ring + s * L.stage;
      mbar_arrive_expect_tx(full + 8 * s, wbytes + (uint32_t)(st_info.z * 2 * I));
      tma_load_3d(st, &tmap, 0, st_info.x, 0, full + 8 * s);  // row < 2^31 (checked on launch)
      bulk_g2s_nohint(st + kDRows * I, down_scale + (size_t)st_info.x * nblk,
                      (uint32_t)(kDRows * nblk), full + 8 * s);
    };
    // lane t < pairs: pair t's FP16 h row
    auto issue_h = [&](uint32_t s, const int4& st_info) {
      if (lane < st_info.z)
        bulk_g2s_nohint(ring + s * L.stage + L.hoff + lane * L.hpitch,
                        hg + (size_t)rt.slots[st_info.y + lane] * I * 2, (uint32_t)(2 * I),
                        full + 8 * s);
    };
    const int npre = min(S, nsteps);
    // the first S steps' weights go out before waiting for the grid that writes h16
    if (lane == 0)
      for (int i = 0; i < npre; ++i)
        if (mine(i)) issue_weights(i, step_tab[step_at(i)]);
    hg = reinterpret_cast<const uint8_t*>(h16) + grid_dependency_wait();
    __syncwarp();
    for (int i = 0; i < npre; ++i)
      if (mine(i)) issue_h(i, step_tab[step_at(i)]);
    int i = npre;
    for (; i < nsteps; ++i) {
      if (!mine(i)) continue;
      const uint32_t s = i % S, r = i / S;  // r >= 1 here
      const int4 st_info = step_tab[step_at(i)];
      bool free = true;
      if (lane == 0) free = mbar_wait(empty + 8 * s, (r - 1) & 1);
      if (!__shfl_sync(0xFFFFFFFFu, free ? 1 : 0, 0)) {
        if (lane == 0 && error_flag) atomicOr(error_flag, 2u);
        break;
      }
      if (lane == 0) issue_weights(s, st_info);
      __syncwarp();
      issue_h(s, st_info);
    }
    if (lane == 0)  // the copies this warp issued last land before the CTA exits
      for (int k = i - S > 0 ? i - S : 0; k < i && k < nsteps; ++k)
        if (mine(k)) (void)mbar_wait(full + 8 * (k % S), (k / S) & 1);
    return;
  }

  // consumers: the routing weights and exponents are read at the end, after
  // the wait for the kernel that writes the exponents (which also orders the
  // writes of `out` after it)
  const uint32_t wait_token = grid_dependency_wait();
  const int g = lane >> 2, tig = lane & 3;
  const int pg = slab_row(g);  // the output dim (of 16) of tile rows g and g + 8
  const float* dtab = reinterpret_cast<const float*>(smem + L.dec);
  float* res = reinterpret_cast<float*>(smem + L.res);
  // this lane's A fragment offsets within a 4-block (128-column) slab, for
  // row pg (row pg + 8 is 1024 bytes further); B and scale offsets at block 0
  uint32_t a_off[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    a_off[u] = (uint32_t)(pg * 128 + ((((u * 2 + (tig >> 1)) ^ (pg & 7))) << 4) + (tig & 1) * 8);
  // B fragment rows: pair g; the tile's columns P..7 hold no pair and are
  // never stored, so their lanes read the last pair row (inside the stage)
  const uint32_t b_off = (uint32_t)(L.hoff + min(g, P - 1) * L.hpitch + tig * 16);
  const uint32_t s_off = (uint32_t)(kDRows * I + pg * nblk);
  bool dead = false;
  for (int i = warp; i < nsteps; i += NW) {
    const uint32_t s = i % S;
    if (!mbar_wait(full + 8 * s, (i / S) & 1)) {
      dead = true;
      break;
    }
    const uint8_t* st = smem + L.ring + s * L.stage;
    // two accumulators (even and odd blocks) halve the scale-FMA chain
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int j4 = 0; j4 < nblk; j4 += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j4 + u;
        const float sc0 = dtab[st[s_off + j]];
        const float sc1 = dtab[st[s_off + 8 * nblk + j]];
        const uint32_t a0 = (uint32_t)(j4 * 512) + a_off[u];  // slab j4 / 4, 2048 bytes each
        const uint2 w0 = *reinterpret_cast<const uint2*>(st + a0);
        const uint2 w1 = *reinterpret_cast<const uint2*>(st + a0 + 1024);
        const uint4 b = *reinterpret_cast<const uint4*>(st + b_off + j * 64);
        // columns 8 tig + 0..3 (first k16 step) and 8 tig + 4..7 (second)
        float cc[4];
        mma_f16_zero(cc, e4m3x2_lo_to_f16x2(w0.x), e4m3x2_lo_to_f16x2(w1.x),
                     e4m3x2_hi_to_f16x2(w0.x), e4m3x2_hi_to_f16x2(w1.x), b.x, b.y);
        mma_f16_acc(cc, e4m3x2_lo_to_f16x2(w0.y), e4m3x2_lo_to_f16x2(w1.y),
                    e4m3x2_hi_to_f16x2(w0.y), e4m3x2_hi_to_f16x2(w1.y), b.z, b.w);
        float(&a)[4] = acc[u & 1];
        a[0] = fmaf(cc[0], sc0, a[0]);
        a[1] = fmaf(cc[1], sc0, a[1]);
        a[2] = fmaf(cc[2], sc1, a[2]);
        a[3] = fmaf(cc[3], sc1, a[3]);
      }
    }
    // every lane is done with the stage (the sums depend on all its reads)
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + 8 * s);
    // this lane's pair columns 2 tig, 2 tig + 1: final sums of those slots
    const int4 st_info = step_tab[step_at(i)];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int pc = 2 * tig + q;
      if (pc < st_info.z) {
        float* r = res + rt.slots[st_info.y + pc] * kDRows;
        r[pg] = acc[0][q] + acc[1][q];
        r[pg + 8] = acc[0][2 + q] + acc[1][2 + q];
      }
    }
  }
  if (dead && lane == 0 && error_flag) atomicOr(error_flag, 2u);
  // all slots' results are in: y = sum over k of result * w * 2^-k, k in order
  named_barrier_sync(1, NW * 32);
  for (int idx = tid; idx < kDRows * B; idx += NW * 32) {
    const int b = idx / kDRows, row = idx - b * kDRows;
    float y = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int slot = b * K + k;
      const int e = rt.ids[slot];
      if (e < 0 || e >= E) continue;
      const int ke = __ldcg(hk + slot + wait_token);
      const float f1 = exp2_int(-(ke >> 1)), f2 = exp2_int(-(ke - (ke >> 1)));
      y = fmaf((res[slot * kDRows + row] * f1) * f2, __ldg(topk_w + slot), y);
    }
    out[(size_t)b * H + d0 + row] = __float2bfloat16_rn(y);
  }
}

namespace {

struct DimShape {
  int NW, S, P;  // consumer warps, ring stages (NW x stages per warp), pairs per step
};

// The built-in shape for I: four consumer warps with two stages each and six
// pairs per step (at I = 768), else the largest of those that fits.
DimShape dim_shape(int I, int want_nw, int want_spw, int want_p) {
  if (want_nw > 0 && want_spw > 0 && want_p > 0) {
    const DimShape d{want_nw, want_nw * want_spw, want_p};
    if (d.NW <= kDMaxWarps && d.S <= kDMaxStages && d.P <= kDMaxPairs &&
        dim_layout(I, d.S, d.P).total <= kDSmemCap)
      return d;
  }
  for (int nw = 4; nw >= 1; --nw)
    if (dim_layout(I, 2 * nw, 6).total <= kDSmemCap) return DimShape{nw, 2 * nw, 6};
  return DimShape{0, 0, 0};
}

}  // namespace

int down_dimblock_shape(int I, int want_nw, int want_spw, int want_p, int* S, int* P) {
  const DimShape d = dim_shape(I, want_nw, want_spw, want_p);
  *S = d.S;
  *P = d.P;
  return d.NW;
}

bool down_dimblock_supported(int B, int H, int I, int E, int K) {
  return B <= kDMaxB && B * K <= kStreamMaxSlots && E <= 4096 && H % kDRows == 0 &&
         I % 128 == 0 && I <= 4096 && (long long)E * H < (1ll << 31) &&
         dim_shape(I, 0, 0, 0).NW >= 1;
}

cudaError_t launch_h_encode(const void* h, void* h16, int32_t* hk, int rows, int I,
                            cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + 1) / 2));
  cfg.blockDim = dim3(64);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_h_encode, reinterpret_cast<const __nv_bfloat16*>(h),
                            reinterpret_cast<__half*>(h16), hk, rows, I);
}

// p.rpw: consumer warps, p.qpl: ring stages, p.pairs: pairs per step (all
// resolved by the plan).  a.h is unused: the operands are `h16` and `hk`
// (moe_h_encode's output for a.h).
cudaError_t launch_down_dimblock(const DownArgs& a, const DownPlan& p, const void* h16,
                                 const int32_t* hk, cudaStream_t stream, bool pdl) {
  if (!down_dimblock_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  int S = 0, P = 0;
  const int NW = down_dimblock_shape(a.I, p.rpw, p.rpw > 0 ? p.qpl / p.rpw : 0, p.pairs, &S, &P);
  if (NW < 1 || S % NW != 0) return cudaErrorInvalidValue;
  const int smem = dim_layout(a.I, S, P).total;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(moe_down_dimblock), smem);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap map;
  if (!encode_row_slab_map(&map, a.down, (uint64_t)a.E * a.H, a.I)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.H / kDRows));
  cfg.blockDim = dim3(32 * (NW + kDProducers));
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_dimblock, map, reinterpret_cast<const __half*>(h16), hk,
                            a.topk_ids, a.topk_w, a.down_scale,
                            reinterpret_cast<__nv_bfloat16*>(a.out), a.error_flag, a.B, a.H, a.I,
                            a.E, a.K, S, NW, P);
}

}  // namespace wd
