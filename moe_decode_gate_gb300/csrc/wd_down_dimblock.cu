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
//   - two producer threads (one per producer warp, even and odd stages)
//     stream each step's weights into an S-stage ring: the expert's 16 down
//     rows (one 3-D tensor-map copy, 128-byte swizzled so that the MMA
//     fragment reads of 8 rows hit 8 different 16-byte bank groups) and their
//     scale codes (one bulk copy of 16 x I/32 bytes).  The weights do not
//     depend on the previous kernels, so the ring fills while they drain;
//   - NS step groups of G consumer warps; group q takes the steps q, q + NS,
//     ... and owns the S / NS stages they use; each warp of a group does its
//     part of I (built-in at I = 768: 4 groups of 2 warps with 12 blocks each,
//     3 stages per group, up to 8 pairs per step).  Each lane requests its B
//     fragments from global memory one step of its group ahead (two register
//     buffers): the FP16 h row of its pair (L2-resident, written by
//     moe_h_encode), 16 bytes per block, so that the h latency overlaps the
//     previous step and h takes no room in the ring.  Per 32-column block: two k16 MMAs (E4M3 -> FP16 straight
//     into the A fragments, exact) from a zero tile, then the tile times the
//     rows' power-of-two block scales (decoded through a 256-entry table)
//     into FP32 sums;
//   - a warp's sums over its part of I are final for the step's pairs: each
//     lane stores them, unscaled, into its part's per-slot result table
//     [B*K][16] (one writer per entry, plain stores);
//   - at the end every output is y = sum over k = 0..K-1 of the slot's result
//     (its parts added in order) times w * 2^-k (the routing weight and the
//     slot's re-encoding exponent), then one BF16 store.
//
// A stage is refilled only after its group's warps released it and every
// stage is used by one step group (NS divides S) and one producer warp, in
// step order, so no wait can be more than one phase behind: the mbarrier
// phase parity is unambiguous.  Every wait is bounded (wd_pipeline.cuh); a
// warp whose wait runs out raises bit 1 of the error flag and stops; the
// producers wait (bounded) for their last copies before exiting.
#include "wd_launch.h"
#include "wd_mma.cuh"
#include "wd_persist.cuh"

namespace wd {

namespace {

constexpr int kDMaxStages = 16;    // ring stages (stages per step group x step groups)
constexpr int kDMaxWarps = 8;      // consumer warps (step groups x warps per step)
constexpr int kDMaxSplit = 4;      // consumer warps sharing one step (each a part of I)
constexpr int kDProducers = 2;     // producer warps (alternate stages)
constexpr int kDRows = 16;         // output dims per CTA
constexpr int kDMaxPairs = 8;      // (token, slot) pairs per step: one 8-column MMA tile
constexpr int kDMaxB = 64;         // tokens
constexpr int kDSmemCap = 227 * 1024;
constexpr int kDMaxSteps = kStreamMaxSlots;  // every step holds at least one pair

__host__ __device__ constexpr int d_round(int v, int a) { return (v + a - 1) / a * a; }

// Stage: [0, 16 I) the 16 down rows as [I/128][16][128] swizzled bytes;
// [16 I, 16 I + 16 I/32) their scale codes [16][I/32].  Before the ring: the
// barriers, the E8M0 decode table (256 FP32), the step list (int4 per step:
// first down row, first pair in the slot lists, pairs) and the per-slot
// results [G][B*K][16] FP32 (one table per part of I when G warps share a
// step).
struct DimLayout {
  int stage, bars, dec, steps, res, fold, ring, total;
};

__host__ __device__ inline DimLayout dim_layout(int I, int S, int G) {
  DimLayout L;
  L.stage = d_round(kDRows * I + kDRows * (I / 32), 1024);
  L.bars = kXOffset;  // full, empty [kDMaxStages] (8 bytes each)
  L.dec = L.bars + 16 * kDMaxStages;
  L.steps = L.dec + 256 * 4;
  L.res = L.steps + kDMaxSteps * 16;
  L.fold = L.res + G * kStreamMaxSlots * kDRows * 4;  // per slot: w * 2^-k split in two factors
  L.ring = d_round(L.fold + kStreamMaxSlots * 8, 1024);
  L.total = L.ring + S * L.stage;
  return L;
}

// 16 bytes of data written by an earlier kernel and not written during this
// one, through the read-only path.
__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Shared-memory loads the compiler may schedule freely (plain asm, no memory
// clobber): a stage's reads carry the token of the mbarrier wait that made it
// visible (so they cannot move above it) and the stage's release takes the
// sums computed from them as inputs (so they cannot move below it).
__device__ __forceinline__ uint32_t ld_s8(uint32_t a) {
  uint16_t v;
  asm("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float ld_sf(uint32_t a) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 ld_s64(uint32_t a) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// Arrive on `bar` once the eight sums (which depend on every read of the
// stage) exist.
__device__ __forceinline__ void mbar_arrive_after(uint32_t bar, const float (&a)[2][4]) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar), "f"(a[0][0]), "f"(a[0][1]),
               "f"(a[0][2]), "f"(a[0][3]), "f"(a[1][0]), "f"(a[1][1]), "f"(a[1][2]), "f"(a[1][3])
               : "memory");
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

// Threads: NW = NS x G consumer warps, then kDProducers producer warps.  The
// consumers form NS step groups of G warps; group q takes the steps q, q + NS,
// ... and owns the S / NS stages they use; within a group, warp part h does
// the NB 32-column blocks [h NB, (h + 1) NB) of every step (NB x G = I / 32).
// P: pairs per step (<= 8).  `tmap`: the down codes as a 3-D byte tensor
// {128, E * H, I / 128} with strides {I, 128}, boxes {128, 16, I / 128},
// 128-byte swizzle.  h16 / hk: moe_h_encode's output for the B * K rows of h.
template <int NB>
__global__ void __launch_bounds__(32 * (kDMaxWarps + kDProducers), 1) moe_down_dimblock(
    const __grid_constant__ CUtensorMap tmap, const __half* __restrict__ h16,
    const int32_t* __restrict__ hk, const int32_t* __restrict__ topk_ids,
    const float* __restrict__ topk_w, const uint8_t* __restrict__ down_scale,
    __nv_bfloat16* __restrict__ out, uint32_t* __restrict__ error_flag, int B, int H, int I,
    int E, int K, int S, int NS, int G, int P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const RoutingTables rt = routing_tables_at(smem);
  const DimLayout L = dim_layout(I, S, G);
  const int NW = NS * G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BK = B * K, nblk = I >> 5;
  const int d0 = blockIdx.x * kDRows;
  const uint32_t base = smem_u32(smem);
  const uint32_t full = base + L.bars, empty = full + 8 * kDMaxStages;
  const uint32_t ring = base + L.ring;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + 8 * s, 1);   // the producer's arrive (with the step's bytes)
      mbar_init(empty + 8 * s, G);  // the stage's consumer warps
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
    if (nsteps == 0 || lane != 0) return;
    const int p = warp - NW;
    auto mine = [&](int i) { return (i % S) % kDProducers == p; };
    const uint32_t wbytes = (uint32_t)(kDRows * I + kDRows * nblk);
    // the stage's byte count, the 16 rows and their scale codes (the weights
    // do not depend on the kernel before this one)
    auto issue = [&](uint32_t s, const int4& st_info) {
      const uint32_t st = ring + s * L.stage;
      mbar_arrive_expect_tx(full + 8 * s, wbytes);
      tma_load_3d(st, &tmap, 0, st_info.x, 0, full + 8 * s);  // row < 2^31 (checked on launch)
      bulk_g2s_nohint(st + kDRows * I, down_scale + (size_t)st_info.x * nblk,
                      (uint32_t)(kDRows * nblk), full + 8 * s);
    };
    int i = 0;
    for (; i < nsteps; ++i) {
      if (!mine(i)) continue;
      const uint32_t s = i % S;
      if (i >= S && !mbar_wait(empty + 8 * s, ((i / S) - 1) & 1)) {
        if (error_flag) atomicOr(error_flag, 2u);
        break;
      }
      issue(s, step_tab[step_at(i)]);
    }
    // the copies this warp issued last land before the CTA exits
    for (int k = i - S > 0 ? i - S : 0; k < i && k < nsteps; ++k)
      if (mine(k)) (void)mbar_wait(full + 8 * (k % S), (k / S) & 1);
    return;
  }

  // consumers: h16 and the exponents come from the kernel before this one,
  // and the writes of `out` below must follow it too
  const uint32_t wait_token = grid_dependency_wait();
  const uint8_t* hg = reinterpret_cast<const uint8_t*>(h16) + wait_token;
  // each slot's factors for the final fold, w * 2^-(k >> 1) and 2^-(k - (k >> 1)),
  // fetched now so that their latency hides behind the steps (0 for bad ids)
  float2* fold = reinterpret_cast<float2*>(smem + L.fold);
  for (int j = tid; j < BK; j += NW * 32) {
    const int e = rt.ids[j];
    float2 f = make_float2(0.0f, 0.0f);
    if (e >= 0 && e < E) {
      const int ke = __ldcg(hk + j + wait_token);
      f = make_float2(__ldg(topk_w + j) * exp2_int(-(ke >> 1)), exp2_int(-(ke - (ke >> 1))));
    }
    fold[j] = f;
  }
  const int g = lane >> 2, tig = lane & 3;
  const int pg = slab_row(g);  // the output dim (of 16) of tile rows g and g + 8
  const int grp = warp % NS, part = warp / NS;
  const int j0 = part * NB;  // this warp's first block
  const uint32_t dtab = base + L.dec;
  float* res = reinterpret_cast<float*>(smem + L.res) + part * BK * kDRows;
  // this lane's A fragment offsets within a 4-block (128-column) slab, for
  // row pg (row pg + 8 is 1024 bytes further), and its scale code offsets
  uint32_t a_off[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    a_off[u] = (uint32_t)(pg * 128 + ((((u * 2 + (tig >> 1)) ^ (pg & 7))) << 4) + (tig & 1) * 8);
  const uint32_t a_base = (uint32_t)(j0 * 512);  // slab of the first block
  const uint32_t s_off = (uint32_t)(kDRows * I + pg * nblk + j0);
  bool dead = false;
  // B fragments of step i: this lane's columns of pair g's FP16 h row, 8
  // values (16 bytes) per block, straight from global memory (written by the
  // kernel before this one, resident in L2).  They are requested one step of
  // the group ahead (two register buffers), so the L2 latency overlaps the
  // previous step's wait and MMAs.  Columns >= pairs stay zero.
  auto load_b = [&](int i, uint4 (&bf)[NB]) {
    const int4 st_info = step_tab[step_at(i)];
    const int slot_g = g < st_info.z ? rt.slots[st_info.y + g] : -1;
    if (slot_g >= 0) {
      const uint8_t* hrow = hg + (size_t)slot_g * I * 2 + (size_t)(j0 * 64 + tig * 16);
#pragma unroll
      for (int m = 0; m < NB; ++m) bf[m] = ld_global_nc_v4(hrow + m * 64);
    } else {
#pragma unroll
      for (int m = 0; m < NB; ++m) bf[m] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // step i of the group uses stage s with phase parity ph (kept incrementally:
  // the group's steps advance the stage by NS, a divisor of S)
  uint32_t s_cur = (uint32_t)grp, ph_cur = 0;
  auto step = [&](int i, const uint4 (&bf)[NB]) {
    const int4 st_info = step_tab[step_at(i)];
    const uint32_t s = s_cur, ph = ph_cur;
    s_cur += NS;
    if (s_cur >= (uint32_t)S) {
      s_cur -= S;
      ph_cur ^= 1u;
    }
    // the result rows of this lane's two pair columns, looked up before the wait
    const int pc0 = 2 * tig;
    float* r0 = pc0 < st_info.z ? res + rt.slots[st_info.y + pc0] * kDRows : nullptr;
    float* r1 = pc0 + 1 < st_info.z ? res + rt.slots[st_info.y + pc0 + 1] * kDRows : nullptr;
    bool ok;
    const uint32_t tok = mbar_wait_token(full + 8 * s, ph, ok);
    if (!ok) {
      dead = true;
      return;
    }
    const uint32_t st = ring + s * L.stage + tok;
    // two accumulators (even and odd blocks) halve the scale-FMA chain
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int m = 0; m < NB; ++m) {
      const float sc0 = ld_sf(dtab + 4 * ld_s8(st + s_off + m));
      const float sc1 = ld_sf(dtab + 4 * ld_s8(st + s_off + 8 * nblk + m));
      const uint32_t a0 = a_base + (uint32_t)((m & ~3) * 512) + a_off[m & 3];  // 2048-byte slabs
      const uint2 w0 = ld_s64(st + a0);
      const uint2 w1 = ld_s64(st + a0 + 1024);
      const uint4 b = bf[m];
      // columns 8 tig + 0..3 (first k16 step) and 8 tig + 4..7 (second)
      float cc[4];
      mma_f16_zero(cc, e4m3x2_lo_to_f16x2(w0.x), e4m3x2_lo_to_f16x2(w1.x),
                   e4m3x2_hi_to_f16x2(w0.x), e4m3x2_hi_to_f16x2(w1.x), b.x, b.y);
      mma_f16_acc(cc, e4m3x2_lo_to_f16x2(w0.y), e4m3x2_lo_to_f16x2(w1.y),
                  e4m3x2_hi_to_f16x2(w0.y), e4m3x2_hi_to_f16x2(w1.y), b.z, b.w);
      float(&a)[4] = acc[m & 1];
      a[0] = fmaf(cc[0], sc0, a[0]);
      a[1] = fmaf(cc[1], sc0, a[1]);
      a[2] = fmaf(cc[2], sc1, a[2]);
      a[3] = fmaf(cc[3], sc1, a[3]);
    }
    // every lane is done with the stage (the sums depend on all its reads)
    __syncwarp();
    if (lane == 0) mbar_arrive_after(empty + 8 * s, acc);
    // this lane's pair columns 2 tig, 2 tig + 1: its part's sums of those slots
    if (r0) {
      r0[pg] = acc[0][0] + acc[1][0];
      r0[pg + 8] = acc[0][2] + acc[1][2];
    }
    if (r1) {
      r1[pg] = acc[0][1] + acc[1][1];
      r1[pg + 8] = acc[0][3] + acc[1][3];
    }
  };
  uint4 bfa[NB], bfb[NB];
  if (grp < nsteps) load_b(grp, bfa);
  for (int i = grp; i < nsteps && !dead; i += 2 * NS) {
    if (i + NS < nsteps) load_b(i + NS, bfb);
    step(i, bfa);
    if (i + NS >= nsteps || dead) break;
    if (i + 2 * NS < nsteps) load_b(i + 2 * NS, bfa);
    step(i + NS, bfb);
  }
  if (dead && lane == 0 && error_flag) atomicOr(error_flag, 2u);
  // all slots' results are in: y = sum over k of result * w * 2^-k, k in order
  named_barrier_sync(1, NW * 32);
  res = reinterpret_cast<float*>(smem + L.res);
  for (int idx = tid; idx < kDRows * B; idx += NW * 32) {
    const int b = idx / kDRows, row = idx - b * kDRows;
    float y = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int slot = b * K + k;
      const int e = rt.ids[slot];
      if (e < 0 || e >= E) continue;
      const float2 f = fold[slot];
      float r = res[slot * kDRows + row];
      for (int h = 1; h < G; ++h) r += res[(h * BK + slot) * kDRows + row];
      y = fmaf(r * f.y, f.x, y);
    }
    out[(size_t)b * H + d0 + row] = __float2bfloat16_rn(y);
  }
}

namespace {

struct DimShape {
  int NS, S, P, G;  // step groups, ring stages (NS x stages per group), pairs per step, warps per step
};

bool dim_fits(int I, const DimShape& d) {
  const int nblk = I / 32;
  const int nb = d.G > 0 ? nblk / d.G : 0;
  return d.NS >= 1 && d.G >= 1 && d.G <= kDMaxSplit && d.NS * d.G <= kDMaxWarps && d.S >= d.NS &&
         d.S % d.NS == 0 && d.S <= kDMaxStages && d.P >= 1 && d.P <= kDMaxPairs &&
         nblk % d.G == 0 && (nb == 4 || nb == 8 || nb == 12 || nb == 16) &&
         dim_layout(I, d.S, d.G).total <= kDSmemCap;
}

// The built-in shape for I: up to four step groups, each warp of a group
// owning at most 16 blocks of 32 columns (two warps of 12 at I = 768), 8
// pairs per step, and as many stages per group as fit (three at I = 768).
DimShape dim_shape(int I, int want_ns, int want_spg, int want_p, int want_g) {
  if (want_ns > 0 && want_spg > 0 && want_p > 0 && want_g > 0) {
    const DimShape d{want_ns, want_ns * want_spg, want_p, want_g};
    if (dim_fits(I, d)) return d;
  }
  for (int g = 1; g <= kDMaxSplit; g *= 2)
    for (int ns = 4; ns >= 1; --ns)
      for (int spg = kDMaxStages / ns; spg >= 2; --spg) {
        const DimShape d{ns, ns * spg, kDMaxPairs, g};
        if (dim_fits(I, d) && d.NS * d.G <= kDMaxWarps) return d;
      }
  return DimShape{0, 0, 0, 0};
}

}  // namespace

int down_dimblock_shape(int I, int want_ns, int want_spg, int want_p, int want_g, int* S, int* P,
                        int* G) {
  const DimShape d = dim_shape(I, want_ns, want_spg, want_p, want_g);
  *S = d.S;
  *P = d.P;
  *G = d.G;
  return d.NS;
}

bool down_dimblock_supported(int B, int H, int I, int E, int K) {
  return B <= kDMaxB && B * K <= kStreamMaxSlots && E <= 4096 && H % kDRows == 0 &&
         I % 128 == 0 && I <= 4096 && (long long)E * H < (1ll << 31) &&
         dim_shape(I, 0, 0, 0, 0).NS >= 1;
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

template <int NB>
static cudaError_t launch_dimblock_t(const DownArgs& a, int S, int NS, int G, int P,
                                     const void* h16, const int32_t* hk, cudaStream_t stream,
                                     bool pdl) {
  const int smem = dim_layout(a.I, S, G).total;
  {
    const cudaError_t e =
        ensure_dynamic_smem(reinterpret_cast<const void*>(moe_down_dimblock<NB>), smem);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap map;
  if (!encode_row_slab_map(&map, a.down, (uint64_t)a.E * a.H, a.I)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.H / kDRows));
  cfg.blockDim = dim3(32 * (NS * G + kDProducers));
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_down_dimblock<NB>, map, reinterpret_cast<const __half*>(h16),
                            hk, a.topk_ids, a.topk_w, a.down_scale,
                            reinterpret_cast<__nv_bfloat16*>(a.out), a.error_flag, a.B, a.H, a.I,
                            a.E, a.K, S, NS, G, P);
}

// p.rpw: step groups, p.qpl: ring stages, p.pairs: pairs per step, p.split:
// warps per step (all resolved by the plan).  a.h is unused: the operands are
// `h16` and `hk` (moe_h_encode's output for a.h).
cudaError_t launch_down_dimblock(const DownArgs& a, const DownPlan& p, const void* h16,
                                 const int32_t* hk, cudaStream_t stream, bool pdl) {
  if (!down_dimblock_supported(a.B, a.H, a.I, a.E, a.K)) return cudaErrorInvalidValue;
  int S = 0, P = 0, G = 0;
  const int NS = down_dimblock_shape(a.I, p.rpw, p.rpw > 0 ? p.qpl / p.rpw : 0, p.pairs, p.split,
                                     &S, &P, &G);
  if (NS < 1 || S % NS != 0) return cudaErrorInvalidValue;
  switch (a.I / 32 / G) {
    case 4: return launch_dimblock_t<4>(a, S, NS, G, P, h16, hk, stream, pdl);
    case 8: return launch_dimblock_t<8>(a, S, NS, G, P, h16, hk, stream, pdl);
    case 12: return launch_dimblock_t<12>(a, S, NS, G, P, h16, hk, stream, pdl);
    case 16: return launch_dimblock_t<16>(a, S, NS, G, P, h16, hk, stream, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wd
