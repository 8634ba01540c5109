// wd_persist.cuh - pieces shared by the persistent gate/up kernels
// (moe_gate_up_persist, moe_gate_up_ring, moe_gate_up_tma): routing-table layout in shared
// memory, the staged FP32 activations, the cost-balanced split of (expert,
// neuron block) items over CTAs, and the transpose-reduction epilogue.
#pragma once

#include "wd_device.cuh"
#include "wd_pipeline.cuh"
#include "wd_routing.cuh"

namespace wd {

constexpr int kPWarps = 8;
constexpr int kPThreads = 32 * kPWarps;

// Staged x starts on a 128-byte boundary after the routing tables (its
// 16-byte vector accesses need at least 16-byte alignment).
constexpr int kXOffset = (routing_table_bytes() + 127) / 128 * 128;
static_assert(kXOffset % 16 == 0 && kXOffset >= routing_table_bytes(), "staged x alignment");

// Shared-memory byte offset of 16-byte chunk c (elements 4c..4c+3) of MXFP8
// block `blk` of staged token t.  Chunks are XOR-swizzled by the low bits of
// the block index (`mask` = 7 or 3) so that the 8 lanes of a quarter-warp,
// one block each, touch 8 different 16-byte bank groups:
//   - mask 7: all lanes read the same chunk c (position c ^ (blk & 7));
//   - mask 3: lanes of odd quads read chunk c ^ 4 while the others read c (the
//     kernels that swap the halves of their weight reads); position
//     c ^ (blk & 3), so lane position = m ^ ((blk & 3) ^ 4q) = m ^ (blk & 7).
__device__ __forceinline__ uint32_t xs_chunk(uint32_t xs, int t, int H, int blk, int c, int mask) {
  return xs + (uint32_t)(t * H + blk * 32) * 4u + (uint32_t)((c ^ (blk & mask)) << 4);
}

__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds_u32x4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Sum over the warp of V values per lane (V a power of two, 2..16), by
// transpose-reduction: lane l ends with the sum of value index l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&v)[V]) {
  constexpr int L = V == 2 ? 1 : (V == 4 ? 2 : (V == 8 ? 3 : 4));
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

// Epilogue of one chunk of TC tokens x NPW neurons: acc[t][r] holds lane
// partials of row r (r < NPW: gate n0+r, else up n0+r-NPW) for token t.  The
// transpose-reduction leaves gate and up of one output in a lane pair; one
// lane stores bf16(SiLU(g) * u).
template <int NPW, int TC, int TCP>
__device__ __forceinline__ void store_chunk(const float (&acc)[TCP][2 * NPW],
                                            __nv_bfloat16* __restrict__ h,
                                            const int* __restrict__ slots, int n0, int I) {
  constexpr int R = 2 * NPW;
  constexpr int V = R * TCP;
  constexpr int L = V == 2 ? 1 : (V == 4 ? 2 : (V == 8 ? 3 : 4));
  const int lane = threadIdx.x & 31;
  float v[V];
#pragma unroll
  for (int t = 0; t < TCP; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) v[t * R + r] = acc[t][r];
  const float s = transpose_reduce<V>(v);
  // value index bit log2(NPW) (gate/up) sits at lane bit 5 - L + log2(NPW)
  const float up = __shfl_xor_sync(0xFFFFFFFFu, s, NPW << (5 - L));
  const int idx = lane >> (5 - L);
  const int t = idx / R, r = idx % R;
  if ((lane & ((1 << (5 - L)) - 1)) == 0 && r < NPW && t < TC)
    h[(size_t)slots[t] * I + n0 + r] = __float2bfloat16_rn(silu(s) * up);
}

// Cost prefix over the routed experts into pc[0..U] (an item of expert u costs
// T_u + base, and every expert has nb items); returns the total.  All threads
// of the CTA call it (it ends with a barrier).
__device__ __forceinline__ int expert_cost_prefix(const RoutingTables& rt, int nb, int base,
                                                  int* pc) {
  const int U = rt.scalar[0];
  if ((threadIdx.x >> 5) == 0) {
    const int lane = threadIdx.x & 31;
    int acc = 0;
    for (int u0 = 0; u0 < U; u0 += 32) {
      const int u = u0 + lane;
      const int c = u < U ? nb * (rt.off[u + 1] - rt.off[u] + base) : 0;
      int excl, total;
      warp_exclusive_scan(c, excl, total);
      if (u < U) pc[u] = acc + excl;
      acc += total;
    }
    if (lane == 0) pc[U] = acc;
  }
  __syncthreads();
  return pc[U];
}

// Largest routed-expert index u with pc[u] <= lo (pc strictly increasing, pc[0] = 0).
__device__ __forceinline__ int first_expert(const int* pc, int U, int lo) {
  int a = 0, b = U - 1;
  while (a < b) {
    const int m = (a + b + 1) >> 1;
    if (pc[m] <= lo) a = m; else b = m - 1;
  }
  return a;
}

// Write the x rows of tokens slots[0..nq) into shared memory as FP32,
// swizzled (xs_chunk with `mask`), with threads 0..nthreads-1 of the CTA (no
// barrier).
__device__ __forceinline__ void stage_x_rows(uint32_t xs, const uint8_t* xg, const int* slots,
                                             int nq, int H, int K, int nthreads, int mask) {
  const int per_row = H >> 2;  // 16-byte FP32 chunks per row
  const int units = nq * per_row;
  for (int i = threadIdx.x; i < units; i += nthreads) {
    const int t = i / per_row;
    const int k = i - t * per_row;  // block k >> 3, chunk k & 7
    const int b = slots[t] / K;
    const uint2 raw = *reinterpret_cast<const uint2*>(xg + ((size_t)b * H + (size_t)k * 4) * 2);
    const float2 lo = bf16x2_to_f32(raw.x), hi = bf16x2_to_f32(raw.y);
    const uint32_t a = xs_chunk(xs, t, H, k >> 3, k & 7, mask);
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(lo.x), "f"(lo.y), "f"(hi.x),
                 "f"(hi.y)
                 : "memory");
  }
}

// stage_x_rows with all threads of the CTA, between two CTA barriers (the
// previous group is no longer read before, the new one is complete after).
__device__ __forceinline__ void stage_x(uint32_t xs, const uint8_t* xg, const int* slots, int nq,
                                        int H, int K, int mask) {
  __syncthreads();
  stage_x_rows(xs, xg, slots, nq, H, K, blockDim.x, mask);
  __syncthreads();
}

// stage_x_rows for the first `nthreads` threads of the CTA only (the consumer
// warps of a warp-specialised kernel), between two named barriers `bar_id`.
__device__ __forceinline__ void stage_x_consumers(uint32_t xs, const uint8_t* xg, const int* slots,
                                                  int nq, int H, int K, int nthreads, int bar_id,
                                                  int mask) {
  named_barrier_sync(bar_id, nthreads);
  stage_x_rows(xs, xg, slots, nq, H, K, nthreads, mask);
  named_barrier_sync(bar_id, nthreads);
}

// Padded layout of staged x (moe_gate_up_persist): each 32-element block of a
// token row takes 144 bytes (32 FP32 + 16 bytes of padding), so chunk c of
// block blk sits at blk * 144 + c * 16.  Lanes on consecutive blocks reading
// the same chunk hit 16-byte bank groups (blk + c) mod 8, all different, and
// every chunk of a lane's block is an immediate offset from one address.
constexpr int kXPadBlockBytes = 144;

__host__ __device__ inline int x_padded_row_bytes(int H) { return (H / 32) * kXPadBlockBytes; }

// stage_x_rows in the padded layout, between two CTA barriers.
__device__ __forceinline__ void stage_x_padded(uint32_t xs, const uint8_t* xg, const int* slots,
                                               int nq, int H, int K) {
  __syncthreads();
  const int per_row = H >> 2;  // 16-byte FP32 chunks per row
  const int row_bytes = x_padded_row_bytes(H);
  for (int i = threadIdx.x; i < nq * per_row; i += blockDim.x) {
    const int t = i / per_row;
    const int k = i - t * per_row;  // block k >> 3, chunk k & 7
    const int b = slots[t] / K;
    const uint2 raw = *reinterpret_cast<const uint2*>(xg + ((size_t)b * H + (size_t)k * 4) * 2);
    const float2 lo = bf16x2_to_f32(raw.x), hi = bf16x2_to_f32(raw.y);
    const uint32_t a = xs + (uint32_t)(t * row_bytes + (k >> 3) * kXPadBlockBytes + (k & 7) * 16);
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(lo.x), "f"(lo.y), "f"(hi.x),
                 "f"(hi.y)
                 : "memory");
  }
  __syncthreads();
}

// Out-of-range ids: CTA 0 zeroes their h rows and raises bit 0 of the flag.
__device__ __forceinline__ void zero_bad_slots(const RoutingTables& rt, __nv_bfloat16* h,
                                               uint32_t* error_flag, int BK, int I, int E) {
  if (!rt.scalar[2] || blockIdx.x != 0) return;
  for (int s = 0; s < BK; ++s) {
    const int e = rt.ids[s];
    if (e < 0 || e >= E)
      for (int n = threadIdx.x; n < I; n += blockDim.x) h[(size_t)s * I + n] = __float2bfloat16_rn(0.0f);
  }
  if (threadIdx.x == 0 && error_flag) atomicOr(error_flag, 1u);
}

}  // namespace wd
