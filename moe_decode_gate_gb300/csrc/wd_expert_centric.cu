// wd_expert_centric.cu - the expert-centric MoE layer that warp decode is
// measured against, built only for the benchmark (declared in
// include/wd_bench.h; no entry point of include/wd_moe.h reaches it).
//
// Cursor, "用 warp decode 实现更好的 MoE 模型推理", section 传统的 MoE 路径 (The
// traditional MoE path): the standard implementation organises the layer
// around experts - it collects each expert's tokens, computes, and reassembles
// the results; five of its eight stages only manage that expert-major data
// layout.  The pages name the stages warp decode removes: padding each
// expert's token list (to a power of two), scattering the activations into an
// expert-major buffer, the per-expert output buffer (8 experts x 2048 BF16 =
// 32 KB per token) and the separate combine that reduces it (sections 阶段消除
// and 消除缓冲区).  This file is that path, one kernel per stage, with the same
// arithmetic as the layer's definition except for the one rounding the
// per-expert output buffer adds (each expert's contribution is stored as
// BF16 before the weighted combine):
//   ec_route    - per-expert token counts, padded to powers of two, offsets
//                 (a block-wide scan), the routed experts' list and tile count,
//                 and each (token, slot) pair's row in the expert-major layout;
//   ec_gather   - x rows copied into the expert-major buffer X_e (zeros in
//                 padding rows);
//   ec_gate_up  - grouped GEMV: a warp per (routed expert, neuron) dequantises
//                 its gate and up rows once and applies them to every row of
//                 the expert (padding included), h_e = bf16(SiLU(g) * u);
//   ec_down     - grouped GEMV: a warp per (routed expert, output dim), into the
//                 per-expert output buffer Y_e (BF16);
//   ec_combine  - out[b,d] = bf16(sum_k w[b,k] * Y_e[row(b,k), d]), k in order.
// The grouped kernels walk a tile list built on the device (routed experts x
// 8-row groups), as a grouped GEMM scheduler does, so no host round trip is
// needed between the stages.
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/wd_bench.h"
#include "wd_device.cuh"

namespace wd {
namespace ec {

constexpr int kRouteThreads = 1024;
constexpr int kTileRows = 8;  // neurons (gate/up) or output dims (down) per CTA tile
constexpr int kTok = 4;       // expert rows per inner pass

__host__ __device__ inline size_t round256(size_t v) { return (v + 255) / 256 * 256; }

struct Layout {
  size_t meta, row_pair, pair_row, xe, he, ye, total;
  int rows_max;
};

// Workspace: meta ints [0] routed experts U, [1] padded rows, [2 .. 2+E) padded
// offsets, [2+E .. 2+2E) fill cursors, [2+2E .. 2+3E) routed experts
// ascending, [2+3E .. 2+4E) their first padded row; row_pair [rows_max] (pair
// of each row, -1 for padding); pair_row [B*K]; X_e [rows_max][H] BF16;
// h_e [rows_max][I] BF16; Y_e [rows_max][H] BF16.
__host__ __device__ inline Layout layout(int B, int H, int I, int E, int K) {
  Layout L;
  const size_t BK = (size_t)B * K;
  L.rows_max = (int)(2 * BK);  // a power-of-two pad at most doubles a list
  L.meta = 0;
  L.row_pair = round256(4 * (2 + 4 * (size_t)E));
  L.pair_row = L.row_pair + round256(4 * (size_t)L.rows_max);
  L.xe = L.pair_row + round256(4 * BK);
  L.he = L.xe + round256(2 * (size_t)L.rows_max * H);
  L.ye = L.he + round256(2 * (size_t)L.rows_max * I);
  L.total = L.ye + round256(2 * (size_t)L.rows_max * H);
  return L;
}

__device__ __forceinline__ int pad_pow2(int n) {
  if (n <= 0) return 0;
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// One CTA.  Counts, padded offsets (exclusive scan), routed-expert list, pair
// rows.  Pairs with an id outside [0, E) get no row.
__global__ void __launch_bounds__(kRouteThreads) ec_route(const int32_t* __restrict__ ids, int BK,
                                                          int E, int* __restrict__ meta,
                                                          int* __restrict__ row_pair,
                                                          int* __restrict__ pair_row, int rows_max) {
  __shared__ int cnt[4096];
  __shared__ long long part[kRouteThreads];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  for (int r = tid; r < rows_max; r += blockDim.x) row_pair[r] = -1;
  __syncthreads();
  for (int j = tid; j < BK; j += blockDim.x) {
    const int e = ids[j];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  // exclusive scan of the padded counts: each thread a contiguous run of experts
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = tid * per, e1 = min(e0 + per, E);
  long long s = 0, u = 0;
  for (int e = e0; e < e1; ++e) {
    s += pad_pow2(cnt[e]);
    u += cnt[e] > 0;
  }
  part[tid] = (s << 20) | u;  // padded rows and routed experts, both < 2^20
  __syncthreads();
  for (int off = 1; off < (int)blockDim.x; off <<= 1) {  // Hillis-Steele inclusive scan
    const long long v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  const long long before = tid > 0 ? part[tid - 1] : 0;
  int row = (int)(before >> 20), ui = (int)(before & 0xFFFFF);
  int* off = meta + 2;
  int* cur = meta + 2 + E;
  int* list = meta + 2 + 2 * E;
  int* first = meta + 2 + 3 * E;
  for (int e = e0; e < e1; ++e) {
    off[e] = row;
    cur[e] = 0;
    if (cnt[e] > 0) {
      list[ui] = e;
      first[ui] = row;
      ++ui;
    }
    row += pad_pow2(cnt[e]);
  }
  if (tid == blockDim.x - 1) {
    meta[0] = (int)(part[tid] & 0xFFFFF);
    meta[1] = (int)(part[tid] >> 20);
  }
  __syncthreads();
  for (int j = tid; j < BK; j += blockDim.x) {
    const int e = ids[j];
    if (e >= 0 && e < E) {
      const int r = off[e] + atomicAdd(&cur[e], 1);
      pair_row[j] = r;
      row_pair[r] = j;
    } else {
      pair_row[j] = -1;
    }
  }
}

// Thread per 16 bytes of a padded row: X_e[r] = x[pair / K] (zeros for padding).
__global__ void ec_gather(const uint4* __restrict__ x, const int* __restrict__ meta,
                          const int* __restrict__ row_pair, uint4* __restrict__ xe, int H, int K) {
  const int chunks = H / 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int rows = meta[1];
  if (i >= (long long)rows * chunks) return;
  const int r = (int)(i / chunks), c = (int)(i - (long long)r * chunks);
  const int j = row_pair[r];
  xe[i] = j >= 0 ? x[(size_t)(j / K) * chunks + c] : make_uint4(0u, 0u, 0u, 0u);
}

// The routed expert of tile t (tiles: routed experts x groups of kTileRows).
__device__ __forceinline__ int tile_expert(const int* meta, int E, int t, int groups, int* u) {
  *u = t / groups;
  return meta[2 + 2 * E + *u];
}

// Grid-stride over tiles; warp w of a tile owns neuron g * 8 + w of expert e:
// its lane keeps its BPL blocks of the gate and up rows in registers and
// applies them to all of the expert's padded rows, kTok rows per pass.
template <int BPL>
__global__ void __launch_bounds__(256) ec_gate_up(const uint8_t* __restrict__ gate_up,
                                                  const uint8_t* __restrict__ gate_up_scale,
                                                  const int* __restrict__ meta,
                                                  const __nv_bfloat16* __restrict__ xe,
                                                  __nv_bfloat16* __restrict__ he, int H, int I,
                                                  int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int groups = I / kTileRows, nblk = H / 32;
  const int tiles = meta[0] * groups;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    int u;
    const int e = tile_expert(meta, E, t, groups, &u);
    const int n = (t - u * groups) * kTileRows + warp;
    const int r0 = meta[2 + 3 * E + u];
    const int nr = (u + 1 < meta[0] ? meta[2 + 3 * E + u + 1] : meta[1]) - r0;
    const size_t grow = (size_t)e * 2 * I + n, urow = grow + I;
    U32x8 wg[BPL], wu[BPL];
    float sg[BPL], su[BPL];
#pragma unroll
    for (int i = 0; i < BPL; ++i) {
      const int blk = lane + 32 * i;
      if (blk < nblk) {
        wg[i] = ld_weights_32B(gate_up + grow * H + (size_t)blk * 32);
        wu[i] = ld_weights_32B(gate_up + urow * H + (size_t)blk * 32);
        sg[i] = e8m0_to_f32(ld_scale(gate_up_scale + grow * nblk + blk));
        su[i] = e8m0_to_f32(ld_scale(gate_up_scale + urow * nblk + blk));
      }
    }
    for (int q0 = 0; q0 < nr; q0 += kTok) {
      float ag[kTok], au[kTok];
#pragma unroll
      for (int q = 0; q < kTok; ++q) {
        ag[q] = au[q] = 0.0f;
        if (q0 + q < nr) {
#pragma unroll
          for (int i = 0; i < BPL; ++i) {
            const int blk = lane + 32 * i;
            if (blk < nblk) {
              const uint8_t* xr = reinterpret_cast<const uint8_t*>(xe + (size_t)(r0 + q0 + q) * H) +
                                  (size_t)blk * 64;
              float2 xf[16];
              unpack_act32(ld_act_32B(xr), ld_act_32B(xr + 32), xf);
              ag[q] = fmaf(sg[i], block_dot(wg[i], xf), ag[q]);
              au[q] = fmaf(su[i], block_dot(wu[i], xf), au[q]);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kTok; ++q) {
        const float g = warp_sum(ag[q]), v = warp_sum(au[q]);
        if (lane == 0 && q0 + q < nr)
          he[(size_t)(r0 + q0 + q) * I + n] = __float2bfloat16_rn(silu(g) * v);
      }
    }
  }
}

// Grid-stride over tiles; warp w of a tile owns output dim g * 8 + w of expert
// e: Y_e[r, d] = bf16(down row d . h_e[r]) for every padded row r.
template <int BPL>
__global__ void __launch_bounds__(256) ec_down(const uint8_t* __restrict__ down,
                                               const uint8_t* __restrict__ down_scale,
                                               const int* __restrict__ meta,
                                               const __nv_bfloat16* __restrict__ he,
                                               __nv_bfloat16* __restrict__ ye, int H, int I, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int groups = H / kTileRows, nblk = I / 32;
  const int tiles = meta[0] * groups;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    int u;
    const int e = tile_expert(meta, E, t, groups, &u);
    const int d = (t - u * groups) * kTileRows + warp;
    const int r0 = meta[2 + 3 * E + u];
    const int nr = (u + 1 < meta[0] ? meta[2 + 3 * E + u + 1] : meta[1]) - r0;
    const size_t row = (size_t)e * H + d;
    U32x8 wv[BPL];
    float sc[BPL];
#pragma unroll
    for (int i = 0; i < BPL; ++i) {
      const int blk = lane + 32 * i;
      if (blk < nblk) {
        wv[i] = ld_weights_32B(down + row * I + (size_t)blk * 32);
        sc[i] = e8m0_to_f32(ld_scale(down_scale + row * nblk + blk));
      }
    }
    for (int q0 = 0; q0 < nr; q0 += kTok) {
      float acc[kTok];
#pragma unroll
      for (int q = 0; q < kTok; ++q) {
        acc[q] = 0.0f;
        if (q0 + q < nr) {
#pragma unroll
          for (int i = 0; i < BPL; ++i) {
            const int blk = lane + 32 * i;
            if (blk < nblk) {
              const uint8_t* hr = reinterpret_cast<const uint8_t*>(he + (size_t)(r0 + q0 + q) * I) +
                                  (size_t)blk * 64;
              float2 hf[16];
              unpack_act32(ld_act_32B(hr), ld_act_32B(hr + 32), hf);
              acc[q] = fmaf(sc[i], block_dot(wv[i], hf), acc[q]);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kTok; ++q) {
        const float y = warp_sum(acc[q]);
        if (lane == 0 && q0 + q < nr) ye[(size_t)(r0 + q0 + q) * H + d] = __float2bfloat16_rn(y);
      }
    }
  }
}

// Thread per output: the weighted sum of the token's K expert outputs, k in order.
__global__ void ec_combine(const __nv_bfloat16* __restrict__ ye, const int* __restrict__ pair_row,
                           const float* __restrict__ w, __nv_bfloat16* __restrict__ out, int B,
                           int H, int K) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * H) return;
  const int b = (int)(i / H), d = (int)(i - (long long)b * H);
  float y = 0.0f;
  for (int k = 0; k < K; ++k) {
    const int r = pair_row[b * K + k];
    if (r >= 0) y = fmaf(w[b * K + k], __bfloat162float(ye[(size_t)r * H + d]), y);
  }
  out[i] = __float2bfloat16_rn(y);
}

}  // namespace ec
}  // namespace wd

extern "C" {

size_t wd_bench_expert_centric_workspace_size(int B, int H, int I, int E, int K) {
  if (B < 1 || H < 32 || I < 32 || E < 1 || K < 1 || E > 4096 || (long long)B * K > 131072 ||
      H > 4096 || I > 4096)
    return 0;
  return wd::ec::layout(B, H, I, E, K).total;
}

int wd_bench_expert_centric(const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* gate_up, const uint8_t* gate_up_scale,
                            const uint8_t* down, const uint8_t* down_scale, void* out,
                            void* workspace, size_t workspace_bytes, int B, int H, int I, int E,
                            int K, void* stream) {
  using namespace wd::ec;
  const size_t need = wd_bench_expert_centric_workspace_size(B, H, I, E, K);
  if (need == 0 || H % 32 || I % 32 || !x || !topk_ids || !topk_w || !gate_up || !gate_up_scale ||
      !down || !down_scale || !out || !workspace || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(x) & 31) ||
      (reinterpret_cast<uintptr_t>(gate_up) & 31) || (reinterpret_cast<uintptr_t>(down) & 31))
    return (int)cudaErrorInvalidValue;
  const Layout L = layout(B, H, I, E, K);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* meta = reinterpret_cast<int*>(ws + L.meta);
  int* row_pair = reinterpret_cast<int*>(ws + L.row_pair);
  int* pair_row = reinterpret_cast<int*>(ws + L.pair_row);
  auto* xe = reinterpret_cast<__nv_bfloat16*>(ws + L.xe);
  auto* he = reinterpret_cast<__nv_bfloat16*>(ws + L.he);
  auto* ye = reinterpret_cast<__nv_bfloat16*>(ws + L.ye);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int BK = B * K;
  ec_route<<<1, kRouteThreads, 0, s>>>(topk_ids, BK, E, meta, row_pair, pair_row, L.rows_max);
  const long long gchunks = (long long)L.rows_max * (H / 8);
  ec_gather<<<(unsigned)((gchunks + 255) / 256), 256, 0, s>>>(
      static_cast<const uint4*>(x), meta, row_pair, reinterpret_cast<uint4*>(xe), H, K);
  // tiles are known on the device only: enough CTAs for the largest tile count
  // seen at decode sizes, grid-striding beyond it
  const int grid = 8 * (sms > 0 ? sms : 132);
  const int bg = (H / 32 + 31) / 32, bd = (I / 32 + 31) / 32;  // blocks per lane
  if (bg == 1) ec_gate_up<1><<<grid, 256, 0, s>>>(gate_up, gate_up_scale, meta, xe, he, H, I, E);
  else if (bg == 2) ec_gate_up<2><<<grid, 256, 0, s>>>(gate_up, gate_up_scale, meta, xe, he, H, I, E);
  else ec_gate_up<4><<<grid, 256, 0, s>>>(gate_up, gate_up_scale, meta, xe, he, H, I, E);
  if (bd == 1) ec_down<1><<<grid, 256, 0, s>>>(down, down_scale, meta, he, ye, H, I, E);
  else if (bd == 2) ec_down<2><<<grid, 256, 0, s>>>(down, down_scale, meta, he, ye, H, I, E);
  else ec_down<4><<<grid, 256, 0, s>>>(down, down_scale, meta, he, ye, H, I, E);
  ec_combine<<<(unsigned)(((long long)B * H + 255) / 256), 256, 0, s>>>(
      ye, pair_row, topk_w, static_cast<__nv_bfloat16*>(out), B, H, K);
  return (int)cudaGetLastError();
}

}  // extern "C"
