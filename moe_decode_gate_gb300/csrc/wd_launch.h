// wd_launch.h - internal launch interface between the C-ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wd_moe.h"

namespace wd {

struct GateUpArgs {
  const void* x;
  const int32_t* topk_ids;
  const uint8_t* gate_up;
  const uint8_t* gate_up_scale;
  void* h;
  uint32_t* error_flag;
  int B, H, I, E, K;
};

struct DownArgs {
  const void* h;
  const int32_t* topk_ids;
  const float* topk_w;
  const uint8_t* down;
  const uint8_t* down_scale;
  void* out;
  uint32_t* error_flag;
  int B, H, I, E, K;
};

// Limits of the shared-row gate/up variant (shared-memory routing tables).
constexpr int kRowShareMaxSlots = 2048;    // B * K
constexpr int kRowShareMaxExperts = 4096;  // E
// Limit of the per-CTA routing tables of the persistent kernels (B * K).
constexpr int kStreamMaxSlots = 256;

enum GateUpVariant {
  kGateUpBatched = 0,   // moe_gate_up_3d_batched: one warp per (token, slot, neuron group)
  kGateUpRowShare = 1,  // moe_gate_up_rowshare: one warp per (expert, neuron group), all its tokens
  kGateUpPersist = 2,   // moe_gate_up_persist: one wave of CTAs over shared expert rows, x staged
  kGateUpMma = 3,       // moe_gate_up_mma: as persist, products by warp-level tensor-core MMAs
};

// Compile-time shape of one kernel instance.
struct GateUpPlan {
  int variant;  // GateUpVariant
  int npw;      // neurons per warp (gate + up rows: 2*npw rows in flight)
  int cpl;      // batched: MXFP8 blocks per lane per row per pass;
                // rowshare, persist: words (4 elements) dequantised per step, 1 or 2
};
enum DownVariant {
  kDownBatched = 0,   // moe_down_3d_batched: one warp per (token, output-dim group)
  kDownDimBlock = 1,  // moe_h_encode + moe_down_dimblock: CTA per 16 output dims, all experts
};
struct DownPlan {
  int rpw;          // batched: output dims per warp; dimblock: step groups
  int qpl;          // batched: virtual blocks per lane per pass; dimblock: ring stages
  int variant = 0;  // DownVariant
  int pairs = 0;    // dimblock: (token, slot) pairs per step
  int split = 0;    // dimblock: consumer warps per step
};

GateUpPlan plan_gate_up(int B, int H, int I, int K, int E);
DownPlan plan_down(int B, int H, int I, int K, int E);
DownPlan batched_down_plan(int B, int I, int K);
// The plans above, downgraded to a non-streamed kernel when the bulk copies'
// 16-byte alignment does not hold for the given pointers.
GateUpPlan plan_gate_up_for(const GateUpArgs& a);
int pdl_mask_for(const GateUpPlan& g, const DownPlan& d);
int launches_for(const DownPlan& d);
DownPlan plan_down_for(const DownArgs& a);

// Scratch of one layer call: [0, 256) error flag, h BF16 [B,K,I], h FP16
// [B,K,I], per-row exponents int32 [B,K] (regions rounded to 256 bytes).
size_t layer_scratch_h_bytes(int B, int K, int I);
size_t layer_scratch_bytes(int B, int K, int I);
// The down stage of a call (pdl bit 0: its first launch, bit 1: its second).
cudaError_t launch_down_stage(const DownArgs& a, const DownPlan& p, void* h16, int32_t* hk,
                              cudaStream_t s, int pdl);
// Both stages with the built-in (or overridden) plan: every entry point that
// runs the whole layer goes through this, so they launch identical work.
cudaError_t launch_layer(const GateUpArgs& ga, const DownArgs& da, void* h16, int32_t* hk,
                         cudaStream_t s);

// WD_OK for cudaSuccess (after also checking cudaGetLastError), else
// WD_ERR_CUDA with the error's name kept for wd_last_error_string.
wd_status cuda_status(cudaError_t e);

// Raise `func`'s dynamic shared-memory limit to at least `bytes` on the current
// device (once per kernel and device; thread-safe).
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

cudaError_t launch_gate_up(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream, bool pdl);
cudaError_t launch_gate_up_rowshare(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                    bool pdl);
cudaError_t launch_gate_up_persist(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                   bool pdl);
bool gate_up_persist_supported(int B, int H, int I, int E, int K);
cudaError_t launch_gate_up_mma(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                               bool pdl);
bool gate_up_mma_supported(int B, int H, int I, int E, int K);
cudaError_t launch_down(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl);
bool down_dimblock_supported(int B, int H, int I, int E, int K);
// moe_down_dimblock's shape for I: step groups (returned), ring stages, pairs
// per step and warps per step; the wanted shape if all four are given and it
// fits, else the built-in one; 0 groups if none fits.
int down_dimblock_shape(int I, int want_ns, int want_spg, int want_p, int want_g, int* S, int* P,
                        int* G);
cudaError_t launch_h_encode(const void* h, void* h16, int32_t* hk, int rows, int I,
                            cudaStream_t stream, bool pdl);
cudaError_t launch_down_dimblock(const DownArgs& a, const DownPlan& p, const void* h16,
                                 const int32_t* hk, cudaStream_t stream, bool pdl);

}  // namespace wd
