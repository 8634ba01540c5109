// wd_launch.h - internal launch interface between the C-ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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
// Limit of the streamed variants' per-CTA routing tables (B * K).
constexpr int kStreamMaxSlots = 256;

enum GateUpVariant {
  kGateUpBatched = 0,   // moe_gate_up_3d_batched: one warp per (token, slot, neuron group)
  kGateUpRowShare = 1,  // moe_gate_up_rowshare: one warp per (expert, neuron group), all its tokens
  kGateUpStream = 2,    // moe_gate_up_stream: rows streamed by bulk copies through shared memory
  kGateUpMixed = 3,     // moe_gate_up_mixed: streamed rows, FP16 x FP16 -> FP32 products
  kGateUpPersist = 4,   // moe_gate_up_persist: one wave of CTAs over shared expert rows, x staged
  kGateUpRing = 5,      // moe_gate_up_ring: as persist, rows through a per-warp bulk-copy ring
  kGateUpTma = 6,       // moe_gate_up_tma: as persist, rows by 2-D TMA into a CTA-wide ring
  kGateUpMma = 7,       // moe_gate_up_mma: as persist, products by warp-level tensor-core MMAs
};

// Compile-time shape of one kernel instance.
struct GateUpPlan {
  int variant;  // GateUpVariant
  int npw;      // neurons per warp (gate + up rows: 2*npw rows in flight)
  int cpl;      // batched: MXFP8 blocks per lane per row per pass;
                // rowshare, persist: words (4 elements) dequantised per step, 1 or 2
};
enum DownVariant {
  kDownBatched = 0,  // moe_down_3d_batched: one warp per (token, output-dim group)
  kDownStream = 1,   // moe_down_stream: rows streamed by bulk copies, lane = token accumulator
  kDownPersist = 2,  // moe_down_3d_batched_persist: batched items walked by one wave of CTAs
  kDownShared = 3,   // moe_down_shared: CTA per output-dim group, expert rows shared by tokens
  kDownMma = 4,      // moe_down_mma: CTA per 16 output dims, products by tensor-core MMAs
  kDown3dMma = 5,    // moe_down_3d_mma: as batched, warp = (token, 16 dims), dots by MMAs
  kDownExpertMma = 6,  // moe_down_expert_mma: CTA per 16 output dims, warp per routed-expert step
};
struct DownPlan {
  int rpw;          // batched, persist: output dims per warp
  int qpl;          // batched, persist: virtual blocks per lane per pass; stream: ring stages
  int variant = 0;  // DownVariant
};

GateUpPlan plan_gate_up(int B, int H, int I, int K, int E);
DownPlan plan_down(int B, int H, int I, int K, int E);
// The plans above, downgraded to a non-streamed kernel when the bulk copies'
// 16-byte alignment does not hold for the given pointers.
GateUpPlan plan_gate_up_for(const GateUpArgs& a);
int pdl_mask_for(const GateUpPlan& g);
DownPlan plan_down_for(const DownArgs& a);

cudaError_t launch_gate_up(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream, bool pdl);
cudaError_t launch_gate_up_rowshare(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                    bool pdl);
cudaError_t launch_gate_up_stream(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                  bool pdl);
bool gate_up_stream_supported(int B, int H, int I, int E, int K, int npw);
cudaError_t launch_gate_up_mixed(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                 bool pdl);
bool gate_up_mixed_supported(int B, int H, int I, int E, int K, int npw);
cudaError_t launch_gate_up_persist(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                   bool pdl);
bool gate_up_persist_supported(int B, int H, int I, int E, int K);
cudaError_t launch_gate_up_ring(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                                bool pdl);
bool gate_up_ring_supported(int B, int H, int I, int E, int K, int stages);
cudaError_t launch_gate_up_tma(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                               bool pdl);
bool gate_up_tma_supported(int B, int H, int I, int E, int K);
cudaError_t launch_gate_up_mma(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream,
                               bool pdl);
bool gate_up_mma_supported(int B, int H, int I, int E, int K);
cudaError_t launch_down(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl);
cudaError_t launch_down_stream(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl);
bool down_stream_supported(int B, int H, int I, int E, int K);
cudaError_t launch_down_shared(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl);
bool down_shared_supported(int B, int H, int I, int E, int K, int rpw);
cudaError_t launch_down_mma(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl);
bool down_mma_supported(int B, int H, int I, int E, int K);
cudaError_t launch_down_3d_mma(const DownArgs& a, const DownPlan& p, cudaStream_t stream,
                               bool pdl);
bool down_3d_mma_supported(int B, int H, int I, int E, int K);
cudaError_t launch_down_expert_mma(const DownArgs& a, const DownPlan& p, cudaStream_t stream,
                                   bool pdl);
bool down_expert_mma_supported(int B, int H, int I, int E, int K);

}  // namespace wd
