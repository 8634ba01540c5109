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

// Compile-time shape of one kernel instance.
struct GateUpPlan {
  int npw;  // neurons per warp (gate + up rows: 2*npw rows in flight)
  int cpl;  // MXFP8 blocks per lane per row per pass
};
struct DownPlan {
  int rpw;  // output dims per warp
  int qpl;  // virtual blocks (over all K routed rows) per lane per pass
};

GateUpPlan plan_gate_up(int B, int H, int I, int K);
DownPlan plan_down(int B, int H, int I, int K);

cudaError_t launch_gate_up(const GateUpArgs& a, const GateUpPlan& p, cudaStream_t stream, bool pdl);
cudaError_t launch_down(const DownArgs& a, const DownPlan& p, cudaStream_t stream, bool pdl);

}  // namespace wd
