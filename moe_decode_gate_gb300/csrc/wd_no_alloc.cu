// wd_no_alloc.cu - wd_moe_decode_no_alloc: the MoE decode layer for callers
// that cannot allocate device memory.
//
// Some callers have no way to obtain the workspace wd_moe_decode asks for: a
// plugin inside a host framework that owns every device allocation and forbids
// new ones while it runs, or a latency-critical loop that cannot afford
// cudaMalloc's possible implicit device synchronisation.  This entry point
// keeps the layer's one scratch buffer (the BF16 intermediate h) in a
// fixed-size array compiled into the library instead, so the caller passes
// only inputs and outputs.
//
// Costs of that choice, all documented in include/wd_moe.h:
//   - every GPU that loads the library holds kNoAllocScratchBytes (1 MiB) for
//     the life of the process, used or not;
//   - all calls share the one array, so calls that may run at the same time on
//     the GPU (different streams, no ordering between them) race on it;
//   - the array's device address is looked up once per device, on the first
//     call made with that device current.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/wd_moe.h"
#include "wd_launch.h"

static constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB: h for B*K*I <= 524288

// The scratch itself.  In host code this name is only a stand-in for the
// device object, not an address a kernel can use; the kernels get the address
// that cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_no_alloc_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" wd_status wd_moe_decode_no_alloc(const void* x, const int32_t* topk_ids,
                                            const float* topk_w, const uint8_t* gate_up,
                                            const uint8_t* gate_up_scale, const uint8_t* down,
                                            const uint8_t* down_scale, void* out, int B, int H,
                                            int I, int E, int K, wd_stream_t stream) {
  if (B < 1 || B > 4096 || K < 1 || K > 64 || E < 1 || K > E) return WD_ERR_INVALID_ARG;
  if (H < 32 || I < 32 || H % 32 || I % 32 || H > 16384 || I > 16384)
    return WD_ERR_UNSUPPORTED_SHAPE;
  if (!x || !topk_ids || !topk_w || !gate_up || !gate_up_scale || !down || !down_scale || !out)
    return WD_ERR_INVALID_ARG;
  if (!aligned(x, 32) || !aligned(gate_up, 32) || !aligned(down, 32) || !aligned(topk_ids, 4) ||
      !aligned(topk_w, 4) || !aligned(out, 4))
    return WD_ERR_INVALID_ARG;
  // h is BF16 [B, K, I]; it must fit the compiled-in scratch
  if ((size_t)B * K * I * 2 > kNoAllocScratchBytes) return WD_ERR_WORKSPACE_TOO_SMALL;

  void* h = nullptr;
  if (scratch_address(&h) != cudaSuccess) return WD_ERR_CUDA;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Nothing in the scratch needs clearing: the first kernel writes every h
  // element the second kernel reads (zeros for out-of-range ids).  No error
  // flag is kept: out-of-range ids contribute nothing and are not reported.
  const wd::GateUpArgs ga{x, topk_ids, gate_up, gate_up_scale, h, nullptr, B, H, I, E, K};
  const wd::GateUpPlan gp = wd::plan_gate_up_for(ga);
  const int pdl = wd::pdl_mask_for(gp);
  cudaError_t e = wd::launch_gate_up(ga, gp, s, (pdl & 1) != 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return WD_ERR_CUDA;
  const wd::DownArgs da{h, topk_ids, topk_w, down, down_scale, out, nullptr, B, H, I, E, K};
  e = wd::launch_down(da, wd::plan_down_for(da), s, (pdl & 2) != 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? WD_OK : WD_ERR_CUDA;
}
