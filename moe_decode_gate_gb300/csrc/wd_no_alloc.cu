// wd_no_alloc.cu - wd_moe_decode_no_alloc: the MoE decode layer for callers
// that cannot allocate device memory.
//
// Some callers have no way to obtain the workspace wd_moe_decode asks for: a
// plugin inside a host framework that owns every device allocation and forbids
// new ones while it runs, or a latency-critical loop that cannot afford
// cudaMalloc's possible implicit device synchronisation.  This entry point
// keeps the layer's scratch (the BF16 intermediate h and, for batches whose
// tokens share experts, its FP16 re-encoding with per-row exponents) in a
// fixed-size array compiled into the library instead, laid out exactly as a
// workspace, so the caller passes only inputs and outputs and the call runs
// the same kernels, in the same order, as wd_moe_decode.
//
// Costs of that choice, all documented in include/wd_moe.h:
//   - every GPU that loads the library holds kNoAllocScratchBytes (2 MiB) for
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

// 2 MiB: the workspace layout of wd_moe_decode for up to B = 85 tokens at K = 8, I = 768
static constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;

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
  // the workspace layout for this call must fit the compiled-in scratch
  const size_t hb = wd::layer_scratch_h_bytes(B, K, I);
  if (wd::layer_scratch_bytes(B, K, I) > kNoAllocScratchBytes) return WD_ERR_WORKSPACE_TOO_SMALL;

  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return wd::cuda_status(e);
  uint8_t* b8 = static_cast<uint8_t*>(base);
  void* h = b8 + 256;
  // Nothing in the scratch needs clearing: every kernel writes each element
  // the next one reads (zeros for out-of-range ids).  No error flag is kept:
  // out-of-range ids contribute nothing and are not reported, and a bounded
  // wait that runs out inside a kernel is not reported either.
  const wd::GateUpArgs ga{x, topk_ids, gate_up, gate_up_scale, h, nullptr, B, H, I, E, K};
  const wd::DownArgs da{h, topk_ids, topk_w, down, down_scale, out, nullptr, B, H, I, E, K};
  return wd::cuda_status(wd::launch_layer(ga, da, b8 + 256 + hb,
                                          reinterpret_cast<int32_t*>(b8 + 256 + 2 * hb),
                                          reinterpret_cast<cudaStream_t>(stream)));
}
