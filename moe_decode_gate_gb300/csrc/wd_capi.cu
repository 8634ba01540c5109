// wd_capi.cu - the C-ABI of the MoE decode layer (declared in include/wd_moe.h).
//
// Host-side argument checks, the per-shape launch plan, and the two launches.
// Nothing here allocates or synchronises except wd_moe_read_error_flag, which
// is documented to synchronise.
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/wd_moe.h"
#include "wd_launch.h"

namespace wd {

// Launch plan.  The batched gate/up kernel keeps 2*npw rows of H bytes in
// flight per warp and does ceil(H/32/32) blocks per lane in passes of cpl; the
// shared-row variants serve every token of an expert from one dequantised row
// and are used once tokens start to share experts.  The down kernel spreads the
// K*I/32 blocks of the K routed rows over the lanes in passes of qpl per lane.
//
// wd_moe_set_plan (or the WD_PLAN environment variable, read at the first
// call) overrides the choice for tuning sweeps and tests:
//   "gu=batched:<npw>:<cpl>" | "gu=rowshare:<npw>:<sbw>" | "gu=persist:<npw>:<prefetch+1>" |
//   "gu=mma[:<stages>[:<consumer warps, 8 or 16>]]",
//   "dn=<rpw>:<qpl>" |
//   "dn=dimblock[:<step groups>:<stages per group>:<pairs per step>:<warps per step>]",
//   "rowshare_min_b=<B>", "pdl=<mask>" (bit i: launch i of the call may overlap
//   the launch before it), comma-separated; "" or NULL restores the defaults.
namespace {

struct PlanOverride {
  int gu_variant = -1, gu_npw = 0, gu_cpl = 0;
  int dn_variant = -1, dn_rpw = 0, dn_qpl = 0, dn_pairs = 0, dn_split = 0;
  int rowshare_min_b = 16;  // shared-row kernel where the persistent one does not apply
  int pdl_mask = -1;        // -1: by the plan (pdl_mask_for)
};

bool parse_plan(const char* spec, PlanOverride* out) {
  PlanOverride p;
  if (spec && *spec) {
    char buf[256];
    strncpy(buf, spec, sizeof(buf) - 1);
    buf[sizeof(buf) - 1] = 0;
    char* save = nullptr;
    for (char* tok = strtok_r(buf, ",", &save); tok; tok = strtok_r(nullptr, ",", &save)) {
      int a = 0, b = 0;
      if (int n = 0; sscanf(tok, "gu=batched:%d:%d%n", &a, &b, &n) == 2 && tok[n] == 0) {
        p.gu_variant = kGateUpBatched;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (sscanf(tok, "gu=mma:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpMma;
        p.gu_npw = b;
        p.gu_cpl = a;
      } else if (sscanf(tok, "gu=mma:%d", &a) == 1) {
        p.gu_variant = kGateUpMma;
        p.gu_npw = 8;
        p.gu_cpl = a;
      } else if (strcmp(tok, "gu=mma") == 0) {
        p.gu_variant = kGateUpMma;
        p.gu_npw = 8;
        p.gu_cpl = 0;
      } else if (sscanf(tok, "gu=persist:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpPersist;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (sscanf(tok, "gu=rowshare:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpRowShare;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (int c = 0, d = 0, n = 0;
                 sscanf(tok, "dn=dimblock:%d:%d:%d:%d%n", &a, &b, &c, &d, &n) == 4 && tok[n] == 0) {
        p.dn_variant = kDownDimBlock;
        p.dn_rpw = a;
        p.dn_qpl = b;
        p.dn_pairs = c;
        p.dn_split = d;
      } else if (strcmp(tok, "dn=dimblock") == 0) {
        p.dn_variant = kDownDimBlock;
        p.dn_qpl = 0;
        p.dn_rpw = 0;
        p.dn_pairs = 0;
        p.dn_split = 0;
      } else if (sscanf(tok, "dn=%d:%d", &a, &b) == 2) {
        p.dn_variant = kDownBatched;
        p.dn_rpw = a;
        p.dn_qpl = b;
      } else if (sscanf(tok, "rowshare_min_b=%d", &a) == 1) {
        p.rowshare_min_b = a;
      } else if (sscanf(tok, "pdl=%d", &a) == 1 && a >= 0 && a <= 7) {
        p.pdl_mask = a;
      } else {
        return false;
      }
    }
  }
  *out = p;
  return true;
}

PlanOverride& plan_override() {
  static PlanOverride o = [] {
    PlanOverride p;
    parse_plan(getenv("WD_PLAN"), &p);
    return p;
  }();
  return o;
}

}  // namespace

GateUpPlan plan_gate_up(int B, int H, int I, int K, int E) {
  const PlanOverride& o = plan_override();
  const bool rowshare_ok = B * K <= kRowShareMaxSlots && E <= kRowShareMaxExperts;
  if (o.gu_variant == kGateUpRowShare && rowshare_ok) return {kGateUpRowShare, o.gu_npw, o.gu_cpl};
  if (o.gu_variant == kGateUpPersist && gate_up_persist_supported(B, H, I, E, K))
    return {kGateUpPersist, o.gu_npw, o.gu_cpl};
  if (o.gu_variant == kGateUpMma && gate_up_mma_supported(B, H, I, E, K))
    return {kGateUpMma, o.gu_npw == 16 ? 16 : 8, o.gu_cpl};
  if (o.gu_variant == kGateUpBatched) return {kGateUpBatched, o.gu_npw, o.gu_cpl};
  // built-in, from GB300 measurements on the 48-layer Qwen-3-style stack
  // (H=2048, I=768, E=128, K=8): one warp per (token, slot, neuron group) while
  // tokens rarely share experts (2*B*K < E); once they do, one wave of
  // persistent CTAs that read each expert row once for all its tokens, with
  // the products on tensor cores where the shape allows.
  if (2 * B * K >= E && gate_up_mma_supported(B, H, I, E, K)) return {kGateUpMma, 8, 0};
  if (2 * B * K >= E && gate_up_persist_supported(B, H, I, E, K)) return {kGateUpPersist, 2, 1};
  if (rowshare_ok && B >= o.rowshare_min_b) return {kGateUpRowShare, 2, 2};
  // one neuron per warp, two passes of 1 KiB per row at H=2048: 64 registers,
  // 4 CTAs per SM (measured: B = 2 21.4 -> 19.3, B = 4 37.2 -> 33.6 us/layer
  // against two neurons per warp at 2 CTAs per SM)
  return {kGateUpBatched, 1, 1};
}

// The per-(token, output dims) kernel's shape for this batch.
DownPlan batched_down_plan(int B, int I, int K) {
  const PlanOverride& o = plan_override();
  if (o.dn_variant == kDownBatched) return DownPlan{o.dn_rpw, o.dn_qpl, kDownBatched};
  if (B >= 4) return DownPlan{4, 1, kDownBatched};  // 4 output dims share each h block
  const int nq = K * (I / 32);
  const int per_lane = (nq + 31) / 32;
  if (B == 1)  // one output dim per warp, all of its K rows in flight at once
    return DownPlan{1, per_lane >= 6 ? 6 : (per_lane >= 4 ? 4 : (per_lane >= 2 ? 2 : 1)),
                    kDownBatched};
  return DownPlan{2, per_lane >= 3 ? 3 : (per_lane >= 2 ? 2 : 1), kDownBatched};
}

static DownPlan dimblock_plan(int I, int ns, int spg, int pairs, int split) {
  int S = 0, P = 0, G = 0;
  const int NS = down_dimblock_shape(I, ns, spg, pairs, split, &S, &P, &G);
  return DownPlan{NS, S, kDownDimBlock, P, G};
}

DownPlan plan_down(int B, int H, int I, int K, int E) {
  const PlanOverride& o = plan_override();
  if (o.dn_variant == kDownBatched) return batched_down_plan(B, I, K);
  if (o.dn_variant == kDownDimBlock && down_dimblock_supported(B, H, I, E, K))
    return dimblock_plan(I, o.dn_rpw, o.dn_qpl, o.dn_pairs, o.dn_split);
  // built-in: once most routed experts serve several (token, slot) pairs
  // (B*K >= E: B >= 16 at K = 8, E = 128), read each routed row once for all
  // of them; before that, one warp per (token, output dims) (measured on
  // GB300: B = 8 59.1 vs 62.7 us/layer, B = 16 equal, B = 32 140.1 vs 124.3)
  if (o.dn_variant < 0 && B * K >= E && down_dimblock_supported(B, H, I, E, K))
    return dimblock_plan(I, 0, 0, 0, 0);
  return batched_down_plan(B, I, K);
}

// Programmatic dependent launch for the launches of one call: bit i lets
// launch i start before launch i - 1 (for i = 0: whatever precedes the call on
// the stream) has finished; each kernel waits for its predecessor's results
// before reading them.
int pdl_mask_for(const GateUpPlan& g, const DownPlan& d) {
  const PlanOverride& o = plan_override();
  if (o.pdl_mask >= 0) return o.pdl_mask;
  if (d.variant == kDownDimBlock) return 7;
  // measured: letting the batched down kernel's CTAs start early while the
  // one-CTA-per-SM tensor-core gate/up kernel runs costs 7-14% of the layer
  return g.variant == kGateUpMma ? 1 : 3;
}

int launches_for(const DownPlan& d) { return d.variant == kDownDimBlock ? 3 : 2; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

GateUpPlan plan_gate_up_for(const GateUpArgs& a) {
  GateUpPlan p = plan_gate_up(a.B, a.H, a.I, a.K, a.E);
  if (p.variant == kGateUpMma && !(aligned16(a.gate_up) && aligned16(a.gate_up_scale)))
    p = gate_up_persist_supported(a.B, a.H, a.I, a.E, a.K) ? GateUpPlan{kGateUpPersist, 2, 1}
                                                           : GateUpPlan{kGateUpBatched, 1, 1};
  return p;
}

DownPlan plan_down_for(const DownArgs& a) {
  DownPlan p = plan_down(a.B, a.H, a.I, a.K, a.E);
  if (p.variant == kDownDimBlock && !(aligned16(a.down) && aligned16(a.down_scale)))
    p = batched_down_plan(a.B, a.I, a.K);
  return p;
}

// The down stage: moe_h_encode then moe_down_dimblock (scratch h16 / hk, both
// 16-byte aligned), or moe_down_3d_batched alone.  pdl: bit 0 for its first
// launch, bit 1 for its second.
cudaError_t launch_down_stage(const DownArgs& a, const DownPlan& p, void* h16, int32_t* hk,
                              cudaStream_t s, int pdl) {
  if (p.variant != kDownDimBlock) return launch_down(a, p, s, (pdl & 1) != 0);
  cudaError_t e = launch_h_encode(a.h, h16, hk, a.B * a.K, a.I, s, (pdl & 1) != 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_down_dimblock(a, p, h16, hk, s, (pdl & 2) != 0);
}

cudaError_t launch_layer(const GateUpArgs& ga, const DownArgs& da, void* h16, int32_t* hk,
                         cudaStream_t s) {
  const GateUpPlan gp = plan_gate_up_for(ga);
  const DownPlan dp = plan_down_for(da);
  const int pdl = pdl_mask_for(gp, dp);
  cudaError_t e = launch_gate_up(ga, gp, s, (pdl & 1) != 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_down_stage(da, dp, h16, hk, s, pdl >> 1);
}

size_t layer_scratch_h_bytes(int B, int K, int I) {
  return ((size_t)B * K * I * 2 + 255) / 256 * 256;
}
size_t layer_scratch_bytes(int B, int K, int I) {
  return 256 + 2 * layer_scratch_h_bytes(B, K, I) + ((size_t)B * K * 4 + 255) / 256 * 256;
}

namespace {
std::mutex g_smem_lock;
struct SmemEntry {
  const void* func;
  int dev, bytes;
};
std::vector<SmemEntry> g_smem_set;
}  // namespace

cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> guard(g_smem_lock);
  for (SmemEntry& s : g_smem_set)
    if (s.func == func && s.dev == dev) {
      if (s.bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) s.bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_set.push_back(SmemEntry{func, dev, bytes});
  return e;
}

}  // namespace wd

namespace {

constexpr int kMaxB = 4096, kMaxK = 64, kMaxDim = 16384;
constexpr size_t kFlagBytes = 256;  // the error flag's slot at the start of the workspace
// bits of the error flag (set by the kernels with atomicOr)
constexpr uint32_t kFlagBadExpertId = 1u;      // an expert id outside [0, E) was skipped
constexpr uint32_t kFlagPipelineTimeout = 2u;  // a bounded wait ran out: the output is invalid

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


wd_status check_dims(int B, int H, int I, int E, int K) {
  if (B < 1 || B > kMaxB || K < 1 || K > kMaxK || E < 1 || K > E) return WD_ERR_INVALID_ARG;
  if (H < 32 || I < 32 || H % 32 || I % 32 || H > kMaxDim || I > kMaxDim)
    return WD_ERR_UNSUPPORTED_SHAPE;
  return WD_OK;
}

// Name of the CUDA error behind this thread's last WD_ERR_CUDA.
thread_local const char* g_last_cuda_error = "none";

}  // namespace

wd_status wd::cuda_status(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) return WD_OK;
  g_last_cuda_error = cudaGetErrorName(e);
  return WD_ERR_CUDA;
}

using wd::cuda_status;

extern "C" {

const char* wd_status_string(wd_status s) {
  switch (s) {
    case WD_OK: return "WD_OK";
    case WD_ERR_INVALID_ARG: return "WD_ERR_INVALID_ARG";
    case WD_ERR_UNSUPPORTED_SHAPE: return "WD_ERR_UNSUPPORTED_SHAPE";
    case WD_ERR_WORKSPACE_TOO_SMALL: return "WD_ERR_WORKSPACE_TOO_SMALL";
    case WD_ERR_CUDA: return "WD_ERR_CUDA";
    case WD_ERR_BAD_EXPERT_ID: return "WD_ERR_BAD_EXPERT_ID";
    case WD_ERR_PIPELINE_TIMEOUT: return "WD_ERR_PIPELINE_TIMEOUT";
  }
  return "WD_ERR_UNKNOWN";
}

size_t wd_moe_workspace_size(int B, int K, int I) {
  if (B <= 0 || K <= 0 || I <= 0) return 0;
  return wd::layer_scratch_bytes(B, K, I);
}

// Workspace layout (wd::layer_scratch_bytes): [0, 256) the error flag; then h
// BF16 [B,K,I], h re-encoded as FP16 [B,K,I] and its per-row exponents int32
// [B,K], each region rounded up to 256 bytes.
static uint32_t* flag_of(void* workspace) { return static_cast<uint32_t*>(workspace); }
static void* h_of(void* workspace) { return static_cast<uint8_t*>(workspace) + kFlagBytes; }
static void* h16_of(void* workspace, int B, int K, int I) {
  return static_cast<uint8_t*>(workspace) + kFlagBytes + wd::layer_scratch_h_bytes(B, K, I);
}
static int32_t* hk_of(void* workspace, int B, int K, int I) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + kFlagBytes +
                                    2 * wd::layer_scratch_h_bytes(B, K, I));
}

wd_status wd_moe_workspace_init(void* workspace, size_t workspace_bytes, wd_stream_t stream) {
  if (!workspace || !aligned(workspace, 256)) return WD_ERR_INVALID_ARG;
  if (workspace_bytes < kFlagBytes) return WD_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(cudaMemsetAsync(flag_of(workspace), 0, sizeof(uint32_t),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

wd_status wd_moe_gate_up(const void* x, const int32_t* topk_ids, const uint8_t* gate_up,
                         const uint8_t* gate_up_scale, void* h, uint32_t* error_flag, int B,
                         int H, int I, int E, int K, wd_stream_t stream) {
  wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  if (!x || !topk_ids || !gate_up || !gate_up_scale || !h) return WD_ERR_INVALID_ARG;
  if (!aligned(x, 32) || !aligned(gate_up, 32) || !aligned(topk_ids, 4) || !aligned(h, 4) ||
      (error_flag && !aligned(error_flag, 4)))
    return WD_ERR_INVALID_ARG;
  const wd::GateUpArgs a{x, topk_ids, gate_up, gate_up_scale, h, error_flag, B, H, I, E, K};
  return cuda_status(wd::launch_gate_up(a, wd::plan_gate_up_for(a),
                                        reinterpret_cast<cudaStream_t>(stream), true));
}

wd_status wd_moe_down(const void* h, const int32_t* topk_ids, const float* topk_w,
                      const uint8_t* down, const uint8_t* down_scale, void* out,
                      uint32_t* error_flag, int B, int H, int I, int E, int K,
                      wd_stream_t stream) {
  wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  if (!h || !topk_ids || !topk_w || !down || !down_scale || !out) return WD_ERR_INVALID_ARG;
  if (!aligned(h, 32) || !aligned(down, 32) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) ||
      !aligned(out, 4) || (error_flag && !aligned(error_flag, 4)))
    return WD_ERR_INVALID_ARG;
  const wd::DownArgs a{h, topk_ids, topk_w, down, down_scale, out, error_flag, B, H, I, E, K};
  // no scratch here: the per-(token, output dims) kernel, launched without
  // programmatic dependent launch (the kernel may read the routing before
  // waiting on its predecessor, which here can be anything)
  wd::DownPlan p = wd::plan_down_for(a);
  if (p.variant != wd::kDownBatched) p = wd::batched_down_plan(B, I, K);
  return cuda_status(wd::launch_down(a, p, reinterpret_cast<cudaStream_t>(stream), false));
}

wd_status wd_moe_h_encode(const void* h, void* h16, int32_t* hk, int rows, int I,
                          wd_stream_t stream) {
  if (!h || !h16 || !hk || rows < 1 || rows > kMaxB * kMaxK) return WD_ERR_INVALID_ARG;
  if (I < 32 || I % 32 || I > kMaxDim) return WD_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(h, 16) || !aligned(h16, 16) || !aligned(hk, 4)) return WD_ERR_INVALID_ARG;
  return cuda_status(
      wd::launch_h_encode(h, h16, hk, rows, I, reinterpret_cast<cudaStream_t>(stream), false));
}

wd_status wd_moe_down_encoded(const void* h16, const int32_t* hk, const int32_t* topk_ids,
                              const float* topk_w, const uint8_t* down, const uint8_t* down_scale,
                              void* out, uint32_t* error_flag, int B, int H, int I, int E, int K,
                              wd_stream_t stream) {
  wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  if (!h16 || !hk || !topk_ids || !topk_w || !down || !down_scale || !out)
    return WD_ERR_INVALID_ARG;
  if (!aligned(h16, 16) || !aligned(hk, 4) || !aligned(down, 32) || !aligned(down_scale, 16) ||
      !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(out, 4) ||
      (error_flag && !aligned(error_flag, 4)))
    return WD_ERR_INVALID_ARG;
  if (!wd::down_dimblock_supported(B, H, I, E, K)) return WD_ERR_UNSUPPORTED_SHAPE;
  const wd::DownArgs a{nullptr, topk_ids, topk_w, down, down_scale, out, error_flag,
                       B, H, I, E, K};
  wd::DownPlan p = wd::plan_down(B, H, I, K, E);
  if (p.variant != wd::kDownDimBlock) {
    int S = 0, P = 0, G = 0;
    const int NS = wd::down_dimblock_shape(I, 0, 0, 0, 0, &S, &P, &G);
    p = wd::DownPlan{NS, S, wd::kDownDimBlock, P, G};
  }
  return cuda_status(wd::launch_down_dimblock(a, p, h16, hk,
                                              reinterpret_cast<cudaStream_t>(stream), false));
}

wd_status wd_moe_down_workspace(const void* h, const int32_t* topk_ids, const float* topk_w,
                                const uint8_t* down, const uint8_t* down_scale, void* out,
                                void* workspace, size_t workspace_bytes, int B, int H, int I,
                                int E, int K, wd_stream_t stream) {
  wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  if (!h || !topk_ids || !topk_w || !down || !down_scale || !out || !workspace)
    return WD_ERR_INVALID_ARG;
  if (!aligned(h, 32) || !aligned(down, 32) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) ||
      !aligned(out, 4) || !aligned(workspace, 256))
    return WD_ERR_INVALID_ARG;
  if (workspace_bytes < wd_moe_workspace_size(B, K, I)) return WD_ERR_WORKSPACE_TOO_SMALL;
  const wd::DownArgs a{h, topk_ids, topk_w, down, down_scale, out, flag_of(workspace),
                       B, H, I, E, K};
  // the first launch waits for nothing it could race with: no overlap with
  // the caller's previous work; the encode -> down pair may overlap
  return cuda_status(wd::launch_down_stage(a, wd::plan_down_for(a), h16_of(workspace, B, K, I),
                                           hk_of(workspace, B, K, I),
                                           reinterpret_cast<cudaStream_t>(stream), 2));
}

wd_status wd_moe_decode(const void* x, const int32_t* topk_ids, const float* topk_w,
                        const uint8_t* gate_up, const uint8_t* gate_up_scale,
                        const uint8_t* down, const uint8_t* down_scale, void* out,
                        void* workspace, size_t workspace_bytes, int B, int H, int I, int E,
                        int K, wd_stream_t stream) {
  wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  if (!x || !topk_ids || !topk_w || !gate_up || !gate_up_scale || !down || !down_scale || !out ||
      !workspace)
    return WD_ERR_INVALID_ARG;
  if (!aligned(x, 32) || !aligned(gate_up, 32) || !aligned(down, 32) || !aligned(topk_ids, 4) ||
      !aligned(topk_w, 4) || !aligned(out, 4) || !aligned(workspace, 256))
    return WD_ERR_INVALID_ARG;
  if (workspace_bytes < wd_moe_workspace_size(B, K, I)) return WD_ERR_WORKSPACE_TOO_SMALL;
  uint32_t* flag = flag_of(workspace);
  void* h = h_of(workspace);
  const wd::GateUpArgs ga{x, topk_ids, gate_up, gate_up_scale, h, flag, B, H, I, E, K};
  const wd::DownArgs da{h, topk_ids, topk_w, down, down_scale, out, flag, B, H, I, E, K};
  return cuda_status(wd::launch_layer(ga, da, h16_of(workspace, B, K, I), hk_of(workspace, B, K, I),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

wd_status wd_moe_read_error_flag(void* workspace, size_t workspace_bytes, wd_stream_t stream,
                                 int* flag) {
  if (!workspace || !flag || !aligned(workspace, 256)) return WD_ERR_INVALID_ARG;
  if (workspace_bytes < kFlagBytes) return WD_ERR_WORKSPACE_TOO_SMALL;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  uint32_t* dflag = flag_of(workspace);
  cudaError_t e = cudaMemcpyAsync(&v, dflag, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dflag, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  *flag = (int)(v & (kFlagBadExpertId | kFlagPipelineTimeout));
  if (v & kFlagPipelineTimeout) return WD_ERR_PIPELINE_TIMEOUT;
  return (v & kFlagBadExpertId) ? WD_ERR_BAD_EXPERT_ID : WD_OK;
}

int wd_moe_launches_per_call(void) { return 3; }

int wd_moe_launches(int B, int H, int I, int E, int K) {
  if (check_dims(B, H, I, E, K) != WD_OK) return 0;
  return wd::launches_for(wd::plan_down(B, H, I, K, E));
}

const char* wd_last_error_string(void) { return g_last_cuda_error; }

wd_status wd_moe_describe_plan(int B, int H, int I, int E, int K, char* buf, size_t bytes) {
  if (!buf || bytes < 128) return WD_ERR_INVALID_ARG;
  const wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  const wd::GateUpPlan g = wd::plan_gate_up(B, H, I, K, E);
  const wd::DownPlan d = wd::plan_down(B, H, I, K, E);
  static const char* const gu_names[] = {"moe_gate_up_3d_batched", "moe_gate_up_rowshare",
                                         "moe_gate_up_persist", "moe_gate_up_mma"};
  static const char* const dn_names[] = {"moe_down_3d_batched", "moe_down_dimblock"};
  const int ngu = (int)(sizeof(gu_names) / sizeof(gu_names[0]));
  const int ndn = (int)(sizeof(dn_names) / sizeof(dn_names[0]));
  const char* gn = (g.variant >= 0 && g.variant < ngu) ? gu_names[g.variant] : "?";
  const char* dn = (d.variant >= 0 && d.variant < ndn) ? dn_names[d.variant] : "?";
  if (d.variant == wd::kDownDimBlock)
    snprintf(buf, bytes, "gate_up=%s<%d,%d> down=%s<%d,%d,%d,%d> pdl=%d launches=%d", gn, g.npw,
             g.cpl, dn, d.rpw, d.qpl / (d.rpw > 0 ? d.rpw : 1), d.pairs, d.split,
             wd::pdl_mask_for(g, d), wd::launches_for(d));
  else
    snprintf(buf, bytes, "gate_up=%s<%d,%d> down=%s<%d,%d> pdl=%d launches=%d", gn, g.npw, g.cpl,
             dn, d.rpw, d.qpl, wd::pdl_mask_for(g, d), wd::launches_for(d));
  return WD_OK;
}

wd_status wd_moe_set_plan(const char* spec) {
  wd::PlanOverride p;
  if (!wd::parse_plan(spec, &p)) return WD_ERR_INVALID_ARG;
  wd::plan_override() = p;
  return WD_OK;
}

}  // extern "C"
