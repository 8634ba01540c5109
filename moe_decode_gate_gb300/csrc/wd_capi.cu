// wd_capi.cu - the C-ABI of the MoE decode layer (declared in include/wd_moe.h).
//
// Host-side argument checks, the per-shape launch plan, and the two launches.
// Nothing here allocates or synchronises except wd_moe_read_error_flag, which
// is documented to synchronise.
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/wd_moe.h"
#include "wd_launch.h"

namespace wd {

// Launch plan.  The batched gate/up kernel keeps 2*npw rows of H bytes in
// flight per warp and does ceil(H/32/32) blocks per lane in passes of cpl; the
// shared-row variant serves every token of an expert from one dequantised row
// and is used once tokens start to share experts.  The down kernel spreads the
// K*I/32 blocks of the K routed rows over the lanes in passes of qpl per lane.
//
// wd_moe_set_plan (or the WD_PLAN environment variable, read at the first
// call) overrides the choice for tuning sweeps and tests:
//   "gu=batched:<npw>:<cpl>" | "gu=rowshare:<npw>:<sbw>" | "gu=stream:<npw>:<stages>" |
//   "gu=mixed:<npw>:<stages>" | "gu=persist:<npw>:<prefetch+1>" | "gu=ring:<stages>" | "gu=tma" |
//   "gu=mma[:<stages>[:<consumer warps, 8 or 16>]]",
//   "dn=<rpw>:<qpl>" | "dn=stream:<stages>" | "dn=persist:<rpw>:<qpl>" | "dn=shared:<rpw>" |
//   "dn=mma[:<stages>]" | "dn=3dmma" | "dn=emma[:<stages>[:<parts of I, 1 or 2>]]",
//   "rowshare_min_b=<B>", "pdl=<mask>" (bit 0: the gate/up launch may overlap the
//   kernel before it, bit 1: the down launch may overlap gate/up), comma-separated;
//   "" or NULL restores the defaults.
namespace {

struct PlanOverride {
  int gu_variant = -1, gu_npw = 0, gu_cpl = 0;
  int dn_variant = -1, dn_rpw = 0, dn_qpl = 0;
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
      if (sscanf(tok, "gu=batched:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpBatched;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (sscanf(tok, "gu=mixed:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpMixed;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (sscanf(tok, "gu=stream:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpStream;
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
      } else if (strcmp(tok, "gu=tma") == 0) {
        p.gu_variant = kGateUpTma;
        p.gu_npw = 2;
        p.gu_cpl = 3;
      } else if (sscanf(tok, "gu=ring:%d", &a) == 1) {
        p.gu_variant = kGateUpRing;
        p.gu_npw = a;
        p.gu_cpl = 0;
      } else if (sscanf(tok, "gu=persist:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpPersist;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (sscanf(tok, "gu=rowshare:%d:%d", &a, &b) == 2) {
        p.gu_variant = kGateUpRowShare;
        p.gu_npw = a;
        p.gu_cpl = b;
      } else if (sscanf(tok, "dn=mma:%d", &a) == 1) {
        p.dn_variant = kDownMma;
        p.dn_qpl = a;
      } else if (sscanf(tok, "dn=emma:%d:%d", &a, &b) == 2) {
        p.dn_variant = kDownExpertMma;
        p.dn_qpl = a;
        p.dn_rpw = b;
      } else if (sscanf(tok, "dn=emma:%d", &a) == 1) {
        p.dn_variant = kDownExpertMma;
        p.dn_qpl = a;
        p.dn_rpw = 1;
      } else if (strcmp(tok, "dn=emma") == 0) {
        p.dn_variant = kDownExpertMma;
        p.dn_qpl = 0;
        p.dn_rpw = 1;
      } else if (strcmp(tok, "dn=3dmma") == 0) {
        p.dn_variant = kDown3dMma;
      } else if (strcmp(tok, "dn=mma") == 0) {
        p.dn_variant = kDownMma;
        p.dn_qpl = 0;
      } else if (sscanf(tok, "dn=stream:%d", &a) == 1) {
        p.dn_variant = kDownStream;
        p.dn_qpl = a;
      } else if (sscanf(tok, "dn=shared:%d", &a) == 1) {
        p.dn_variant = kDownShared;
        p.dn_rpw = a;
      } else if (sscanf(tok, "dn=persist:%d:%d", &a, &b) == 2) {
        p.dn_variant = kDownPersist;
        p.dn_rpw = a;
        p.dn_qpl = b;
      } else if (sscanf(tok, "dn=%d:%d", &a, &b) == 2) {
        p.dn_variant = kDownBatched;
        p.dn_rpw = a;
        p.dn_qpl = b;
      } else if (sscanf(tok, "rowshare_min_b=%d", &a) == 1) {
        p.rowshare_min_b = a;
      } else if (sscanf(tok, "pdl=%d", &a) == 1 && a >= 0 && a <= 3) {
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
  if (o.gu_variant == kGateUpStream && gate_up_stream_supported(B, H, I, E, K, o.gu_npw))
    return {kGateUpStream, o.gu_npw, o.gu_cpl};
  if (o.gu_variant == kGateUpMixed && gate_up_mixed_supported(B, H, I, E, K, o.gu_npw))
    return {kGateUpMixed, o.gu_npw, o.gu_cpl};
  if (o.gu_variant == kGateUpRowShare && rowshare_ok) return {kGateUpRowShare, o.gu_npw, o.gu_cpl};
  if (o.gu_variant == kGateUpPersist && gate_up_persist_supported(B, H, I, E, K))
    return {kGateUpPersist, o.gu_npw, o.gu_cpl};
  if (o.gu_variant == kGateUpRing && gate_up_ring_supported(B, H, I, E, K, o.gu_npw))
    return {kGateUpRing, o.gu_npw, 0};
  if (o.gu_variant == kGateUpTma && gate_up_tma_supported(B, H, I, E, K))
    return {kGateUpTma, 2, 3};
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
  if (B == 1) return {kGateUpBatched, 1, 1};
  return {kGateUpBatched, 2, 1};  // two passes of 1 KiB per row at H=2048, 4 rows in flight
}

DownPlan plan_down(int B, int H, int I, int K, int E) {
  const PlanOverride& o = plan_override();
  if (o.dn_variant == kDownStream && down_stream_supported(B, H, I, E, K))
    return DownPlan{0, o.dn_qpl, kDownStream};
  if (o.dn_variant == kDownBatched) return DownPlan{o.dn_rpw, o.dn_qpl, kDownBatched};
  if (o.dn_variant == kDownPersist) return DownPlan{o.dn_rpw, o.dn_qpl, kDownPersist};
  if (o.dn_variant == kDownShared && down_shared_supported(B, H, I, E, K, o.dn_rpw))
    return DownPlan{o.dn_rpw, 0, kDownShared};
  if (o.dn_variant == kDownMma && down_mma_supported(B, H, I, E, K))
    return DownPlan{16, o.dn_qpl, kDownMma};
  if (o.dn_variant == kDown3dMma && down_3d_mma_supported(B, H, I, E, K))
    return DownPlan{16, 0, kDown3dMma};
  if (o.dn_variant == kDownExpertMma && down_expert_mma_supported(B, H, I, E, K))
    return DownPlan{o.dn_rpw == 2 ? 2 : 1, o.dn_qpl, kDownExpertMma};
  if (B >= 4) return DownPlan{4, 1, kDownBatched};  // 4 output dims share each h block
  const int nq = K * (I / 32);
  const int per_lane = (nq + 31) / 32;
  if (B == 1)  // one output dim per warp, all of its K rows in flight at once
    return DownPlan{1, per_lane >= 6 ? 6 : (per_lane >= 4 ? 4 : (per_lane >= 2 ? 2 : 1)),
                    kDownBatched};
  return DownPlan{2, per_lane >= 3 ? 3 : (per_lane >= 2 ? 2 : 1), kDownBatched};
}

// Programmatic dependent launch for the two launches of one call (bit 0:
// gate/up after whatever precedes it on the stream, bit 1: down after gate/up).
int pdl_mask_for(const GateUpPlan& g) {
  const PlanOverride& o = plan_override();
  if (o.pdl_mask >= 0) return o.pdl_mask;
  // measured: letting the down kernel's CTAs start early while the one-CTA-per-SM
  // tensor-core gate/up kernel runs costs 7-14% of the layer at B = 8..32
  return g.variant == kGateUpMma ? 1 : 3;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

GateUpPlan plan_gate_up_for(const GateUpArgs& a) {
  GateUpPlan p = plan_gate_up(a.B, a.H, a.I, a.K, a.E);
  if ((p.variant == kGateUpStream || p.variant == kGateUpMixed || p.variant == kGateUpRing ||
       p.variant == kGateUpTma || p.variant == kGateUpMma) &&
      !(aligned16(a.gate_up) && aligned16(a.gate_up_scale)))
    p = gate_up_persist_supported(a.B, a.H, a.I, a.E, a.K) ? GateUpPlan{kGateUpPersist, 2, 1}
                                                           : GateUpPlan{kGateUpBatched, 2, 1};
  return p;
}

DownPlan plan_down_for(const DownArgs& a) {
  DownPlan p = plan_down(a.B, a.H, a.I, a.K, a.E);
  if ((p.variant == kDownStream && !(aligned16(a.down) && aligned16(a.down_scale))) ||
      ((p.variant == kDownMma || p.variant == kDown3dMma || p.variant == kDownExpertMma) &&
       !(aligned16(a.down) && aligned16(a.down_scale) && aligned16(a.h)))) {
    const int per_lane = (a.K * (a.I / 32) + 31) / 32;
    p = DownPlan{2, per_lane >= 3 ? 3 : (per_lane >= 2 ? 2 : 1), kDownBatched};
  }
  return p;
}

}  // namespace wd

namespace {

constexpr int kMaxB = 4096, kMaxK = 64, kMaxDim = 16384;
constexpr size_t kFlagBytes = 256;  // the error flag's slot at the start of the workspace

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t h_bytes(int B, int K, int I) {
  const size_t raw = (size_t)B * K * I * 2;
  return (raw + 255) / 256 * 256;
}

wd_status check_dims(int B, int H, int I, int E, int K) {
  if (B < 1 || B > kMaxB || K < 1 || K > kMaxK || E < 1 || K > E) return WD_ERR_INVALID_ARG;
  if (H < 32 || I < 32 || H % 32 || I % 32 || H > kMaxDim || I > kMaxDim)
    return WD_ERR_UNSUPPORTED_SHAPE;
  return WD_OK;
}

// Name of the CUDA error behind this thread's last WD_ERR_CUDA.
thread_local const char* g_last_cuda_error = "none";

wd_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) return WD_OK;
  g_last_cuda_error = cudaGetErrorName(e);
  return WD_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* wd_status_string(wd_status s) {
  switch (s) {
    case WD_OK: return "WD_OK";
    case WD_ERR_INVALID_ARG: return "WD_ERR_INVALID_ARG";
    case WD_ERR_UNSUPPORTED_SHAPE: return "WD_ERR_UNSUPPORTED_SHAPE";
    case WD_ERR_WORKSPACE_TOO_SMALL: return "WD_ERR_WORKSPACE_TOO_SMALL";
    case WD_ERR_CUDA: return "WD_ERR_CUDA";
    case WD_ERR_BAD_EXPERT_ID: return "WD_ERR_BAD_EXPERT_ID";
  }
  return "WD_ERR_UNKNOWN";
}

size_t wd_moe_workspace_size(int B, int K, int I) {
  if (B <= 0 || K <= 0 || I <= 0) return 0;
  return kFlagBytes + h_bytes(B, K, I);
}

static uint32_t* flag_of(void* workspace) { return static_cast<uint32_t*>(workspace); }
static void* h_of(void* workspace) { return static_cast<uint8_t*>(workspace) + kFlagBytes; }

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
  // launched without programmatic dependent launch: the kernel may read the
  // routing before waiting on its predecessor, which here can be anything
  return cuda_status(wd::launch_down(a, wd::plan_down_for(a),
                                     reinterpret_cast<cudaStream_t>(stream), false));
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
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* flag = flag_of(workspace);
  void* h = h_of(workspace);
  const wd::GateUpArgs ga{x, topk_ids, gate_up, gate_up_scale, h, flag, B, H, I, E, K};
  const wd::GateUpPlan gp = wd::plan_gate_up_for(ga);
  const int pdl = wd::pdl_mask_for(gp);
  st = cuda_status(wd::launch_gate_up(ga, gp, s, (pdl & 1) != 0));
  if (st != WD_OK) return st;
  const wd::DownArgs da{h, topk_ids, topk_w, down, down_scale, out, flag, B, H, I, E, K};
  return cuda_status(wd::launch_down(da, wd::plan_down_for(da), s, (pdl & 2) != 0));
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
  if (e != cudaSuccess) return WD_ERR_CUDA;
  *flag = v ? 1 : 0;
  return v ? WD_ERR_BAD_EXPERT_ID : WD_OK;
}

int wd_moe_launches_per_call(void) { return 2; }

const char* wd_last_error_string(void) { return g_last_cuda_error; }

wd_status wd_moe_describe_plan(int B, int H, int I, int E, int K, char* buf, size_t bytes) {
  if (!buf || bytes < 128) return WD_ERR_INVALID_ARG;
  const wd_status st = check_dims(B, H, I, E, K);
  if (st != WD_OK) return st;
  const wd::GateUpPlan g = wd::plan_gate_up(B, H, I, K, E);
  const wd::DownPlan d = wd::plan_down(B, H, I, K, E);
  static const char* const gu_names[] = {"moe_gate_up_3d_batched", "moe_gate_up_rowshare",
                                         "moe_gate_up_stream", "moe_gate_up_mixed",
                                         "moe_gate_up_persist", "moe_gate_up_ring",
                                         "moe_gate_up_tma", "moe_gate_up_mma"};
  static const char* const dn_names[] = {"moe_down_3d_batched", "moe_down_stream",
                                         "moe_down_3d_batched_persist", "moe_down_shared",
                                         "moe_down_mma", "moe_down_3d_mma",
                                         "moe_down_expert_mma"};
  const char* gn = (g.variant >= 0 && g.variant <= 7) ? gu_names[g.variant] : "?";
  const char* dn = (d.variant >= 0 && d.variant <= 6) ? dn_names[d.variant] : "?";
  snprintf(buf, bytes, "gate_up=%s<%d,%d> down=%s<%d,%d> pdl=%d", gn, g.npw, g.cpl, dn, d.rpw,
           d.qpl, wd::pdl_mask_for(g));
  return WD_OK;
}

wd_status wd_moe_set_plan(const char* spec) {
  wd::PlanOverride p;
  if (!wd::parse_plan(spec, &p)) return WD_ERR_INVALID_ARG;
  wd::plan_override() = p;
  return WD_OK;
}

}  // extern "C"
