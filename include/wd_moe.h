/*
 * wd_moe.h - small-batch MoE decode layer on MXFP8 expert weights ("warp decode").
 *
 * The layer (Cursor, "用 warp decode 实现更好的 MoE 模型推理" [Better MoE
 * inference with warp decode], section 两个 kernel 如何工作 [How the two kernels
 * work]): for each token b with routed experts e_k = topk_ids[b,k] and routing
 * weights w_k = topk_w[b,k], k < K,
 *
 *     h[b,k,n] = bf16( SiLU(Wg[e_k] x[b])_n * (Wu[e_k] x[b])_n ),   n < I
 *     y[b,d]   = sum_k w_k * (Wd[e_k] h[b,k,:])_d,                  d < H
 *     out[b,d] = bf16(y[b,d])
 *
 * computed as two kernels organised around outputs rather than experts:
 *   moe_gate_up_3d_batched - one warp per (token, routed expert, intermediate
 *                            neuron): streams that neuron's gate and up rows
 *                            once, dots both against x, writes one BF16 value;
 *   moe_down_3d_batched    - one warp per (token, output dim): walks all K
 *                            routed experts' down rows and folds the weighted
 *                            contributions into one FP32 register accumulator,
 *                            reduces across the warp with shuffles, writes once.
 * There is no padding, no gather of activations into expert-major buffers and no
 * combine pass (section 阶段消除 [Stage elimination], section 消除缓冲区
 * [Eliminating buffers]).  Activations are BF16, accumulation is FP32 and the
 * weights are dequantised from MXFP8 as they stream in (section 精度提升
 * [Accuracy gains]).
 *
 * Formats (OCP Microscaling Formats (MX) v1.0):
 *   weights: E4M3 codes (1 byte) with one E8M0 scale byte (2^(s-127)) per 32
 *            consecutive elements along the reduction dimension;
 *   x, h, out: BF16 (IEEE binary32 upper half), round to nearest even on store.
 *
 * Memory layout (all row-major, contiguous, device memory, caller-owned):
 *   x              bf16  [B, H]
 *   topk_ids       int32 [B, K]
 *   topk_w         fp32  [B, K]
 *   gate_up        e4m3  [E, 2I, H]   rows [0, I) = gate, rows [I, 2I) = up
 *   gate_up_scale  e8m0  [E, 2I, H/32]
 *   down           e4m3  [E, H, I]
 *   down_scale     e8m0  [E, H, I/32]
 *   out            bf16  [B, H]
 *   workspace      wd_moe_workspace_size(B, K, I) bytes, 256-byte aligned:
 *                  bytes [0, 4) a 32-bit error flag, bytes [256, ...) the
 *                  BF16 intermediate h [B, K, I]; a workspace sized for a
 *                  batch B serves every smaller batch
 *
 * Requirements checked on the host (a violation returns an error, nothing is
 * launched): non-null pointers; B >= 1; 1 <= K <= E; H and I multiples of 32
 * with H <= 16384 and I <= 16384; K <= 64; B <= 4096; x, gate_up and down
 * 32-byte aligned; gate_up_scale, down_scale, topk_ids, topk_w, out and
 * workspace 4-byte aligned (the workspace 256-byte aligned); workspace_bytes
 * large enough.
 *
 * Expert ids are range-checked on the device: an id outside [0, E) contributes
 * nothing (its h entries are written as 0) and sets the workspace error flag,
 * which stays set until wd_moe_read_error_flag reads and clears it.  Duplicate
 * ids within a token are allowed; their contributions add.
 *
 * Every entry point that launches work is asynchronous on `stream`: it never
 * synchronises, never allocates, and returns after the launches.  Launch
 * failures are reported as WD_ERR_CUDA (cudaGetLastError after the launch).
 * Calls on different streams must not share a workspace.  `out` must not alias
 * `x`, the weights or the workspace.
 */
#ifndef WD_MOE_H_
#define WD_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifndef WD_API
#define WD_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* wd_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum wd_status {
  WD_OK = 0,
  WD_ERR_INVALID_ARG = 1,         /* null/misaligned pointer, B/K/E out of range */
  WD_ERR_UNSUPPORTED_SHAPE = 2,   /* H or I not a multiple of 32, or too large   */
  WD_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < wd_moe_workspace_size(...) */
  WD_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed        */
  WD_ERR_BAD_EXPERT_ID = 5        /* reported by wd_moe_read_error_flag only     */
} wd_status;

/* Human-readable name of a status code (static string, never NULL). */
WD_API const char* wd_status_string(wd_status s);

/* Bytes of workspace wd_moe_decode needs for (B, K, I): 256 bytes holding the
 * error flag plus the BF16 intermediate h [B, K, I] rounded up to 256 bytes.
 * Returns 0 when B, K or I is not positive. */
WD_API size_t wd_moe_workspace_size(int B, int K, int I);

/* Zero the workspace's error flag (one 4-byte cudaMemsetAsync on `stream`).
 * Call once after allocating a workspace, before its first use. */
WD_API wd_status wd_moe_workspace_init(void* workspace, size_t workspace_bytes,
                                       wd_stream_t stream);

/* The MoE decode layer: both kernels, back to back on `stream` (the second
 * launched as a programmatic dependent of the first, so that its weight
 * prefetch overlaps the first kernel's tail).  See the file comment for the
 * layout and the definition.  h is left in the workspace. */
WD_API wd_status wd_moe_decode(const void* x, const int32_t* topk_ids, const float* topk_w,
                        const uint8_t* gate_up, const uint8_t* gate_up_scale,
                        const uint8_t* down, const uint8_t* down_scale, void* out,
                        void* workspace, size_t workspace_bytes, int B, int H, int I, int E,
                        int K, wd_stream_t stream);

/* First kernel alone (moe_gate_up_3d_batched; section 两个 kernel 如何工作,
 * gate/up paragraph): h [B, K, I] BF16 (caller-owned, 4-byte aligned) from x,
 * topk_ids and the gate/up weights.  `error_flag` is a device uint32 that is
 * OR-ed with 1 when an expert id is out of range (may be NULL). */
WD_API wd_status wd_moe_gate_up(const void* x, const int32_t* topk_ids, const uint8_t* gate_up,
                         const uint8_t* gate_up_scale, void* h, uint32_t* error_flag, int B,
                         int H, int I, int E, int K, wd_stream_t stream);

/* Second kernel alone (moe_down_3d_batched; section 两个 kernel 如何工作, down
 * paragraph): out [B, H] BF16 from h [B, K, I] BF16 (32-byte aligned),
 * topk_ids, topk_w and the down weights. */
WD_API wd_status wd_moe_down(const void* h, const int32_t* topk_ids, const float* topk_w,
                      const uint8_t* down, const uint8_t* down_scale, void* out,
                      uint32_t* error_flag, int B, int H, int I, int E, int K,
                      wd_stream_t stream);

/* Copy the workspace's error flag to `*flag` (1 if any call since the last read
 * saw an expert id outside [0, E), else 0) and clear it.  This call
 * SYNCHRONISES `stream`.  Returns WD_ERR_BAD_EXPERT_ID when the flag was set. */
WD_API wd_status wd_moe_read_error_flag(void* workspace, size_t workspace_bytes,
                                       wd_stream_t stream, int* flag);

/* Name of the CUDA error (cudaGetErrorName) behind the calling thread's most
 * recent WD_ERR_CUDA, or "none".  Static storage; never NULL. */
WD_API const char* wd_last_error_string(void);

/* Number of kernel launches wd_moe_decode issues per call (for accounting). */
WD_API int wd_moe_launches_per_call(void);

/* Override the per-shape launch plan (tuning and tests; not needed in normal
 * use).  `spec` is a comma-separated list of
 *   "gu=batched:<neurons per warp>:<blocks per lane per pass>"
 *   "gu=rowshare:<neurons per warp>:<words per step>"   (tokens share rows)
 *   "gu=persist:<neurons per warp>:<1 + L2 prefetch distance>"
 *   "gu=ring:<bulk-copy ring stages per warp>" | "gu=tma" |
 *   "gu=mma[:<ring stages, 2..4>[:<consumer warps, 8 or 16>]]"
 *                                   (tensor-core products; B*K <= 256,
 *                                    H % 512 == 0, H <= 2048, I % 16 == 0)
 *   "gu=stream:<variant>:<stages>" | "gu=mixed:<variant>:<stages>"
 *   "dn=<output dims per warp>:<blocks per lane per pass>"
 *   "dn=persist:<output dims per warp>:<blocks per lane per pass>"
 *   "dn=stream:<stages>" | "dn=shared:<output dims per CTA>"
 *   "dn=3dmma"   (warp per (token, 16 output dims), dots on tensor cores;
 *                 H % 16 == 0, I % 256 == 0, I <= 1024, K <= 32)
 *   "dn=mma[:<ring stages, 2..7>]"  (tensor-core products; B <= 64,
 *                                    B*K <= 256, H % 16 == 0, I % 128 == 0)
 *   "dn=emma[:<ring stages, 8..16>[:<parts of I per step, 1 or 2>]]"
 *                (tensor-core products, one warp per routed-expert step;
 *                 B <= 64, B*K <= 256, H % 16 == 0, I % 128 == 0, and a
 *                 ring of 8 stages fitting in shared memory: any such B up
 *                 to I = 768, small B up to I = 1024)
 *   "rowshare_min_b=<smallest batch that uses the shared-row gate/up kernel
 *                    where the persistent one does not apply>"
 *   "pdl=<0..3>" (programmatic dependent launch: bit 0 lets the gate/up
 *                 launch overlap the kernel before it, bit 1 lets the down
 *                 launch overlap gate/up)
 * NULL or "" restores the built-in plan.  Returns WD_ERR_INVALID_ARG for an
 * unparsable spec (the plan is then unchanged); a variant that does not
 * support the call's shape falls back to the built-in choice, and an
 * unsupported parameter combination makes later launches fail with
 * WD_ERR_CUDA.  Process-wide; do not call while another thread is inside a
 * wd_moe_* call.  The WD_PLAN environment variable, read at the first launch,
 * sets the initial override. */
WD_API wd_status wd_moe_set_plan(const char* spec);

/* Write the kernels wd_moe_decode would launch for this shape under the
 * current plan (16-byte-aligned weight pointers assumed), as
 * "gate_up=<kernel><params> down=<kernel><params> pdl=<mask>" (the mask as in
 * wd_moe_set_plan's "pdl="), NUL-terminated, into
 * `buf` (`bytes` long; 128 bytes always suffice).  Host-only: launches
 * nothing.  Returns WD_ERR_INVALID_ARG for a NULL or too small buffer and the
 * status wd_moe_decode would return for invalid dimensions. */
WD_API wd_status wd_moe_describe_plan(int B, int H, int I, int E, int K, char* buf, size_t bytes);

/* The same layer as wd_moe_decode, for callers that cannot allocate device
 * memory and so cannot provide a workspace: for example a plugin whose host
 * framework owns all device memory and forbids allocating while it runs, or a
 * latency-critical caller that cannot pay for cudaMalloc's possible implicit
 * device synchronisation.  The blog has no counterpart: this is a property of
 * this library's interface, not of the method.
 *
 * The intermediate h lives in a 1 MiB array compiled into the library
 * (file-scope device memory that every GPU loading the library holds until the
 * process exits), so B * K * I * 2 must be at most 1048576 bytes (B <= 85 at
 * K = 8, I = 768); larger sizes return WD_ERR_WORKSPACE_TOO_SMALL before any
 * launch.  The function allocates nothing and calls no allocating routine.
 *
 * The first call made with a given device current looks up that device's
 * address of the array (cudaGetSymbolAddress); make that first call before any
 * stream capture.  All calls share the one array: calls that can overlap on the
 * GPU (for instance on two streams with no ordering between them) race on it
 * and must not be issued.  Nothing in the array needs clearing, since each call
 * writes every h element it later reads.  Out-of-range expert ids contribute
 * nothing, as in wd_moe_decode, but are not reported (no error flag is kept).
 * Arguments, layouts and the other checks are those of wd_moe_decode. */
WD_API wd_status wd_moe_decode_no_alloc(const void* x, const int32_t* topk_ids,
                                        const float* topk_w, const uint8_t* gate_up,
                                        const uint8_t* gate_up_scale, const uint8_t* down,
                                        const uint8_t* down_scale, void* out, int B, int H, int I,
                                        int E, int K, wd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WD_MOE_H_ */
