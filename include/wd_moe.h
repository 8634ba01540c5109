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
 * computed by kernels organised around outputs rather than experts.  While
 * tokens rarely share experts (2*B*K < E: B <= 4 at K = 8, E = 128) they are
 * the pages' two kernels:
 *   moe_gate_up_3d_batched - one warp per (token, routed expert, intermediate
 *                            neuron): streams that neuron's gate and up rows
 *                            once, dots both against x, writes one BF16 value;
 *   moe_down_3d_batched    - one warp per (token, output dim): walks all K
 *                            routed experts' down rows and folds the weighted
 *                            contributions into one FP32 register accumulator,
 *                            reduces across the warp with shuffles, writes once.
 * Once tokens share experts, the same outputs come from kernels that read and
 * dequantise every routed row once for all (token, slot) pairs routed to its
 * expert, with the products on the tensor cores (mma.sync, FP16 operands
 * re-encoded exactly from E4M3 and from BF16 by per-row powers of two, FP32
 * accumulation):
 *   moe_gate_up_mma        - one CTA per SM over (expert, 16 neurons) items;
 *   moe_h_encode           - h re-encoded once per call as FP16 x 2^k per row;
 *   moe_down_dimblock      - one CTA per 16 output dims over every routed
 *                            expert, each output written once.
 * wd_moe_describe_plan names the kernels a shape gets.  There is no padding, no
 * gather of activations into expert-major buffers and no combine pass (section
 * 阶段消除 [Stage elimination], section 消除缓冲区 [Eliminating buffers]).
 * Activations are BF16, accumulation is FP32 and the weights are dequantised
 * from MXFP8 as they stream in (section 精度提升 [Accuracy gains]).
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
 *                  BF16 intermediate h [B, K, I], then its FP16 re-encoding
 *                  [B, K, I] and int32 exponents [B, K] (each region rounded
 *                  up to 256 bytes); a workspace sized for a batch B serves
 *                  every smaller batch
 *
 * Requirements checked on the host (a violation returns an error, nothing is
 * launched): non-null pointers; B >= 1; 1 <= K <= E; H and I multiples of 32
 * with H <= 16384 and I <= 16384; K <= 64; B <= 4096; x, gate_up and down
 * 32-byte aligned; gate_up_scale, down_scale, topk_ids, topk_w, out and
 * workspace 4-byte aligned (the workspace 256-byte aligned); workspace_bytes
 * large enough.
 *
 * Expert ids are range-checked on the device: an id outside [0, E) contributes
 * nothing (its h entries are written as 0) and sets bit 0 of the workspace
 * error flag, which stays set until wd_moe_read_error_flag reads and clears
 * it.  Duplicate ids within a token are allowed; their contributions add.
 * No kernel reduces through atomics: every result is bit-reproducible from
 * run to run.
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
  WD_ERR_BAD_EXPERT_ID = 5,       /* reported by wd_moe_read_error_flag only     */
  WD_ERR_PIPELINE_TIMEOUT = 6     /* reported by wd_moe_read_error_flag only     */
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

/* The MoE decode layer: the plan's two or three kernels back to back on
 * `stream` (wd_moe_describe_plan names them and says which are launched as
 * programmatic dependents of the one before, so that their weight loads start
 * while it drains; each waits for its predecessor's results before reading
 * them).  See the file comment for the layout and the definition.  h is left
 * in the workspace. */
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

/* The down stage alone with a workspace (the kernels wd_moe_decode runs after
 * the gate/up kernel, chosen by the same plan): out [B, H] BF16 from a
 * caller-given h [B, K, I] BF16 (32-byte aligned; it may be the workspace's
 * own h region), topk_ids, topk_w and the down weights.  The workspace
 * (wd_moe_workspace_size(B, K, I) bytes, initialised) supplies the scratch of
 * the shared-row form (h re-encoded as FP16 with per-row exponents) and the
 * error flag.  Section 两个 kernel 如何工作, down paragraph. */
WD_API wd_status wd_moe_down_workspace(const void* h, const int32_t* topk_ids,
                                       const float* topk_w, const uint8_t* down,
                                       const uint8_t* down_scale, void* out, void* workspace,
                                       size_t workspace_bytes, int B, int H, int I, int E, int K,
                                       wd_stream_t stream);

/* The first kernel of the shared-row down stage alone (moe_h_encode): each
 * of the `rows` rows of h (BF16 [rows, I], 16-byte aligned) is written to h16
 * (FP16 [rows, I], 16-byte aligned) as h * 2^k with k = hk[row] (int32
 * [rows]) chosen so that the row's largest magnitude lies in [2^14, 2^15)
 * (k = 0 for a row that is all zero or holds Inf/NaN).  Power-of-two scaling
 * is exact; every BF16 value within 2^31 of its row's largest magnitude is
 * exactly an FP16 value after it. */
WD_API wd_status wd_moe_h_encode(const void* h, void* h16, int32_t* hk, int rows, int I,
                                 wd_stream_t stream);

/* The second kernel of the shared-row down stage alone (moe_down_dimblock):
 * out [B, H] BF16 from moe_h_encode's output for the B*K rows of h (h16
 * 16-byte aligned, hk), topk_ids, topk_w and the down weights (down_scale
 * 16-byte aligned).  `error_flag` as in wd_moe_gate_up (may be NULL).  Needs
 * B <= 64, B*K <= 256, H % 16 == 0, I % 128 == 0, I <= 2048 and E*H < 2^31,
 * else WD_ERR_UNSUPPORTED_SHAPE.  Runs with the plan's ring depth where the
 * plan picks this kernel for the shape, else the deepest that fits.  Section 两个 kernel 如何工作, down paragraph. */
WD_API wd_status wd_moe_down_encoded(const void* h16, const int32_t* hk, const int32_t* topk_ids,
                                     const float* topk_w, const uint8_t* down,
                                     const uint8_t* down_scale, void* out, uint32_t* error_flag,
                                     int B, int H, int I, int E, int K, wd_stream_t stream);

/* Copy the workspace's error flag to `*flag` and clear it.  This call
 * SYNCHRONISES `stream`.  The flag is a bit mask accumulated over every call
 * since the last read:
 *   bit 0 (1): an expert id outside [0, E) was seen; that (token, slot)
 *              contributed nothing and the rest of the output is valid;
 *   bit 1 (2): a bounded wait inside a kernel that streams weights through a
 *              shared-memory ring ran out (about 2 s of SM clock without the
 *              awaited copy landing); the kernel stopped early and the output
 *              of that call is INVALID.
 * Returns WD_ERR_PIPELINE_TIMEOUT when bit 1 is set (whatever bit 0 is), else
 * WD_ERR_BAD_EXPERT_ID when bit 0 is set, else WD_OK; `*flag` receives the
 * mask (0..3) in every case where the copy succeeded. */
WD_API wd_status wd_moe_read_error_flag(void* workspace, size_t workspace_bytes,
                                       wd_stream_t stream, int* flag);

/* Name of the CUDA error (cudaGetErrorName) behind the calling thread's most
 * recent WD_ERR_CUDA, or "none".  Static storage; never NULL. */
WD_API const char* wd_last_error_string(void);

/* The most kernel launches one wd_moe_decode call issues (3). */
WD_API int wd_moe_launches_per_call(void);

/* Kernel launches wd_moe_decode issues for this shape under the current plan
 * (2 or 3; 0 for invalid dimensions).  Host-only. */
WD_API int wd_moe_launches(int B, int H, int I, int E, int K);

/* Override the per-shape launch plan (tuning and tests; not needed in normal
 * use).  `spec` is a comma-separated list of
 *   "gu=batched:<neurons per warp>:<blocks per lane per pass>"
 *   "gu=rowshare:<neurons per warp>:<words per step>"   (tokens share rows)
 *   "gu=persist:<neurons per warp>:<1 + L2 prefetch distance>"
 *   "gu=mma[:<ring stages, 2..4>[:<consumer warps, 8 or 16>]]"
 *                                   (tensor-core products; B*K <= 256,
 *                                    H % 512 == 0, H <= 2048, I % 16 == 0)
 *   "dn=<output dims per warp>:<blocks per lane per pass>"
 *   "dn=dimblock[:<ring stages, even, 2..8; consumer warps = stages / 2>]"
 *                 (moe_h_encode + moe_down_dimblock; B <= 64, B*K <= 256,
 *                 H % 16 == 0, I % 128 == 0, a two-stage ring fitting in
 *                 shared memory: I <= 2048)
 *   "rowshare_min_b=<smallest batch that uses the shared-row gate/up kernel
 *                    where the persistent one does not apply>"
 *   "pdl=<0..7>" (programmatic dependent launch: bit i lets launch i of the
 *                 call start before launch i - 1 has finished; for i = 0,
 *                 whatever precedes the call on the stream)
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
 * "gate_up=<kernel><params> down=<kernel><params> pdl=<mask> launches=<n>" (the
 * mask as in wd_moe_set_plan's "pdl="; down=moe_down_dimblock stands for
 * moe_h_encode followed by moe_down_dimblock), NUL-terminated, into
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
 * The scratch that wd_moe_decode keeps in its workspace (the intermediate h
 * and, where the plan uses it, h's FP16 re-encoding and exponents) lives here
 * in a 2 MiB array compiled into the library (file-scope device memory that
 * every GPU loading the library holds until the process exits), laid out as a
 * workspace, so wd_moe_workspace_size(B, K, I) must be at most 2097152 bytes
 * (B <= 85 at K = 8, I = 768); larger sizes return WD_ERR_WORKSPACE_TOO_SMALL
 * before any launch.  The call launches the same kernels in the same order as
 * wd_moe_decode and gives the same output bit for bit.  The function
 * allocates nothing and calls no allocating routine.
 *
 * The first call made with a given device current looks up that device's
 * address of the array (cudaGetSymbolAddress); make that first call before any
 * stream capture.  All calls share the one array: calls that can overlap on the
 * GPU (for instance on two streams with no ordering between them) race on it
 * and must not be issued.  Nothing in the array needs clearing, since each
 * kernel of a call writes every element the next one reads.  No error flag is
 * kept: out-of-range expert ids contribute nothing, as in wd_moe_decode, but
 * are not reported, and neither is a bounded wait that runs out inside a
 * kernel (whose output is then invalid).  Arguments, layouts and the other
 * checks are those of wd_moe_decode. */
WD_API wd_status wd_moe_decode_no_alloc(const void* x, const int32_t* topk_ids,
                                        const float* topk_w, const uint8_t* gate_up,
                                        const uint8_t* gate_up_scale, const uint8_t* down,
                                        const uint8_t* down_scale, void* out, int B, int H, int I,
                                        int E, int K, wd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WD_MOE_H_ */
