/*
 * wd_bench.h - memory-bandwidth reference kernels for measuring the layer.
 *
 * The warp-decode blog (Cursor, "用 warp decode 实现更好的 MoE 模型推理",
 * section 硬件效率 [Hardware efficiency]) states its layer throughput as a
 * fraction of the peak a copy kernel reaches with sequential reads.  These
 * kernels give that denominator on the machine at hand:
 *   wd_bench_copy  - dst[i] = src[i], 32-byte vectors, grid-stride with four
 *                    loads in flight per thread; bytes moved = 2 * bytes
 *                    (read + write), the copy-kernel convention;
 *   wd_bench_read  - streams src once (read only) and folds it into *sink;
 *   wd_bench_fill  - writes a pattern over buf (used to evict L2 between timed
 *                    runs when buf is larger than L2);
 *   wd_bench_hold  - occupies `stream` for a while with one thread, so that the
 *                    host can queue a long run of short launches behind it and
 *                    time each one on the device without the gaps of the
 *                    host's own launch rate.
 * All pointers are device pointers owned by the caller; src/dst/buf must be
 * 32-byte aligned and `bytes` a multiple of 32.  `blocks` is the grid size
 * (0: 8 CTAs of 256 threads per SM).  Asynchronous on `stream`; returns 0 on
 * success, else the cudaError_t of the launch.
 */
#ifndef WD_BENCH_H_
#define WD_BENCH_H_

#include <stddef.h>
#include <stdint.h>

#ifndef WD_API
#define WD_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

WD_API int wd_bench_copy(void* dst, const void* src, size_t bytes, int blocks, void* stream);
WD_API int wd_bench_read(const void* src, size_t bytes, uint32_t* sink, int blocks, void* stream);
WD_API int wd_bench_fill(void* buf, size_t bytes, uint32_t value, int blocks, void* stream);

/* One single-thread kernel on `stream` that returns after `microseconds`
 * (at most 1,000,000; larger values return cudaErrorInvalidValue) of the
 * device's global timer have passed.  0 on success, else the launch's error. */
WD_API int wd_bench_hold(unsigned int microseconds, void* stream);

/*
 * The expert-centric layer warp decode is compared against (benchmark only;
 * no wd_moe.h entry point reaches it).  Cursor, "用 warp decode 实现更好的 MoE
 * 模型推理", section 传统的 MoE 路径 [The traditional MoE path], and the stages
 * that sections 阶段消除 [Stage elimination] and 消除缓冲区 [Eliminating buffers]
 * say warp decode removes.  Five launches on `stream`:
 *   routing metadata (per-expert counts padded to powers of two, offsets),
 *   gather of x into an expert-major buffer, grouped gate/up GEMV into an
 *   expert-major h, grouped down GEMV into a per-expert output buffer (BF16,
 *   K rows of H per token), and the weighted combine into out.
 * Same arguments, layouts and alignment as wd_moe_decode (include/wd_moe.h);
 * `workspace` (256-byte aligned, at least
 * wd_bench_expert_centric_workspace_size bytes, device memory owned by the
 * caller) holds the metadata and the three buffers.  The result is the
 * layer's definition with one extra BF16 rounding of each expert's
 * contribution (the per-expert output buffer) before the combine.  Ids
 * outside [0, E) contribute nothing and are not reported.  Returns 0, or
 * cudaErrorInvalidValue (1) for bad arguments or shapes (H, I multiples of 32
 * up to 4096, E <= 4096, B*K <= 131072), or the launch's cudaError_t.
 */
WD_API size_t wd_bench_expert_centric_workspace_size(int B, int H, int I, int E, int K);
WD_API int wd_bench_expert_centric(const void* x, const int32_t* topk_ids, const float* topk_w,
                                   const uint8_t* gate_up, const uint8_t* gate_up_scale,
                                   const uint8_t* down, const uint8_t* down_scale, void* out,
                                   void* workspace, size_t workspace_bytes, int B, int H, int I,
                                   int E, int K, void* stream);

/* Number of streaming multiprocessors of the current device (or -1). */
WD_API int wd_bench_sm_count(void);

/* Spec DRAM bandwidth of the current device in GB/s: 2 (double data rate)
 * x peak memory clock x bus width / 8, from the device attributes; -1 on error. */
WD_API double wd_bench_spec_gbs(void);

#ifdef __cplusplus
}
#endif

#endif /* WD_BENCH_H_ */
