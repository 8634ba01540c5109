// wd_bench.cu - copy / read / fill kernels that measure this GPU's memory
// bandwidth for the layer's roofline (declared in include/wd_bench.h).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wd_bench.h"
#include "wd_device.cuh"

namespace {

// 32 bytes, read-only, no L1 allocation.  The copy kernel's loads are plain
// asm (the compiler may batch them: their values feed the stores); the read
// kernel's are volatile so that its loop is issued as written.
__device__ __forceinline__ wd::U32x8 ld_copy_32B(const void* p) {
  wd::U32x8 r;
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
        "=r"(r.v[6]), "=r"(r.v[7])
      : "l"(p));
  return r;
}

__device__ __forceinline__ void st_32B(void* p, const wd::U32x8& v) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.v[0]),
               "r"(v.v[1]), "r"(v.v[2]), "r"(v.v[3]), "r"(v.v[4]), "r"(v.v[5]), "r"(v.v[6]),
               "r"(v.v[7])
               : "memory");
}

__device__ __forceinline__ wd::U32x8 ld_stream_32B(const void* p) {
  wd::U32x8 r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]),
                 "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
               : "l"(p));
  return r;
}

// Grid-stride copy with four 32-byte loads in flight per thread before their
// stores.
__global__ void __launch_bounds__(256) copy_kernel(uint8_t* __restrict__ dst,
                                                   const uint8_t* __restrict__ src, size_t n32) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n32; i += 4 * stride) {
    const wd::U32x8 a = ld_copy_32B(src + i * 32);
    const wd::U32x8 b = ld_copy_32B(src + (i + stride) * 32);
    const wd::U32x8 c = ld_copy_32B(src + (i + 2 * stride) * 32);
    const wd::U32x8 d = ld_copy_32B(src + (i + 3 * stride) * 32);
    st_32B(dst + i * 32, a);
    st_32B(dst + (i + stride) * 32, b);
    st_32B(dst + (i + 2 * stride) * 32, c);
    st_32B(dst + (i + 3 * stride) * 32, d);
  }
  for (; i < n32; i += stride) st_32B(dst + i * 32, ld_copy_32B(src + i * 32));
}

__global__ void __launch_bounds__(256) read_kernel(const uint8_t* __restrict__ src, size_t n32,
                                                   uint32_t* __restrict__ sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  uint32_t acc = 0;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  // two loads in flight per iteration
  for (; i + stride < n32; i += 2 * stride) {
    const wd::U32x8 a = ld_stream_32B(src + i * 32);
    const wd::U32x8 b = ld_stream_32B(src + (i + stride) * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc ^= a.v[k] + b.v[k];
  }
  for (; i < n32; i += stride) {
    const wd::U32x8 a = ld_stream_32B(src + i * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc ^= a.v[k];
  }
  if (acc == 0x9E3779B9u) atomicAdd(sink, 1u);  // keeps the loads live; practically never taken
}

__global__ void __launch_bounds__(256) fill_kernel(uint8_t* __restrict__ buf, size_t n32,
                                                   uint32_t value) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n32; i += stride)
    asm volatile("st.global.v8.u32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1};" ::"l"(buf + i * 32),
                 "r"(value)
                 : "memory");
}

// One thread that returns once `ns` nanoseconds of %globaltimer have passed
// (or after a fixed number of polls, whichever comes first).
__global__ void hold_kernel(unsigned long long ns) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < (1 << 22); ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= ns) break;
    __nanosleep(1000);
  }
}

bool ok32(const void* p, size_t bytes) {
  return p && (reinterpret_cast<uintptr_t>(p) % 32) == 0 && bytes % 32 == 0;
}

int blocks_or_default(int blocks) {
  if (blocks > 0) return blocks;
  int sms = wd_bench_sm_count();
  return sms > 0 ? sms * 8 : 1024;
}

}  // namespace

extern "C" {

int wd_bench_sm_count(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

double wd_bench_spec_gbs(void) {
  int dev = 0, khz = 0, bits = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1.0;
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrMemoryClockRate, dev) != cudaSuccess) return -1.0;
  if (cudaDeviceGetAttribute(&bits, cudaDevAttrGlobalMemoryBusWidth, dev) != cudaSuccess) return -1.0;
  return 2.0 * khz * 1e3 * (bits / 8.0) / 1e9;
}

int wd_bench_copy(void* dst, const void* src, size_t bytes, int blocks, void* stream) {
  if (!ok32(dst, bytes) || !ok32(src, bytes)) return (int)cudaErrorInvalidValue;
  copy_kernel<<<blocks_or_default(blocks), 256, 0, (cudaStream_t)stream>>>(
      (uint8_t*)dst, (const uint8_t*)src, bytes / 32);
  return (int)cudaGetLastError();
}

int wd_bench_read(const void* src, size_t bytes, uint32_t* sink, int blocks, void* stream) {
  if (!ok32(src, bytes) || !sink) return (int)cudaErrorInvalidValue;
  read_kernel<<<blocks_or_default(blocks), 256, 0, (cudaStream_t)stream>>>((const uint8_t*)src,
                                                                          bytes / 32, sink);
  return (int)cudaGetLastError();
}

int wd_bench_fill(void* buf, size_t bytes, uint32_t value, int blocks, void* stream) {
  if (!ok32(buf, bytes)) return (int)cudaErrorInvalidValue;
  fill_kernel<<<blocks_or_default(blocks), 256, 0, (cudaStream_t)stream>>>((uint8_t*)buf,
                                                                          bytes / 32, value);
  return (int)cudaGetLastError();
}

int wd_bench_hold(unsigned int microseconds, void* stream) {
  if (microseconds > 1000000u) return (int)cudaErrorInvalidValue;
  hold_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(1000ull * microseconds);
  return (int)cudaGetLastError();
}

}  // extern "C"
