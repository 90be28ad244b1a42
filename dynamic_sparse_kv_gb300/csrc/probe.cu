// Read-only streaming probe (fastocr_read_probe): the bandwidth at which this
// GPU delivers a large buffer that is only read, once. The attend kernels
// only read the K/V cache, so this is the honest ceiling for their streaming;
// a copy (read + write) is the other denominator a benchmark can report.
#include <stdint.h>

#include <cuda_runtime.h>

#include "fastocr.h"

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;   // 16-byte loads in flight per thread

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Every 16-byte word of src[0, n16) is loaded once (grid-stride, kProbeUnroll
// independent loads per thread per round) and folded into one XOR that is
// ORed into *sink, so no load can be dropped.
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4* __restrict__ src,
                                                                  size_t n16, uint32_t* sink) {
  const size_t stride = (size_t)gridDim.x * kProbeThreads;
  size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_stream(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc == 0x5eed5eedu) atomicOr(sink, acc);
}

}  // namespace

extern "C" fastocr_status fastocr_read_probe(const void* src, int64_t bytes, uint32_t* sink,
                                             fastocr_stream stream) {
  if (!src || !sink) return FASTOCR_ERR_NULL;
  if (bytes < 16 || bytes % 16 != 0) return FASTOCR_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return FASTOCR_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FASTOCR_ERR_NO_DEVICE;
  // four 512-thread blocks fill an SM's 2048 thread slots
  read_probe_kernel<<<4 * sms, kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), (size_t)bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? FASTOCR_OK : FASTOCR_ERR_CUDA;
}
