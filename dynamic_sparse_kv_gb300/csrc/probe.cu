// Streaming utilities around the method's kernels.
//
// fastocr_read_probe: the bandwidth at which this GPU delivers a large buffer
// that is only read, once. The attend kernels only read the K/V cache, so
// this is the honest ceiling for their streaming; a copy (read + write) is
// the other denominator a benchmark can report.
//
// fastocr_copy: a copy done by the SMs instead of a copy engine, so that it
// sits in a chain of kernels launched with programmatic dependent launch.
// Either side may be page-locked host memory, which the SMs address directly
// under unified addressing (over NVLink-C2C on a Grace-Blackwell node).
#include <stdint.h>

#include <algorithm>

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

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;   // 16-byte loads in flight per thread before its stores

// dst[0, n16) = src[0, n16), grid-stride. The kernel before it in the stream
// may still read dst or write src until it completes, so the copy starts
// after griddepcontrol.wait; the next kernel may start its own pre-wait work
// at once (it waits for this grid to complete before it reads dst).
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4* __restrict__ dst,
                                                            const uint4* __restrict__ src,
                                                            size_t n16) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * stride < n16; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) v[u] = ld_stream(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) dst[i] = ld_stream(src + i);
}

// The address the device uses for p: device or managed memory as it is,
// page-locked host memory through its device mapping; nullptr for memory the
// device cannot address (pageable host memory) or that CUDA does not know.
const void* device_address(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return a.devicePointer;
    default:
      return nullptr;
  }
}

}  // namespace

extern "C" fastocr_status fastocr_copy(void* dst, const void* src, int64_t bytes,
                                       fastocr_stream stream) {
  if (!dst || !src) return FASTOCR_ERR_NULL;
  if (bytes < 0 || bytes % 16 != 0) return FASTOCR_ERR_INVALID;
  if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) != 0)
    return FASTOCR_ERR_ALIGN;
  const char* d = static_cast<const char*>(dst);
  const char* s = static_cast<const char*>(src);
  if (bytes > 0 && d < s + bytes && s < d + bytes) return FASTOCR_ERR_INVALID;   // overlap
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FASTOCR_ERR_NO_DEVICE;
  const void* dd = device_address(dst);
  const void* sd = device_address(src);
  if (!dd || !sd) return FASTOCR_ERR_INVALID;
  if (bytes == 0) return FASTOCR_OK;
  const size_t n16 = (size_t)bytes / 16;
  const size_t per_cta = (size_t)kCopyThreads * kCopyUnroll;
  const unsigned grid = (unsigned)std::min<size_t>((n16 + per_cta - 1) / per_cta, 4 * (size_t)sms);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, copy_kernel, static_cast<uint4*>(const_cast<void*>(dd)),
                                           static_cast<const uint4*>(sd), n16);
  return e == cudaSuccess ? FASTOCR_OK : FASTOCR_ERR_CUDA;
}

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
