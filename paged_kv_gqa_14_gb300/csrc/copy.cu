// pkv_copy: a byte copy between two buffers the GPU can address -- device memory, or pinned
// host memory under unified addressing -- done by a kernel instead of a copy engine.  On a
// Grace-Blackwell part the SMs reach pinned host memory over NVLink-C2C, so a step's staged
// inputs can go up, and its output come back, as one stream-ordered kernel each.
#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                            int64_t n16) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" PKV_API int pkv_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes) & 15u) return PKV_ERR_ALIGN;
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  const int64_t want = (n16 + kCopyThreads - 1) / kCopyThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 4;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  // the launch's own status (not cudaGetLastError, which would also report, and clear, an
  // error left by unrelated earlier work)
  const cudaError_t e = launch_kernel(false, copy_kernel, dim3(grid), dim3(kCopyThreads), 0,
                                      static_cast<cudaStream_t>(stream), static_cast<uint4*>(dst),
                                      static_cast<const uint4*>(src), n16);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
