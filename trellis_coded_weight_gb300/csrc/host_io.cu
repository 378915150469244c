// host_io.cu -- moving a matvec's input in from host memory and its output back, for the host-buffer call
// (trellis_matvec_axis1_host): the decode call of the pages takes one token's activations from the host and
// hands the projected row back.
//
// GB300 design.  The GPU reaches the Grace host's memory over NVLink-C2C, and pinned host memory is mapped into
// the GPU's address space.  A copy-engine transfer on either side of the matvec costs little bandwidth but
// serialises the stream: the kernel behind a copy cannot start early, and the copy behind a kernel waits for its
// completion.  For pinned buffers the host call therefore
//   * brings x in with a small kernel (every thread one 16-byte load from host memory and one store into the
//     caller's device buffer), launched with programmatic dependent launch so that it and the matvec behind it
//     are scheduled while the previous kernel on the stream is still finishing;
//   * lets the matvec store its output rows straight into the pinned output buffer.
// Pageable buffers (or ones without a device mapping, or not 16-byte aligned) keep the copy-engine path.
#include <cstdint>
#include <cuda_runtime.h>

#include "launch.h"
#include "pdl.cuh"

namespace trellis {
namespace {

constexpr int kFetchThreads = 128;

// dst[i] = src[i] for i < n (16-byte units).  src lies in host memory (its device mapping).  The wait comes first:
// the grid ahead may still be writing memory this grid reads (a caller may pass the previous call's output buffer
// as this call's input), and every access of this grid follows stream order after it.
__global__ void __launch_bounds__(kFetchThreads) fetch_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                              int64_t n) {
  pdl_enter();
  const int64_t i = (int64_t)blockIdx.x * kFetchThreads + threadIdx.x;
  if (i < n) dst[i] = src[i];
}

}  // namespace

const void* mapped_host_view(const void* host) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr || a.hostPointer == nullptr) return nullptr;
  // hostPointer and devicePointer name the same byte (the allocation's first, or `host` itself), so the offset of
  // `host` from hostPointer carries over to the device mapping.
  const uintptr_t off = reinterpret_cast<uintptr_t>(host) - reinterpret_cast<uintptr_t>(a.hostPointer);
  return static_cast<const char*>(a.devicePointer) + off;
}

cudaError_t launch_fetch16(void* dst, const void* src_view, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  if (bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(dst) & 15u) || (reinterpret_cast<uintptr_t>(src_view) & 15u))
    return cudaErrorInvalidValue;
  const int64_t n = (int64_t)(bytes / 16);
  const int64_t blocks = (n + kFetchThreads - 1) / kFetchThreads;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  return launch_pdl(fetch_kernel, dim3((unsigned)blocks), dim3(kFetchThreads), 0, st, static_cast<uint4*>(dst),
                    static_cast<const uint4*>(src_view), n);
}

}  // namespace trellis
