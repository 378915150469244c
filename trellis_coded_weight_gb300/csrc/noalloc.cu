// noalloc.cu -- trellis_matvec_axis0_noalloc: the axis-0 matvec for callers
// that cannot allocate device memory.
//
// trellis_matvec_axis0 needs a caller-supplied workspace for its split-row
// partial sums and arrival counters.  Some callers have no way to provide one:
// a custom-operator slot in an inference engine that hands a kernel only its
// input and output tensors, or a serving runtime that plans all device memory
// up front and forbids cudaMalloc afterwards (cudaMalloc can synchronise the
// device and can fail once memory is fragmented).  This entry point takes the
// workspace from a fixed array in device memory that the library itself
// defines, so it allocates nothing at call time.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes bytes.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address: each call looks the
// address up with cudaGetSymbolAddress (with the caller's device current) and
// keeps it per device.  A call made while its stream is being captured into a
// CUDA graph uses the kept address instead of looking it up, so the first call
// on each device should come before any stream capture.  Looking the address
// up again on ordinary calls keeps it valid after cudaDeviceReset, which
// reloads the module and may move the array.  All calls share the one array:
// the arrival counters are cleared on the caller's stream before every
// launch, and calls whose executions overlap on the GPU race on the shared
// partial sums.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "launch.h"
#include "trellis.h"

namespace {

constexpr size_t kNoAllocScratchBytes = TRELLIS_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDev];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device, or nullptr on a
// CUDA error (or during capture before any ordinary call on this device).
void* scratch_for_current_device(cudaStream_t s) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return nullptr;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int trellis_matvec_axis0_noalloc(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                            uint16_t* out, int M, const trellis_geom_t* g,
                                            trellis_stream_t stream) {
  const int st = trellis_check_geom(g);
  if (st) return st;
  if (g->axis != 0) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!codes || !scales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(out)) return TRELLIS_EALIGN;
  const size_t need = trellis_workspace_bytes(M, g);
  if (need == 0 || need > kNoAllocScratchBytes) return TRELLIS_EWORKSPACE;

  int major = 0, minor = 0, dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3) {
    cudaGetLastError();
    return TRELLIS_EDEVICE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = scratch_for_current_device(s);
  if (!ws) return TRELLIS_ECUDA;

  // The arrival counters follow the partial sums; they must start at zero.
  const size_t counters = need - (((size_t)(g->cols / g->T) * sizeof(uint32_t) + 15) & ~(size_t)15);
  if (cudaMemsetAsync(static_cast<char*>(ws) + counters, 0, need - counters, s) != cudaSuccess) return TRELLIS_ECUDA;
  const cudaError_t e =
      trellis::launch_matvec_axis0(codes, scales, x, out, M, g->k, g->L, g->rows, g->cols, g->interleave, ws, s);
  return e == cudaSuccess ? TRELLIS_OK : TRELLIS_ECUDA;
}
