// launch.h -- internal host-side launchers of the CUDA kernels (C++ only; the
// public C ABI is include/trellis.h).  Arguments are validated by abi.cu
// before these are called.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace trellis {

constexpr int kT_host = 256;  // positions per block, the only T the kernels support

// interleave: 0 row-major codes, 2 the k=3 axis-0 layout [cols/512][rows][48].
cudaError_t launch_expand_bf16(const uint32_t* codes, const uint16_t* scales, uint16_t* out, int k, int L,
                               int64_t rows, int64_t cols, int interleave, cudaStream_t st);

// Axis-1 matvec and fused gate/up (matvec_axis1_tc.cu): M = 1 on the CUDA cores, M >= 2 with y*x accumulated
// on the tensor cores.  The _fma forms take the CUDA-core path for every M.
cudaError_t launch_matvec_axis1(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                cudaStream_t st);
// The same two layers with the accumulation on the CUDA cores (packed fp32 FMA, matvec_axis1.cu).
cudaError_t launch_matvec_axis1_fma(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                    uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                    cudaStream_t st);
cudaError_t launch_gateup_swiglu_fma(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                                     const uint16_t* uscales, const uint16_t* x, uint16_t* out, int M, int k,
                                     int L, int64_t rows, int64_t cols, cudaStream_t st);
// Warps per CTA of the CUDA-core axis-1 kernel for a row of nb blocks at the given register count.
int mv1_splits(int nb, int regs);

// The same matvecs with bf16-rounded weights (bf16(value * scale) before the FMA).
cudaError_t launch_matvec_axis1_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                      uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                      cudaStream_t st);
cudaError_t launch_matvec_axis0_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                      uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                      void* workspace, cudaStream_t st);

cudaError_t launch_gateup_swiglu(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                                 const uint16_t* uscales, const uint16_t* x, uint16_t* out, int M, int k,
                                 int L, int64_t rows, int64_t cols, cudaStream_t st);

// Host buffers (host_io.cu).  mapped_host_view: the device address of pinned host memory mapped into the
// current device's address space, or nullptr (pageable memory, no mapping, a failed query).  launch_fetch16:
// copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from such a mapping into device memory with a
// kernel launched behind the stream's previous kernel by programmatic dependent launch.
const void* mapped_host_view(const void* host);
cudaError_t launch_fetch16(void* dst, const void* src_view, size_t bytes, cudaStream_t st);

// Workspace of the axis-0 matvec: fp32 partials followed by per-column-block
// arrival counters.  launch_matvec_axis0 takes the tensor-core kernel for M >= 3
// and the CUDA-core kernel for M <= 2.
size_t axis0_workspace_bytes(int M, int64_t rows, int64_t cols);
cudaError_t launch_matvec_axis0(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                void* workspace, cudaStream_t st);
// The two kernels behind it (same workspace layout): y * x*scale on the tensor cores (matvec_axis0_tc.cu, every
// M), or packed fp32 FMA on the CUDA cores (matvec_axis0.cu, every M; also the bf16-weight variant's kernel).
cudaError_t launch_matvec_axis0_tc(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                   uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                   void* workspace, cudaStream_t st);
cudaError_t launch_matvec_axis0_fma(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                    uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                    void* workspace, cudaStream_t st);

cudaError_t launch_gemm_prefill(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                uint16_t* out, int M, int k, int L, int axis, int64_t rows, int64_t cols,
                                cudaStream_t st);
// The prefill for small M: the decode in registers and mma.sync bf16 (up to four 8-token tiles), on axis 1
// (prefill_small.cu) and on axis 0 (prefill_axis0_small.cu, clusters folding the split reduction);
// launch_gemm_prefill takes them up to the measured crossovers with the tcgen05 kernel: 24 tokens on axis 1,
// 32 on axis 0.
constexpr int kPrefillSmallMaxM1 = 24;
constexpr int kPrefillSmallMaxM0 = 32;
constexpr int prefill_small_max_m(int axis) { return axis == 1 ? kPrefillSmallMaxM1 : kPrefillSmallMaxM0; }
cudaError_t launch_prefill_small(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                                 int M, int k, int L, int64_t rows, int64_t cols, cudaStream_t st);
cudaError_t launch_prefill_axis0_small(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                       uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                       cudaStream_t st);

// Tile plan of the prefill GEMM (host arithmetic only): tokens per tile and up
// to two launches over the output tiles, each [t0, t0 + count) with S CTAs per
// tile (S > 1: a cluster splitting the tile's reduction).  Returns the number
// of launches; 0 (and 0 tokens per tile) where the call takes a
// register-decode kernel instead (M <= prefill_small_max_m(axis)).
struct PrefillLaunch {
  int t0, count, S;
};
int prefill_plan(int M, int axis, int64_t nOut, int64_t Kd, int sms, int* tokens_per_tile, PrefillLaunch* launches);
// SM count of the current device (148 if it cannot be read).
int device_sm_count();

// Load-only floor of the axis-1 access pattern (no decode): out[r] = XOR of row r's words.
cudaError_t launch_load_floor(const uint32_t* codes, uint32_t* out, int k, int64_t rows, int64_t cols,
                              cudaStream_t st);
// Coalesced load floor: a warp per stored row, lanes on consecutive 16-byte chunks.
cudaError_t launch_load_floor_rows(const uint32_t* codes, uint32_t* out, int k, int64_t rows, int64_t cols,
                                   cudaStream_t st);

// Device error word of the tensor-core kernels (bounded waits that gave up).
int read_device_error(int reset);
// Limit of each bounded wait of the tensor-core kernels for later launches (ns; 0: the 2 s default).
void set_wait_limit_ns(uint64_t ns);

}  // namespace trellis
