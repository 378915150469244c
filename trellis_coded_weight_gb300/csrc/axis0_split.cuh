// axis0_split.cuh -- the balanced split of an axis-0 matvec over the GPU and the deterministic fold of its
// partial sums, shared by the CUDA-core kernel (matvec_axis0.cu) and the tensor-core kernel
// (matvec_axis0_tc.cu).
//
// The sum over stored rows is split as the pages split it ("trellis-linear.ts" diff page: the scatter path's
// partial fold; "trellis-balanced-scatter.ts"), but balanced: the work is the list of (column block, stored
// row) pairs, column block major, and CTA c of G takes the contiguous range [c*N/G, (c+1)*N/G).  A range
// crosses at most a few column blocks; each piece is a segment.  At the end of a segment a CTA writes one fp32
// partial per output to the workspace in slot c + cb (unique per CTA and column block).  The last CTA to
// arrive for a column block (an atomic counter against the known number of CTAs that cover it) folds the
// partials in CTA order, applies 1/d (default numerics), stores bf16 and resets the counter -- one launch,
// deterministic, no atomics on data.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace trellis {

constexpr int kAx0MaxCtas = 256;         // bound on the grid (sizes the workspace)
constexpr int64_t kAx0MinRows = 64;      // fewest (column block, row) pairs per CTA
constexpr int kAx0MaxPending = 4;        // segments whose arrival waits for one fence

struct Ax0Params {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* out;
  float* part;        // [kAx0MaxCtas + nb][M][256]
  uint32_t* counter;  // [nb]
  int64_t R, C, N;    // rows, cols, N = nb * R work items
  int nb, G;          // column blocks, CTAs
  int stage;          // rows of x staged at once (CUDA-core kernel)
};

// CTAs of a launch over N work items: one per SM, at most kAx0MaxCtas, and at least kAx0MinRows items each.
inline int ax0_grid(int64_t N) {
  int64_t G = device_sm_count();
  if (G > kAx0MaxCtas) G = kAx0MaxCtas;
  if (G > (N + kAx0MinRows - 1) / kAx0MinRows) G = (N + kAx0MinRows - 1) / kAx0MinRows;
  return G < 1 ? 1 : (int)G;
}

// The CTA whose range holds work item f: the largest c with c*N/G <= f.
__device__ __forceinline__ int ax0_cta_of(int64_t f, int64_t N, int G) { return (int)(((f + 1) * G - 1) / N); }

// Publishes the partial just written for column block cb (slot c + cb).  Arrival is deferred: a range that
// crosses column blocks publishes up to kAx0MaxPending partials with one fence.  `range_done` marks the CTA's
// last segment.  Every thread of the CTA calls this; it ends with a barrier, so shared memory written before
// it may be reused after it.  BW: the partials already hold scaled weights (no 1/d).
// Counter arrival with acquire-release semantics at GPU scope: the CTA's partials (written before the barrier
// that precedes this call) are visible to whichever CTA later reads the counter's final value, and the last CTA
// sees every other CTA's partials.
__device__ __forceinline__ uint32_t ax0_arrive(uint32_t* counter) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

template <int M, bool BW>
__device__ __forceinline__ void ax0_publish(const Ax0Params& p, int (&pend)[kAx0MaxPending],
                                            uint32_t (&is_last)[kAx0MaxPending], int& npend, int cb,
                                            bool range_done) {
  if (threadIdx.x == 0) pend[npend] = cb;
  if (++npend == kAx0MaxPending || range_done) {
    __syncthreads();  // every thread's partial stores precede thread 0's release
    if (threadIdx.x == 0)
      for (int i = 0; i < npend; ++i) {
        const int pc = pend[i];
        const int first = ax0_cta_of((int64_t)pc * p.R, p.N, p.G);
        const int last = ax0_cta_of((int64_t)pc * p.R + p.R - 1, p.N, p.G);
        is_last[i] = (ax0_arrive(p.counter + pc) == (uint32_t)(last - first)) ? 1u : 0u;
      }
    __syncthreads();  // ... and thread 0's acquire precedes every thread's loads below
    for (int i = 0; i < npend; ++i) {
      if (!is_last[i]) continue;
      // the last CTA to arrive folds the column block's partials in CTA order, all of a thread's loads in flight
      // at once (M*256 outputs over at least 256 threads: at most 4 per thread)
      const int pc = pend[i];
      const int first = ax0_cta_of((int64_t)pc * p.R, p.N, p.G);
      const int ns = ax0_cta_of((int64_t)pc * p.R + p.R - 1, p.N, p.G) - first + 1;
      const float* ps = p.part + (int64_t)(first + pc) * M * kT;
      constexpr int kPer = (M * kT + 255) / 256;
      constexpr int kBatch = 16 / kPer;  // partials per output in flight: 16 loads per thread
      float v[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) v[u] = 0.f;
      for (int s0 = 0; s0 < ns; s0 += kBatch) {
        float q[kPer][kBatch];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int e = threadIdx.x + u * (int)blockDim.x;
#pragma unroll
          for (int j = 0; j < kBatch; ++j)
            q[u][j] = (e < M * kT && s0 + j < ns) ? __ldcg(ps + (int64_t)(s0 + j) * M * kT + e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u)
#pragma unroll
          for (int j = 0; j < kBatch; ++j)
            if (s0 + j < ns) v[u] += q[u][j];
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = threadIdx.x + u * (int)blockDim.x;
        if (e < M * kT) {
          const int m = e / kT, t = e - m * kT;
          p.out[(int64_t)m * p.C + (int64_t)pc * kT + t] = f32_to_bf16_rn(BW ? v[u] : __fmul_rn(v[u], kRcpD));
        }
      }
      if (threadIdx.x == 0) p.counter[pc] = 0u;
    }
    npend = 0;
  }
  __syncthreads();  // shared memory of the segment (and pend, is_last) may be reused
}

}  // namespace trellis
