// expand.cu -- decode a whole stored trellis matrix to bf16, bit-exact.
//
// What is computed ("trellis-linear.ts" diff page: expandTrellis /
// EXPAND_SOURCE; "trellis-vector-expand.ts"):
//   out[r][c] = bf16( fl32( value(s(r,c)) * scale[r] ) ),
// value = the correctly rounded fp32 quotient y / 147.800537109375.
//
// GB300 design: one warp per (row, block); lane j owns the 8 adjacent
// positions 8j .. 8j+7, whose windows all lie in one 64-bit span that starts
// at bit (T-8(j+1))*k.  The lane aligns the two words covering the span once,
// takes its 8 windows with compile-time shifts, and writes its 16 output
// bytes with one 128-bit streaming store, so the warp's store covers the
// block's 512 output bytes contiguously.  The kernel is bound by the HBM write
// of the 2-byte outputs (plus the k/8-byte code reads).
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace trellis {

template <int K, int L>
__global__ void __launch_bounds__(256) expand_kernel(const uint32_t* __restrict__ codes,
                                                     const uint16_t* __restrict__ scales,
                                                     uint16_t* __restrict__ out, int64_t rows, int nb) {
  constexpr int WPB = kT * K / 32;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= rows * nb) return;
  const int64_t row = gw / nb;
  const int blk = (int)(gw - row * nb);
  const uint32_t* bw = codes + (row * nb + blk) * WPB;

  const int lo = (kT - 8 * (lane + 1)) * K;  // first bit of the lane's span
  const int wa = lo >> 5, sh = lo & 31;
  const uint32_t a = __ldg(bw + wa);
  const uint32_t b = __ldg(bw + (wa + 1 == WPB ? 0 : wa + 1));
  uint32_t w[2];
  w[0] = __funnelshift_r(a, b, sh);
  w[1] = b >> sh;
  const float scale = f16_to_f32(__ldg(scales + row));

  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t s = window_at<L, 2>(w, (7 - i) * K);  // position 8*lane + i
    v[i] = __fmul_rn(value_rn(code_y(s)), scale);
  }
  uint4 o;
  o.x = pack_bf16x2(v[0], v[1]);
  o.y = pack_bf16x2(v[2], v[3]);
  o.z = pack_bf16x2(v[4], v[5]);
  o.w = pack_bf16x2(v[6], v[7]);
  __stcs(reinterpret_cast<uint4*>(out + (row * nb + blk) * kT) + lane, o);
}

cudaError_t launch_expand_bf16(const uint32_t* codes, const uint16_t* scales, uint16_t* out, int k, int L,
                               int64_t rows, int64_t cols, cudaStream_t st) {
  const int nb = (int)(cols / kT);
  const int64_t warps = rows * nb;
  const dim3 block(256), grid((unsigned)((warps + 7) / 8));
  if (L == 16) {
    if (k == 2) expand_kernel<2, 16><<<grid, block, 0, st>>>(codes, scales, out, rows, nb);
    else if (k == 3) expand_kernel<3, 16><<<grid, block, 0, st>>>(codes, scales, out, rows, nb);
    else expand_kernel<4, 16><<<grid, block, 0, st>>>(codes, scales, out, rows, nb);
  } else {
    if (k == 2) expand_kernel<2, 12><<<grid, block, 0, st>>>(codes, scales, out, rows, nb);
    else if (k == 3) expand_kernel<3, 12><<<grid, block, 0, st>>>(codes, scales, out, rows, nb);
    else expand_kernel<4, 12><<<grid, block, 0, st>>>(codes, scales, out, rows, nb);
  }
  return cudaGetLastError();
}

}  // namespace trellis
