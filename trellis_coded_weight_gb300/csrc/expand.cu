// expand.cu -- decode a whole stored trellis matrix to bf16, bit-exact.
//
// What is computed ("trellis-linear.ts" diff page: expandTrellis /
// EXPAND_SOURCE; "trellis-vector-expand.ts"):
//   out[r][c] = bf16( fl32( value(s(r,c)) * scale[r] ) ),
// value = the correctly rounded fp32 quotient y / 147.800537109375.
//
// GB300 design: each warp walks (row, block) items with a grid stride; lane j
// owns the 8 adjacent positions 8j .. 8j+7, whose windows all lie in one
// 64-bit span that starts at bit (T-8(j+1))*k.  The lane loads the two words
// covering the span for the next item while it decodes the current one,
// aligns them once, takes its 8 windows with compile-time shifts, and writes
// its 16 output bytes with one 128-bit streaming store, so the warp's store
// covers the block's 512 output bytes contiguously.  The value y/d is
// computed as fma(y, r_hi, y*r_lo) (correctly rounded for every reachable y)
// in packed f32x2 arithmetic.  The kernel is bound by the HBM write of the
// 2-byte outputs (plus the k/8-byte code reads).
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace trellis {

namespace {
constexpr int kExpandThreads = 256;
}  // namespace

template <int K, int L>
__global__ void __launch_bounds__(kExpandThreads) expand_kernel(const uint32_t* __restrict__ codes,
                                                               const uint16_t* __restrict__ scales,
                                                               uint16_t* __restrict__ out, int64_t rows, int nb,
                                                               int interleave) {
  constexpr int WPB = kT * K / 32;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (kExpandThreads / 32);
  const int64_t items = rows * nb;
  int64_t it = (int64_t)blockIdx.x * (kExpandThreads / 32) + (threadIdx.x >> 5);

  const int lo = (kT - 8 * (lane + 1)) * K;  // first bit of the lane's span
  const int wa = lo >> 5, sh = lo & 31;
  const int wb = (wa + 1 == WPB) ? 0 : wa + 1;
  const float2 nmagic = make_float2(-kMagic, -kMagic);

  // block (row, blk) of item i: row-major, or the interleaved [nb/2][rows][2*WPB] layout
  auto block_of = [&](int64_t i) -> const uint32_t* {
    if (!interleave) return codes + i * WPB;
    const int64_t row = i / nb;
    const int blk = (int)(i - row * nb);
    return codes + ((int64_t)(blk >> 1) * rows + row) * (2 * WPB) + (blk & 1) * WPB;
  };
  uint32_t a = 0, b = 0;
  uint16_t sc16 = 0;
  if (it < items) {
    const uint32_t* bw = block_of(it);
    a = __ldg(bw + wa);
    b = __ldg(bw + wb);
    sc16 = __ldg(scales + it / nb);
  }
  for (; it < items; it += nwarps) {
    // prefetch the next item's words and scale
    const int64_t nx = it + nwarps;
    uint32_t na = 0, nbw = 0;
    uint16_t nsc = 0;
    if (nx < items) {
      const uint32_t* bw = block_of(nx);
      na = __ldg(bw + wa);
      nbw = __ldg(bw + wb);
      nsc = __ldg(scales + nx / nb);
    }
    uint32_t w[2];
    w[0] = __funnelshift_r(a, b, sh);
    w[1] = b >> sh;
    const float scale = f16_to_f32(sc16);
    const float2 sc = make_float2(scale, scale);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {  // positions 8*lane + i, 8*lane + i + 1
      const uint32_t s0 = window_at<L, 2>(w, (7 - i) * K);
      const uint32_t s1 = window_at<L, 2>(w, (6 - i) * K);
      const float2 y = __fadd2_rn(make_float2(__uint_as_float(code_magic(s0)), __uint_as_float(code_magic(s1))),
                                  nmagic);
      const float2 v = value_rn2(y);
      const float2 wv = __fmul2_rn(v, sc);
      o[i / 2] = pack_bf16x2(wv.x, wv.y);
    }
    __stcs(reinterpret_cast<uint4*>(out + it * kT) + lane, make_uint4(o[0], o[1], o[2], o[3]));
    a = na; b = nbw; sc16 = nsc;
  }
}

cudaError_t launch_expand_bf16(const uint32_t* codes, const uint16_t* scales, uint16_t* out, int k, int L,
                               int64_t rows, int64_t cols, int interleave, cudaStream_t st) {
  const int nb = (int)(cols / kT);
  const int64_t warps = rows * nb;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t nblk = (warps + 7) / 8;
  if (nblk > (int64_t)sms * 8) nblk = (int64_t)sms * 8;  // eight 256-thread CTAs per SM, grid-stride
  const dim3 block(kExpandThreads), grid((unsigned)nblk);
  if (L == 16) {
    if (k == 2) expand_kernel<2, 16><<<grid, block, 0, st>>>(codes, scales, out, rows, nb, interleave);
    else if (k == 3) expand_kernel<3, 16><<<grid, block, 0, st>>>(codes, scales, out, rows, nb, interleave);
    else expand_kernel<4, 16><<<grid, block, 0, st>>>(codes, scales, out, rows, nb, interleave);
  } else {
    if (k == 2) expand_kernel<2, 12><<<grid, block, 0, st>>>(codes, scales, out, rows, nb, interleave);
    else if (k == 3) expand_kernel<3, 12><<<grid, block, 0, st>>>(codes, scales, out, rows, nb, interleave);
    else expand_kernel<4, 12><<<grid, block, 0, st>>>(codes, scales, out, rows, nb, interleave);
  }
  return cudaGetLastError();
}

}  // namespace trellis
