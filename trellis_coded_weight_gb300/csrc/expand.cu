// expand.cu -- decode a whole stored trellis matrix to bf16, bit-exact.
//
// What is computed ("trellis-linear.ts" diff page: expandTrellis /
// EXPAND_SOURCE; "trellis-vector-expand.ts"):
//   out[r][c] = bf16( fl32( value(s(r,c)) * scale[r] ) ),
// value = the correctly rounded fp32 quotient y / 147.800537109375.
//
// GB300 design: the (row, block) items are cut into one contiguous range per
// warp, which the warp walks two items at a time, one per half-warp, keeping
// (row, block) by increments (no division in the loop).  Lane j of a half
// owns the 16 adjacent positions 16j .. 16j+15: it loads the two (even k) or
// three (k = 3) words that cover their windows for the next item while it
// decodes the current one, takes the windows with compile-time shifts (two
// 16-bit windows per funnel shift for L = 16 and even k), and writes its
// 32 output bytes with two 128-bit streaming stores, so a half-warp covers
// the block's 512 output bytes contiguously.  The value y/d is computed as
// fma(y, r_hi, y*r_lo) (correctly rounded for every reachable y) in packed
// f32x2 arithmetic.  The kernel is bound by the HBM write of the 2-byte
// outputs (plus the k/8-byte code reads).
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "devcache.h"
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
  constexpr bool kEven = (K % 2) == 0;
  constexpr int NR = (15 * K + L + (kEven ? 0 : 16) + 31) / 32;  // words of a lane's 16-position run
  const int lane = threadIdx.x & 31, half = lane >> 4, j = lane & 15;
  const int64_t nwarps = (int64_t)gridDim.x * (kExpandThreads / 32);
  const int64_t wid = (int64_t)blockIdx.x * (kExpandThreads / 32) + (threadIdx.x >> 5);
  const int64_t items = rows * nb;
  const int64_t i0 = wid * items / nwarps, i1 = (wid + 1) * items / nwarps;  // this warp's items

  // positions 16j .. 16j+15 of a block start at block bits (255-16j-i)*K, the lowest at lo
  const int lo = (kT - 16 * (j + 1)) * K;
  const int wa = lo >> 5, sh = lo & 31;
  int widx[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) widx[i] = (wa + i >= WPB) ? wa + i - WPB : wa + i;
  const float2 nmagic = make_float2(-kMagic, -kMagic);

  // item it = i0 + 2s + half is (row, blk); both advance by two items per step
  int64_t row = 0;
  int blk = 0;
  if (i0 + half < i1) {
    row = (i0 + half) / nb;
    blk = (int)(i0 + half - row * nb);
  }
  auto block_ptr = [&](int64_t r, int b) -> const uint32_t* {
    return interleave ? codes + ((int64_t)(b >> 1) * rows + r) * (2 * WPB) + (b & 1) * WPB
                      : codes + (r * nb + b) * WPB;
  };
  auto advance = [&](int64_t& r, int& b) {
    b += 2;
    if (b >= nb) { b -= nb; ++r; }
    if (b >= nb) { b -= nb; ++r; }  // nb == 1
  };
  uint32_t cur[NR], nxt[NR];
  uint16_t csc = 0, nsc = 0;
  bool have = i0 + half < i1;
  if (have) {
    const uint32_t* bw = block_ptr(row, blk);
#pragma unroll
    for (int q = 0; q < NR; ++q) cur[q] = __ldg(bw + widx[q]);
    csc = __ldg(scales + row);
  }
  for (int64_t it = i0 + half; __any_sync(0xffffffffu, it < i1); it += 2) {
    // prefetch the item two ahead of this half (the next step's)
    int64_t nrow = row;
    int nblk = blk;
    advance(nrow, nblk);
    const bool nhave = it + 2 < i1;
    if (nhave) {
      const uint32_t* bw = block_ptr(nrow, nblk);
#pragma unroll
      for (int q = 0; q < NR; ++q) nxt[q] = __ldg(bw + widx[q]);
      nsc = __ldg(scales + nrow);
    }
    if (have) {
      uint32_t w[NR];
      if constexpr (kEven) {
#pragma unroll
        for (int i = 0; i < NR; ++i) w[i] = cur[i];
      } else {
#pragma unroll
        for (int i = 0; i + 1 < NR; ++i) w[i] = __funnelshift_r(cur[i], cur[i + 1], sh);
        w[NR - 1] = cur[NR - 1] >> sh;
      }
      uint32_t s[16];
      run_states<K, L, 16, NR>(w, s);
      const float scale = f16_to_f32(csc);
      const float2 sc = make_float2(scale, scale);
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {  // positions 16j + i, 16j + i + 1
        // y by the float-bias subtraction on the FMA pipes or, for every second pair at k = 3 and 4, by the
        // int-to-float conversion on the ALU pipe (both exact): the split that measured fastest per k
        const float2 y = (K >= 3 && (i & 2) == 0)
                             ? code_y2_alu(s[i], s[i + 1])
                             : __fadd2_rn(make_float2(__uint_as_float(code_magic(s[i])), __uint_as_float(code_magic(s[i + 1]))),
                                          nmagic);
        const float2 v = value_rn2(y);
        const float2 wv = __fmul2_rn(v, sc);
        o[i / 2] = pack_bf16x2(wv.x, wv.y);
      }
      uint4* dst = reinterpret_cast<uint4*>(out + (row * nb + blk) * kT) + 2 * j;
      __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
      __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
    }
#pragma unroll
    for (int q = 0; q < NR; ++q) cur[q] = nxt[q];
    csc = nsc;
    row = nrow;
    blk = nblk;
    have = nhave;
  }
}

template <int K, int L>
static cudaError_t expand_launch(const uint32_t* codes, const uint16_t* scales, uint16_t* out, int64_t rows, int nb,
                                int interleave, cudaStream_t st) {
  // one wave: as many CTAs as fit on every SM at once, each warp one item range
  static PerDevice<int> per_sm_of;  // per instantiation and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const int per_sm = per_sm_of.get(dev, [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, expand_kernel<K, L>, kExpandThreads, 0) != cudaSuccess) {
      cudaGetLastError();
      n = 1;
    }
    return n < 1 ? 1 : n;
  }, 1);
  const int sms = device_sm_count();
  const int64_t items = rows * nb;
  int64_t nblk = (items + 2 * (kExpandThreads / 32) - 1) / (2 * (kExpandThreads / 32));  // >= two items per warp
  if (nblk > (int64_t)sms * per_sm) nblk = (int64_t)sms * per_sm;
  expand_kernel<K, L><<<(unsigned)nblk, kExpandThreads, 0, st>>>(codes, scales, out, rows, nb, interleave);
  return cudaGetLastError();
}

cudaError_t launch_expand_bf16(const uint32_t* codes, const uint16_t* scales, uint16_t* out, int k, int L,
                               int64_t rows, int64_t cols, int interleave, cudaStream_t st) {
  const int nb = (int)(cols / kT);
  if (L == 16) {
    if (k == 2) return expand_launch<2, 16>(codes, scales, out, rows, nb, interleave, st);
    if (k == 3) return expand_launch<3, 16>(codes, scales, out, rows, nb, interleave, st);
    return expand_launch<4, 16>(codes, scales, out, rows, nb, interleave, st);
  }
  if (k == 2) return expand_launch<2, 12>(codes, scales, out, rows, nb, interleave, st);
  if (k == 3) return expand_launch<3, 12>(codes, scales, out, rows, nb, interleave, st);
  return expand_launch<4, 12>(codes, scales, out, rows, nb, interleave, st);
}

}  // namespace trellis
