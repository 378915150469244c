// matvec_axis1_tc.cu -- decode-fused matvec over axis-1 trellis matrices, M = 1..4, and the fused gate/up
// SwiGLU layer, with the y*x accumulation on the tensor cores.
//
// What is computed ("trellis-linear.ts" diff page: REDUCE_SOURCE, GATEUP_SOURCE; "trellis-shared-m.ts": the
// shared-M variants):
//   out[m][r] = bf16( sum_c (y(r,c)/d * scale[r]) * x[m][c] )
// with the pages' default packed numerics (fp32 weight, no bf16 rounding), and for gate/up the bf16 cast chain
// gate -> up -> sigmoid -> silu -> product.  The per-row factor scale[r]/d multiplies the sum of y*x once.
//
// GB300 design.  The decode (window, 1MAD multiply, byte sum) runs on the CUDA cores and costs the same for every
// M; the y*x products go to the tensor cores through mma.sync m16n8k8 with tf32 operands, so M = 1..4 costs what
// M = 1 costs (the MMA has 8 token columns; absent tokens read zeros).  The operands are exact in tf32: y is an
// integer in [-510, 510] (11 significant bits), x is bf16 (8), so every product is exact and only the fp32
// accumulation rounds, as in the pages' fp32 sums.
//   * A warp owns 16 rows of a CTA's 64 and every fourth block of the row (a k-slice).  Lane (g, t) of the warp
//     decodes rows g and g+8 at positions [64t, 64t+64) of a block: 2K words per row loaded with 16-byte loads,
//     the spill word (the next lane's first word, or word 0 where the block wraps) taken by a shuffle.  Within a
//     block, MMA j uses k-slot t for position 64t+2j and k-slot t+4 for position 64t+2j+1, so the A fragment is
//     this lane's own decoded y values and the B fragment two adjacent x values.
//   * x is staged once per CTA in shared memory as fp32 (bf16 widened, exact), laid out so that the 8-byte B
//     fragment loads of the 4*M real lanes fall in distinct banks; lanes of absent tokens read a zero area.
//   * y comes from the byte sum (dp4a) and an int-to-float conversion (ALU pipe), which leaves the FMA pipes to
//     the 1MAD multiply and the byte sum; at K = 3 or L = 12, whose window extraction loads the ALU pipe more,
//     one row of the lane takes the float-bias subtraction (FMA pipe) instead.  With L = 16 and K in {2, 4} one funnel shift
//     yields the states of two positions 16 bits apart.
//   * M = 1 goes to the CUDA-core kernel (matvec_axis1.cu): with one token the packed FMA costs no more than
//     the MMA, and that kernel stages no x; measured at 17408 x 5120 it is as fast or faster for k = 2..4.
//   * Each block's MMAs accumulate into a fresh fragment that is added to the running fp32 sums, so no tensor-core
//     accumulation chain is longer than one block (32 MMAs).
//   * Two register sets of code words take turns: the loads of a warp's next block are in flight while it
//     decodes the current one; the first block's loads are issued before x is staged.
//   * The k-slices of a row fold through shared memory in a fixed order (deterministic), then scale/d, the cast
//     (or the SwiGLU chain) and the store.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "mma_tf32.cuh"
#include "pdl.cuh"

namespace trellis {
namespace {

constexpr int kRowGroups = 4;    // 16-row groups per CTA (64 rows)
constexpr int kTStride = 264;    // bytes per lane-quarter (64 fp32 positions) of one token's block, padded
constexpr int kTokStride = 1056; // bytes per token per block (4 quarters)
constexpr int kZeroBytes = 512;  // zero area for absent tokens: lanes read 32*M + 8j, j < 32

// A lane's 2K words of one block (positions [64t, 64t+64)) with 16-byte loads.  For K = 3 the 24 bytes start on
// an 8-byte boundary: two aligned 16-byte loads cover them and the lane keeps the right 6 words.
template <int K>
__device__ __forceinline__ void load_quarter(uint32_t (&w)[2 * K + 1], const uint32_t* blk, int t) {
  if constexpr (K == 3) {
    const uint4* p = reinterpret_cast<const uint4*>(blk) + (((3 - t) * 24) >> 4);
    const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const bool aligned = (t & 1) != 0;
#pragma unroll
    for (int i = 0; i < 6; ++i) w[i] = aligned ? u[i] : u[i + 2];
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(blk + (3 - t) * 2 * K);
#pragma unroll
    for (int i = 0; i < K / 2; ++i) {
      const uint4 v = __ldg(p + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

template <int M>
constexpr int seg_blocks_max(int ks) {  // blocks of x staged at once: at most ~84 KB of fp32 x
  return ((80 / M) / ks) * ks;
}

template <int K, int L, int M, bool GU>
struct TcCfg {
  static constexpr int NMAT = GU ? 2 : 1;
  static constexpr int KS = GU ? 2 : 4;  // k-slices per row group (gate/up: two matrices share the warps)
  static constexpr int Warps = kRowGroups * KS * NMAT;
  static constexpr int Threads = 32 * Warps;
  static constexpr int SBMax = seg_blocks_max<M>(KS);
  static constexpr size_t RedBytes = (size_t)NMAT * KS * kRowGroups * 16 * 4 * sizeof(float);
  static size_t smem(int sb) { return kZeroBytes + (size_t)sb * M * kTokStride + RedBytes; }
};

template <int K, int L, int M, bool GU>
__global__ void __launch_bounds__(TcCfg<K, L, M, GU>::Threads, 2)
    mvtc_kernel(const uint32_t* __restrict__ c0, const uint16_t* __restrict__ s0, const uint32_t* __restrict__ c1,
                const uint16_t* __restrict__ s1, const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                int64_t R, int64_t C, int SB) {
  using Cfg = TcCfg<K, L, M, GU>;
  constexpr int KS = Cfg::KS;
  constexpr int WPB = 8 * K;
  constexpr int NW = 2 * K + 1;
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int rg = warp % kRowGroups, ks = (warp / kRowGroups) % KS, mt = warp / (kRowGroups * KS);
  const int nb = (int)(C / kT);
  unsigned char* xs = smem + kZeroBytes;                                     // [SB][M][4][kTStride]
  float* red = reinterpret_cast<float*>(xs + (size_t)SB * M * kTokStride);  // [NMAT][KS][kRowGroups][16][4]
  if (threadIdx.x < kZeroBytes / 4) reinterpret_cast<uint32_t*>(smem)[threadIdx.x] = 0u;

  const int64_t rbase = (int64_t)blockIdx.x * (16 * kRowGroups) + rg * 16;
  const uint32_t* const cm = mt ? c1 : c0;
  const uint32_t* crow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t r = rbase + g + 8 * h;
    crow[h] = cm + (r < R ? r : R - 1) * (int64_t)nb * WPB;  // rows past the end load valid memory, store nothing
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int src = (lane & ~3) | ((t + 3) & 3);  // the lane whose first word is this lane's spill word

  uint32_t wA[2][NW], wB[2][NW];
  auto load_blk = [&](uint32_t (&w)[2][NW], int blk) {
#pragma unroll
    for (int h = 0; h < 2; ++h) load_quarter<K>(w[h], crow[h] + (int64_t)blk * WPB, t);
  };

  for (int seg0 = 0; seg0 < nb; seg0 += SB) {
    const int nseg = nb - seg0 < SB ? nb - seg0 : SB;
    if (ks < nseg) load_blk(wA, seg0 + ks);  // in flight while x is staged
    // x of blocks [seg0, seg0 + nseg) as fp32: 16-byte chunk c of a token holds positions 8c..8c+7, i.e. block
    // c/32, lane quarter (c%32)/8, byte offset 32*(c%8) in the quarter
    const int nch = nseg * 32;
    for (int i = threadIdx.x; i < M * nch; i += Cfg::Threads) {
      const int m = i / nch, c = i - m * nch;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)m * C + (int64_t)seg0 * kT) + c);
      const int b = c >> 5, cc = c & 31;
      uint2* dst = reinterpret_cast<uint2*>(xs + ((size_t)b * M + m) * kTokStride + (cc >> 3) * kTStride + (cc & 7) * 32);
      dst[0] = make_uint2(v.x << 16, v.x & 0xFFFF0000u);
      dst[1] = make_uint2(v.y << 16, v.y & 0xFFFF0000u);
      dst[2] = make_uint2(v.z << 16, v.z & 0xFFFF0000u);
      dst[3] = make_uint2(v.w << 16, v.w & 0xFFFF0000u);
    }
    __syncthreads();

    auto process = [&](uint32_t (&w)[2][NW], int b) {
#pragma unroll
      for (int h = 0; h < 2; ++h) w[h][2 * K] = __shfl_sync(0xFFFFFFFFu, w[h][0], src);
      const unsigned char* xb = g < M ? xs + (size_t)b * M * kTokStride + g * kTokStride + t * kTStride : smem + 32 * M;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      constexpr bool kPair = (L == 16) && (K == 2 || K == 4);
      constexpr int kPart = 16 / (2 * K);  // MMA distance of positions 16 bits apart (K = 2: 4, K = 4: 2)
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int ja = kPair ? ((jj / kPart) * 2 * kPart + (jj % kPart)) : 2 * jj;
        const int jb = kPair ? ja + kPart : ja + 1;
        const uint2 xa = *reinterpret_cast<const uint2*>(xb + 8 * ja);
        const uint2 xc = *reinterpret_cast<const uint2*>(xb + 8 * jb);
        uint32_t fa[2][2], fb[2][2];  // [row g / g+8][k-slot t / t+4]
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int qa = 2 * ja + i, qb = 2 * jb + i;  // lane-relative positions; q starts at bit (63-q)*K
            uint32_t sa, sb;
            if constexpr (kPair) {
              const int o = (63 - qb) * K;  // qb's window; qa's starts 16 bits higher
              const uint32_t F = (o & 31) ? __funnelshift_r(w[h][o >> 5], w[h][(o >> 5) + 1], o & 31) : w[h][o >> 5];
              sb = F & 0xFFFFu;
              sa = F >> 16;
            } else {
              sa = window_at<L, NW>(w[h], (63 - qa) * K);
              sb = window_at<L, NW>(w[h], (63 - qb) * K);
            }
            // y through the int-to-float conversion (ALU pipe); at K = 3 or L = 12, whose window extraction
            // takes more ALU work, row g+8 through the float-bias subtraction (FMA pipe) instead
            constexpr bool kAluBoth = K != 3 && L == 16;
            fa[h][i] = (h == 0 || kAluBoth) ? code_f32<true>(sa) : code_f32<false>(sa);
            fb[h][i] = (h == 0 || kAluBoth) ? code_f32<true>(sb) : code_f32<false>(sb);
          }
        mma_tf32(d, fa[0][0], fa[1][0], fa[0][1], fa[1][1], xa.x, xa.y);
        mma_tf32(d, fb[0][0], fb[1][0], fb[0][1], fb[1][1], xc.x, xc.y);
      }
      acc[0] += d[0]; acc[1] += d[1]; acc[2] += d[2]; acc[3] += d[3];
    };

    for (int b = ks; b < nseg; b += 2 * KS) {
      if (b + KS < nseg) load_blk(wB, seg0 + b + KS);
      process(wA, b);
      if (b + KS >= nseg) break;
      if (b + 2 * KS < nseg) load_blk(wA, seg0 + b + 2 * KS);
      process(wB, b + KS);
    }
    __syncthreads();  // the staged x is replaced by the next segment's
  }

  // fold: red[mt][ks][rg][row][token]; lanes t < 2 hold tokens 2t, 2t+1 (D fragment columns)
  if (t < 2) {
    float* r = red + (((mt * KS + ks) * kRowGroups + rg) * 16) * 4;
    r[g * 4 + 2 * t] = acc[0];
    r[g * 4 + 2 * t + 1] = acc[1];
    r[(g + 8) * 4 + 2 * t] = acc[2];
    r[(g + 8) * 4 + 2 * t + 1] = acc[3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kRowGroups * 16 * M; idx += Cfg::Threads) {
    const int m = idx % M, rr = (idx / M) % 16, rgi = idx / (16 * M);
    const int64_t row = (int64_t)blockIdx.x * (16 * kRowGroups) + rgi * 16 + rr;
    if (row >= R) continue;
    float v[Cfg::NMAT];
#pragma unroll
    for (int q = 0; q < Cfg::NMAT; ++q) {
      float a = 0.f;
#pragma unroll
      for (int k2 = 0; k2 < KS; ++k2) a += red[(((q * KS + k2) * kRowGroups + rgi) * 16 + rr) * 4 + m];
      v[q] = __fmul_rn(a, __fmul_rn(f16_to_f32((q ? s1 : s0)[row]), kRcpD));
    }
    uint16_t o;
    if constexpr (GU) o = swiglu_chain(v[0], v[Cfg::NMAT - 1]);
    else o = f32_to_bf16_rn(v[0]);
    out[(int64_t)m * R + row] = o;
  }
}

template <int K, int L, int M, bool GU>
cudaError_t tc_launch(const uint32_t* c0, const uint16_t* s0, const uint32_t* c1, const uint16_t* s1,
                      const uint16_t* x, uint16_t* out, int64_t R, int64_t C, cudaStream_t st) {
  using Cfg = TcCfg<K, L, M, GU>;
  auto kern = mvtc_kernel<K, L, M, GU>;
  static PerDevice<cudaError_t> attr_of;  // function attributes are per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const cudaError_t attr_err = attr_of.get(dev, [kern] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::smem(Cfg::SBMax));
  }, cudaErrorInvalidDevice);
  if (attr_err != cudaSuccess) return attr_err;
  const int nb = (int)(C / kT);
  const int SB = nb < Cfg::SBMax ? nb : Cfg::SBMax;
  const unsigned grid = (unsigned)((R + 16 * kRowGroups - 1) / (16 * kRowGroups));
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(Cfg::Threads), Cfg::smem(SB), st, c0, s0, c1, s1, x, out,
                                   R, C, SB);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int K, int L, bool GU>
cudaError_t tc_launch_m(int M, const uint32_t* c0, const uint16_t* s0, const uint32_t* c1, const uint16_t* s1,
                        const uint16_t* x, uint16_t* out, int64_t R, int64_t C, cudaStream_t st) {
  switch (M) {  // M = 1 takes the CUDA-core kernel
    case 2: return tc_launch<K, L, 2, GU>(c0, s0, c1, s1, x, out, R, C, st);
    case 3: return tc_launch<K, L, 3, GU>(c0, s0, c1, s1, x, out, R, C, st);
    case 4: return tc_launch<K, L, 4, GU>(c0, s0, c1, s1, x, out, R, C, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool GU>
cudaError_t tc_dispatch(const uint32_t* c0, const uint16_t* s0, const uint32_t* c1, const uint16_t* s1,
                        const uint16_t* x, uint16_t* out, int M, int k, int L, int64_t R, int64_t C, cudaStream_t st) {
  if (L == 16) {
    if (k == 2) return tc_launch_m<2, 16, GU>(M, c0, s0, c1, s1, x, out, R, C, st);
    if (k == 3) return tc_launch_m<3, 16, GU>(M, c0, s0, c1, s1, x, out, R, C, st);
    return tc_launch_m<4, 16, GU>(M, c0, s0, c1, s1, x, out, R, C, st);
  }
  if (k == 2) return tc_launch_m<2, 12, GU>(M, c0, s0, c1, s1, x, out, R, C, st);
  if (k == 3) return tc_launch_m<3, 12, GU>(M, c0, s0, c1, s1, x, out, R, C, st);
  return tc_launch_m<4, 12, GU>(M, c0, s0, c1, s1, x, out, R, C, st);
}

}  // namespace

cudaError_t launch_matvec_axis1(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                                int M, int k, int L, int64_t rows, int64_t cols, cudaStream_t st) {
  if (M == 1) return launch_matvec_axis1_fma(codes, scales, x, out, M, k, L, rows, cols, st);
  return tc_dispatch<false>(codes, scales, codes, scales, x, out, M, k, L, rows, cols, st);
}

cudaError_t launch_gateup_swiglu(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                                 const uint16_t* uscales, const uint16_t* x, uint16_t* out, int M, int k, int L,
                                 int64_t rows, int64_t cols, cudaStream_t st) {
  if (M == 1) return launch_gateup_swiglu_fma(gcodes, gscales, ucodes, uscales, x, out, M, k, L, rows, cols, st);
  return tc_dispatch<true>(gcodes, gscales, ucodes, uscales, x, out, M, k, L, rows, cols, st);
}

}  // namespace trellis
