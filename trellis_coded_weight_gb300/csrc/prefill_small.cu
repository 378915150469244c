// prefill_small.cu -- the axis-1 prefill GEMM for small M (M <= 24): out[m][r] = bf16( sum_c w(r,c) x[m][c] )
// with the prefill's weight numerics w = bf16(fl32(value * scale[r])), the expand weight ("trellis-tiled-prefill.ts"
// diff page: decode into the tile, then the matrix product; "trellis-vector-expand.ts" for the weight).
//
// GB300 design.  At small M the tcgen05 prefill spends its time writing every decoded weight through shared memory
// for a narrow MMA, on 136 row tiles of 128 rows (16 of 152 SMs idle).  Here the decode stays in registers, as in
// the tensor-core matvec (matvec_axis1_tc.cu), and the products go through mma.sync m16n8k16 bf16 with one 8-token
// tile per 8 tokens (the kernel takes up to four; the launcher routes M <= 24 here, below its measured crossover
// with the tcgen05 kernel between 24 and 28 tokens):
//   * a CTA owns 64 rows (four 16-row groups) and the row's blocks split over KS warps per group; lane (g, t)
//     decodes rows g and g+8 of its group at positions [64t, 64t+64) of a block from 2K words (16-byte loads) and
//     the spill word of the neighbouring lane (a shuffle).
//   * MMA j of a block takes, per row, two pairs of the lane's positions: k-slots 2t, 2t+1 and 2t+8, 2t+9.  A pair
//     is two positions whose windows are 16 bits apart (8 positions for k = 2, 4 for k = 4), so one funnel shift
//     yields both states; for k = 3 (or L = 12) a pair is two neighbouring positions.  The pair's two weights are
//     rounded to bf16 and packed by one conversion: that register is the A fragment.
//   * x is staged in shared memory as bf16 in the same permuted order, so the B fragment of a token tile is one
//     8-byte load; the strides put the 16 lanes of a half warp on distinct bank pairs.  Tokens past M are staged
//     as zeros.
//   * the MMAs accumulate a warp's whole share of the row in fp32 (as the tensor-memory accumulators of the tcgen05
//     path do); the k-slices fold through shared memory in a fixed order.
//   * measured at 17408 x 5120, k = 2 (this kernel / the tcgen05 kernel, us): M = 8 33.9 / 48.7, M = 16 40.3 /
//     48.7, M = 24 48.5 / 48.8, M = 32 53.0 / 48.7.  Each 8-token tile adds ~6.5 us, about 23 cycles per mma.sync
//     m16n8k16 per scheduler, so above 16 tokens the tcgen05 kernel takes over.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "pdl.cuh"

namespace trellis {
namespace {

constexpr int kPsRowGroups = 4;  // 16-row groups per CTA (64 rows)
constexpr int kPsKS = 2;         // warps per row group (k-slices of the row's blocks)
constexpr int kPsThreads = 32 * kPsRowGroups * kPsKS;
constexpr int kPsQStride = 34;   // words per lane quarter of one token's staged block (32 + 2)
constexpr int kPsTStride = 136;  // words per token per staged block (4 quarters; = 8 mod 32)

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Pairs of a lane's 64 positions (q, q + D): base q takes the high half of a packed register, q + D the low half.
template <int K, int L>
struct PsPairs {
  static constexpr int D = (L == 16 && K == 2) ? 8 : (L == 16 && K == 4) ? 4 : 1;
  // base position of pair i (0..31): the i-th q in increasing order with (q mod 2D) < D
  static __host__ __device__ constexpr int base(int i) { return (i / D) * 2 * D + (i % D); }
  // pair index of a base position
  static __host__ __device__ constexpr int index(int q) { return (q / (2 * D)) * D + (q % (2 * D)); }
};

template <int K, int L, int NT>
__global__ void __launch_bounds__(kPsThreads, 2)
    pfs_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
               const uint16_t* __restrict__ x, uint16_t* __restrict__ out, int64_t R, int64_t C, int M, int SB) {
  using PP = PsPairs<K, L>;
  constexpr int WPB = 8 * K;
  constexpr int NW = 2 * K + 1;
  constexpr int MP = 8 * NT;  // staged tokens (a multiple of 8)
  extern __shared__ __align__(16) uint32_t xs[];                              // [SB][MP][4][kPsQStride] words
  float* red = reinterpret_cast<float*>(xs + (size_t)SB * MP * kPsTStride);  // [KS][rg][16][MP]
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int rg = warp % kPsRowGroups, ks = warp / kPsRowGroups;
  const int nb = (int)(C / kT);

  const int64_t rbase = (int64_t)blockIdx.x * (16 * kPsRowGroups) + rg * 16;
  const uint32_t* crow[2];
  float sc[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t r = rbase + g + 8 * h;
    const int64_t rc = r < R ? r : R - 1;  // rows past the end load valid memory and store nothing
    crow[h] = codes + rc * (int64_t)nb * WPB;
    sc[h] = f16_to_f32(__ldg(scales + rc));
  }
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  const int src = (lane & ~3) | ((t + 3) & 3);  // the lane whose first word is this lane's spill word

  uint32_t wA[2][NW], wB[2][NW];
  auto load_blk = [&](uint32_t (&w)[2][NW], int blk) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t* bp = crow[h] + (int64_t)blk * WPB;
      if constexpr (K == 3) {  // the lane's 24 bytes start on an 8-byte boundary: two aligned 16-byte loads
        const uint4* p = reinterpret_cast<const uint4*>(bp) + (((3 - t) * 24) >> 4);
        const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
        const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        const bool aligned = (t & 1) != 0;
#pragma unroll
        for (int i = 0; i < 6; ++i) w[h][i] = aligned ? u[i] : u[i + 2];
      } else {
        const uint4* p = reinterpret_cast<const uint4*>(bp + (3 - t) * 2 * K);
#pragma unroll
        for (int i = 0; i < K / 2; ++i) {
          const uint4 v = __ldg(p + i);
          w[h][4 * i] = v.x; w[h][4 * i + 1] = v.y; w[h][4 * i + 2] = v.z; w[h][4 * i + 3] = v.w;
        }
      }
    }
  };

  // The packed bf16 weights of pair i of row h: high half the weight of position base(i), low half of base(i)+D.
  auto pair_weights = [&](const uint32_t (&w)[NW], float s, int i) -> uint32_t {
    const int qh = PP::base(i), ql = qh + PP::D;  // lane-relative positions; q's window starts at bit (63-q)*K
    uint32_t sh, sl;
    if constexpr (PP::D > 1) {  // the two windows are 16 bits apart: one funnel shift
      const int o = (63 - ql) * K;
      const uint32_t F = (o & 31) ? __funnelshift_r(w[o >> 5], w[(o >> 5) + 1], o & 31) : w[o >> 5];
      sl = F & 0xFFFFu;
      sh = F >> 16;
    } else {
      sh = window_at<L, NW>(w, (63 - qh) * K);
      sl = window_at<L, NW>(w, (63 - ql) * K);
    }
    // y through the int-to-float conversion on the ALU pipe (exact), leaving the FMA pipes to the 1MAD
    // multiply, the byte sum and the value and scale products
    const float2 y = code_y2_alu(sl, sh);
    const float2 v = __fmul2_rn(value_rn2(y), make_float2(s, s));
    return pack_bf16x2(v.x, v.y);  // low half: position ql
  };

  for (int seg0 = 0; seg0 < nb; seg0 += SB) {
    const int nseg = nb - seg0 < SB ? nb - seg0 : SB;
    if (ks < nseg) load_blk(wA, seg0 + ks);  // in flight while x is staged
    // x of blocks [seg0, seg0 + nseg): a thread takes runs of 16 consecutive positions of one token (32 bytes),
    // i.e. the 8 pairs (q, q + D) whose base q lies in the run, and stores each pair as one word at
    // [block][token][quarter][2 * (pair / 2) + pair % 2]
    const int nruns = nseg * 16;  // runs of 16 positions per token
    constexpr int kRunsInFlight = 4;  // a thread's runs whose loads are issued before any of them is stored
    for (int i0 = threadIdx.x; i0 < MP * nruns; i0 += kRunsInFlight * kPsThreads) {
      uint32_t e[kRunsInFlight][8];
#pragma unroll
      for (int r = 0; r < kRunsInFlight; ++r) {
        const int i = i0 + r * kPsThreads;
        const int m = i / nruns, u = i - m * nruns;
        if (i < MP * nruns && m < M) {
          const int bb = u >> 4, qt = (u >> 2) & 3, q0 = (u & 3) * 16;  // block, quarter, first lane position
          const uint4* sp =
              reinterpret_cast<const uint4*>(x + (int64_t)m * C + (int64_t)(seg0 + bb) * kT + qt * 64 + q0);
          const uint4 v0 = __ldg(sp), v1 = __ldg(sp + 1);
          e[r][0] = v0.x; e[r][1] = v0.y; e[r][2] = v0.z; e[r][3] = v0.w;
          e[r][4] = v1.x; e[r][5] = v1.y; e[r][6] = v1.z; e[r][7] = v1.w;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) e[r][q] = 0u;  // tokens past M stage zeros
        }
      }
#pragma unroll
      for (int r = 0; r < kRunsInFlight; ++r) {
        const int i = i0 + r * kPsThreads;
        if (i >= MP * nruns) break;
        const int m = i / nruns, u = i - m * nruns;
        const int bb = u >> 4, qt = (u >> 2) & 3, q0 = (u & 3) * 16;
        uint32_t* dst = xs + ((size_t)bb * MP + m) * kPsTStride + qt * kPsQStride;
        // q0 is a multiple of 16 and 2D divides 16, so which run positions are pair bases, and where each pair
        // goes (pair index q0/2 + index(q)), are known at compile time
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (q % (2 * PP::D) < PP::D) {
            const int pi = q0 / 2 + PP::index(q);
            const uint32_t lo = (e[r][(q + PP::D) >> 1] >> (16 * ((q + PP::D) & 1))) & 0xFFFFu;
            const uint32_t hi = (e[r][q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
            dst[2 * (pi >> 1) + (pi & 1)] = lo | (hi << 16);
          }
        }
      }
    }
    __syncthreads();

    auto process = [&](uint32_t (&w)[2][NW], int b) {
#pragma unroll
      for (int h = 0; h < 2; ++h) w[h][2 * K] = __shfl_sync(0xFFFFFFFFu, w[h][0], src);
      const uint32_t* xb = xs + (size_t)b * MP * kPsTStride + g * kPsTStride + t * kPsQStride;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        // A: rows g (h = 0) and g+8 (h = 1); k-slots 2t, 2t+1 = pair 2j, k-slots 2t+8, 2t+9 = pair 2j+1
        const uint32_t a0 = pair_weights(w[0], sc[0], 2 * j), a1 = pair_weights(w[1], sc[1], 2 * j);
        const uint32_t a2 = pair_weights(w[0], sc[0], 2 * j + 1), a3 = pair_weights(w[1], sc[1], 2 * j + 1);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint2 bv = *reinterpret_cast<const uint2*>(xb + (size_t)n * 8 * kPsTStride + 2 * j);
          mma_bf16(acc[n], a0, a1, a2, a3, bv.x, bv.y);
        }
      }
    };

    for (int b = ks; b < nseg; b += 2 * kPsKS) {
      if (b + kPsKS < nseg) load_blk(wB, seg0 + b + kPsKS);
      process(wA, b);
      if (b + kPsKS >= nseg) break;
      if (b + 2 * kPsKS < nseg) load_blk(wA, seg0 + b + 2 * kPsKS);
      process(wB, b + kPsKS);
    }
    __syncthreads();  // the staged x is replaced by the next segment's
  }

  // fold: red[ks][rg][row][token]; lane (g, t) holds tokens 8n + 2t, 8n + 2t + 1 of rows g and g+8
  {
    float* r = red + ((ks * kPsRowGroups + rg) * 16) * MP;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      r[g * MP + 8 * n + 2 * t] = acc[n][0];
      r[g * MP + 8 * n + 2 * t + 1] = acc[n][1];
      r[(g + 8) * MP + 8 * n + 2 * t] = acc[n][2];
      r[(g + 8) * MP + 8 * n + 2 * t + 1] = acc[n][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kPsRowGroups * 16 * M; idx += kPsThreads) {
    const int m = idx % M, rr = (idx / M) % 16, rgi = idx / (16 * M);
    const int64_t row = (int64_t)blockIdx.x * (16 * kPsRowGroups) + rgi * 16 + rr;
    if (row >= R) continue;
    float a = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < kPsKS; ++k2) a += red[((k2 * kPsRowGroups + rgi) * 16 + rr) * MP + m];
    out[(int64_t)m * R + row] = f32_to_bf16_rn(a);
  }
}

template <int K, int L, int NT>
size_t pfs_smem(int SB) {
  return (size_t)SB * 8 * NT * kPsTStride * sizeof(uint32_t) +
         (size_t)kPsKS * kPsRowGroups * 16 * 8 * NT * sizeof(float);
}

template <int K, int L, int NT>
cudaError_t pfs_launch(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                       int64_t R, int64_t C, cudaStream_t st) {
  constexpr size_t kBudget = 100 * 1024;  // two CTAs per SM
  const int nb = (int)(C / kT);
  int SB = (int)((kBudget - pfs_smem<K, L, NT>(0)) / ((size_t)8 * NT * kPsTStride * sizeof(uint32_t)));
  SB = (SB / kPsKS) * kPsKS;
  if (SB < kPsKS) SB = kPsKS;
  if (SB > nb) SB = nb;
  const int segs = (nb + SB - 1) / SB;  // segments of equal length (a multiple of KS where possible)
  const int even = ((nb + segs - 1) / segs + kPsKS - 1) / kPsKS * kPsKS;
  if (even < SB) SB = even;
  auto kern = pfs_kernel<K, L, NT>;
  static PerDevice<cudaError_t> attr_of;  // function attributes are per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const cudaError_t attr_err = attr_of.get(dev, [kern] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBudget);
  }, cudaErrorInvalidDevice);
  if (attr_err != cudaSuccess) return attr_err;
  const unsigned grid = (unsigned)((R + 16 * kPsRowGroups - 1) / (16 * kPsRowGroups));
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kPsThreads), pfs_smem<K, L, NT>(SB), st, codes, scales, x,
                                   out, R, C, M, SB);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int K, int L>
cudaError_t pfs_launch_nt(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                          int64_t R, int64_t C, cudaStream_t st) {
  switch ((M + 7) / 8) {
    case 1: return pfs_launch<K, L, 1>(codes, scales, x, out, M, R, C, st);
    case 2: return pfs_launch<K, L, 2>(codes, scales, x, out, M, R, C, st);
    case 3: return pfs_launch<K, L, 3>(codes, scales, x, out, M, R, C, st);
    default: return pfs_launch<K, L, 4>(codes, scales, x, out, M, R, C, st);
  }
}

}  // namespace

cudaError_t launch_prefill_small(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                                 int k, int L, int64_t rows, int64_t cols, cudaStream_t st) {
  if (M < 1 || M > kPrefillSmallMaxM1) return cudaErrorInvalidValue;
  if (L == 16) {
    if (k == 2) return pfs_launch_nt<2, 16>(codes, scales, x, out, M, rows, cols, st);
    if (k == 3) return pfs_launch_nt<3, 16>(codes, scales, x, out, M, rows, cols, st);
    return pfs_launch_nt<4, 16>(codes, scales, x, out, M, rows, cols, st);
  }
  if (k == 2) return pfs_launch_nt<2, 12>(codes, scales, x, out, M, rows, cols, st);
  if (k == 3) return pfs_launch_nt<3, 12>(codes, scales, x, out, M, rows, cols, st);
  return pfs_launch_nt<4, 12>(codes, scales, x, out, M, rows, cols, st);
}

}  // namespace trellis
