// prefill_axis0_small.cu -- the axis-0 prefill GEMM (a stored W^T, the down projection) for small M (M <= 32):
//   out[m][c] = bf16( sum_r w(r,c) x[m][r] ),  w = bf16(fl32(value * scale[r])), the expand weight,
// accumulated in fp32 ("trellis-splitk-prefill.ts" diff page: the reduction over stored rows split across
// workers and the partials summed; "trellis-vector-expand.ts" for the weight).
//
// GB300 design.  At small M the tcgen05 axis-0 prefill decodes each weight into a shared-memory tile for a narrow
// MMA.  Here the decode stays in registers, with the lane layout of the tensor-core axis-0 matvec
// (matvec_axis0_tc.cu), and the products go through mma.sync m16n8k16 bf16:
//   * a thread-block cluster of S CTAs owns one 256-output column block; CTA r of the cluster takes the stored rows
//     [b_r, b_{r+1}) (multiples of 16), so the clusters' CTAs cover the GPU in one wave.  The partial sums of the
//     cluster's CTAs are folded through distributed shared memory in rank order: deterministic, no workspace.
//   * a CTA stages its rows through shared memory in pieces of kPaPiece rows, in a ring of three, all by 16-byte
//     cp.async: the code words of a piece, its x rows (bf16, token-major) and its fp16 scales.  One barrier per
//     piece.
//   * 16 warps: 4 column quarters (64 outputs, four MMA tiles of 16) x 4 row slices (every fourth 16-row k-step).
//     Lane (g, t) decodes stored rows 2t, 2t+1, 2t+8, 2t+9 of the k-step (the MMA's k-slots) at the 8 outputs
//     of its A rows (axis0_windows.cuh).  The weights of rows 2t and 2t+1 at one output are one packed bf16 pair,
//     an A register; the B register is x of rows 2t, 2t+1 of one token, a 32-bit load.
//   * the MMAs accumulate a warp's whole share in fp32 (as the tcgen05 kernel's tensor-memory accumulators do);
//     the row slices fold through shared memory in a fixed order, then the cluster.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "axis0_windows.cuh"
#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "pdl.cuh"
#include "tc_ptx.cuh"

namespace trellis {
namespace {

constexpr int kPaWarps = 16;
constexpr int kPaSlices = kPaWarps / 4;
constexpr int kPaThreads = 32 * kPaWarps;
constexpr int kPaPiece = 256;       // stored rows per staged piece (a multiple of 16 * kPaSlices)
constexpr int kPaBufs = 3;          // pieces in flight: decoded, landed, arriving
constexpr int kPaXStride = 264;     // bf16 per token row of a staged piece: 132 words = 4 mod 32

// Staged words per code row: lanes t = 0..3 read rows 2t (then 2t+1, ...) in one instruction, so 2 * stride must
// be 8 mod 32 for the four rows to fall 8 banks apart.
template <int K>
constexpr int pa_stride() { return K == 2 ? 20 : 36; }

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct PaParams {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* out;
  int64_t R, C;
  int M, nb, S;
};

template <int K, int NT>
constexpr size_t pa_ring_bytes() {
  return (size_t)kPaBufs * ((size_t)kPaPiece * pa_stride<K>() * 4 + (size_t)8 * NT * kPaXStride * 2 + kPaPiece * 2);
}

template <int K, int L, int NT>
__global__ void __launch_bounds__(kPaThreads, 1) pa_kernel(const PaParams p) {
  using Win = A0Windows<K, L>;
  constexpr int WPB = kT * K / 32;
  constexpr int CH = WPB / 4;  // 16-byte chunks of a row's block
  constexpr int ST = pa_stride<K>();
  constexpr int MP = 8 * NT;
  constexpr int kBufBytes = kPaPiece * ST * 4 + MP * kPaXStride * 2 + kPaPiece * 2;
  extern __shared__ __align__(16) unsigned char smem[];
  // ring buffer b: code rows [kPaPiece][ST] words, x rows [MP][kPaXStride] bf16, scales [kPaPiece] fp16
  auto codes_of = [&](int b) { return reinterpret_cast<uint32_t*>(smem + (size_t)b * kBufBytes); };
  auto x_of = [&](int b) { return reinterpret_cast<uint16_t*>(smem + (size_t)b * kBufBytes + kPaPiece * ST * 4); };
  auto sc_of = [&](int b) {
    return reinterpret_cast<uint16_t*>(smem + (size_t)b * kBufBytes + kPaPiece * ST * 4 + MP * kPaXStride * 2);
  };
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int Q = warp & 3, slice = warp >> 2;
  const Win win(Q, g);
  const int cb = blockIdx.x / p.S, rank = blockIdx.x - cb * p.S;
  // this CTA's stored rows: multiples of 16, the last range ending at R
  auto bound = [&](int r) { return r >= p.S ? p.R : ((int64_t)r * p.R / p.S) / 16 * 16; };
  const int64_t r_begin = bound(rank), r_end = bound(rank + 1);
  const int64_t rowWords = (int64_t)p.nb * WPB;
  const uint32_t* cblk = p.codes + (int64_t)cb * WPB;

  // tokens past M are zero in every buffer (never overwritten); rows past a piece are zeroed when it is issued
  for (int i = threadIdx.x; i < kPaBufs * (MP - p.M) * kPaXStride; i += kPaThreads) {
    const int b = i / ((MP - p.M) * kPaXStride), e = i - b * (MP - p.M) * kPaXStride;
    x_of(b)[p.M * kPaXStride + e] = 0;
  }

  // issue piece [r0, r0 + nr) into buffer b: 16-byte copies of code rows, x rows (rows are multiples of 8 and R is,
  // so every chunk is whole) and scales; the x rows and scales of the tail up to the next 16 rows are zeroed
  auto issue = [&](int64_t r0, int nr, int b) {
    uint32_t* cd = codes_of(b);
    for (int i = threadIdx.x; i < nr * CH; i += kPaThreads) {
      const int r = i / CH, ch = i - r * CH;
      cp16(cd + r * ST + 4 * ch, cblk + (r0 + r) * rowWords + 4 * ch);
    }
    uint16_t* xd = x_of(b);
    const int xch = (nr + 7) / 8;  // 16-byte chunks of a token's rows
    for (int i = threadIdx.x; i < p.M * xch; i += kPaThreads) {
      const int m = i / xch, c = i - m * xch;
      cp16(xd + m * kPaXStride + 8 * c, p.x + (int64_t)m * p.R + r0 + 8 * c);
    }
    const int nr16 = (nr + 15) & ~15;
    for (int i = threadIdx.x; i < p.M * (nr16 - 8 * xch); i += kPaThreads) {
      const int m = i / (nr16 - 8 * xch), e = i - m * (nr16 - 8 * xch);
      xd[m * kPaXStride + 8 * xch + e] = 0;
    }
    uint16_t* sd = sc_of(b);
    for (int c = threadIdx.x; c < xch; c += kPaThreads) cp16(sd + 8 * c, p.scales + r0 + 8 * c);
    // the scales of the tail rows are zeroed too: a stale or never-written value could be a NaN pattern, and a NaN
    // weight times a zero x row is still NaN
    for (int e = 8 * xch + threadIdx.x; e < nr16; e += kPaThreads) sd[e] = 0;
  };

  float acc[4][NT][4];
#pragma unroll
  for (int J = 0; J < 4; ++J)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[J][n][0] = acc[J][n][1] = acc[J][n][2] = acc[J][n][3] = 0.f;

  // the weights of rows ra (low half) and ra+1 (high half) at the output of state pair (sa, sb), packed bf16
  auto pair_w = [&](uint32_t sa, uint32_t sb, float2 sc) -> uint32_t {
    // y through the int-to-float conversion on the ALU pipe (exact), leaving the FMA pipes to the 1MAD
    // multiply, the byte sum and the value and scale products; at K = 2 with L = 12 windows the float-bias
    // subtraction on the FMA pipes measured faster
    constexpr bool kAlu = !(K == 2 && L == 12);
    const float2 y = kAlu ? code_y2_alu(sa, sb)
                          : __fadd2_rn(make_float2(__uint_as_float(code_magic(sa)), __uint_as_float(code_magic(sb))),
                                       make_float2(-kMagic, -kMagic));
    const float2 v = __fmul2_rn(value_rn2(y), sc);
    return pack_bf16x2(v.x, v.y);
  };

  const int npieces = (int)((r_end - r_begin + kPaPiece - 1) / kPaPiece);
  auto piece_nr = [&](int j) {
    const int64_t n = r_end - (r_begin + (int64_t)j * kPaPiece);
    return (int)(n < kPaPiece ? n : kPaPiece);
  };
  if (npieces > 0) issue(r_begin, piece_nr(0), 0);
  cp_commit();
  if (npieces > 1) issue(r_begin + kPaPiece, piece_nr(1), 1);
  cp_commit();
  for (int j = 0, b = 0; j < npieces; ++j, b = (b + 1 == kPaBufs) ? 0 : b + 1) {
    cp_wait<1>();  // this thread's copies of piece j have landed
    __syncthreads();           // ... and every thread's; piece j-1 is no longer read
    if (j + 2 < npieces) issue(r_begin + (int64_t)(j + 2) * kPaPiece, piece_nr(j + 2), (b + 2) % kPaBufs);
    cp_commit();

    const int nks = (piece_nr(j) + 15) >> 4;
    const uint32_t* cw = codes_of(b);
    const uint16_t* xs = x_of(b);
    const __half2* scp = reinterpret_cast<const __half2*>(sc_of(b));
    for (int ks = slice; ks < nks; ks += kPaSlices) {
      const int rb = 16 * ks + 2 * t;  // this lane's k-slot rows: rb, rb+1, rb+8, rb+9
      uint32_t s0[4][2], s1[4][2], s2[4][2], s3[4][2];
      win.states(cw + rb * ST, s0);
      win.states(cw + (rb + 1) * ST, s1);
      win.states(cw + (rb + 8) * ST, s2);
      win.states(cw + (rb + 9) * ST, s3);
      // rows past the piece: stale code words (finite y), zero scales and zero x rows
      const float2 scA = __half22float2(scp[rb >> 1]), scB = __half22float2(scp[(rb + 8) >> 1]);
#pragma unroll
      for (int J = 0; J < 4; ++J) {
        const uint32_t a0 = pair_w(s0[J][0], s1[J][0], scA), a1 = pair_w(s0[J][1], s1[J][1], scA);
        const uint32_t a2 = pair_w(s2[J][0], s3[J][0], scB), a3 = pair_w(s2[J][1], s3[J][1], scB);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint16_t* xr = xs + (8 * n + g) * kPaXStride + rb;
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xr), b1 = *reinterpret_cast<const uint32_t*>(xr + 8);
          mma_bf16(acc[J][n], a0, a1, a2, a3, b0, b1);
        }
      }
    }
  }
  cp_wait<0>();
  __syncthreads();  // the ring is free: it now holds the slices' sums, then the CTA's partial

  // red[slice][m][256]: lane (g, t) holds tokens 8n + 2t, 8n + 2t + 1 of outputs col(J, 0) (d0, d1) and
  // col(J, 1) (d2, d3)
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int J = 0; J < 4; ++J)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = 8 * n + 2 * t + e;
        if (m < p.M) {
          red[(slice * MP + m) * kT + win.col(J, 0)] = acc[J][n][e];
          red[(slice * MP + m) * kT + win.col(J, 1)] = acc[J][n][2 + e];
        }
      }
  __syncthreads();
  float* part = red + kPaSlices * MP * kT;  // [MP][256]: this CTA's partial, read by the cluster
  for (int i = threadIdx.x; i < p.M * kT; i += kPaThreads) {
    float s = red[i];
#pragma unroll
    for (int sl = 1; sl < kPaSlices; ++sl) s += red[sl * MP * kT + i];
    part[i] = s;
  }
  if (p.S > 1) tc::cluster_sync_all();  // every CTA's partial is complete and visible to the cluster
  else __syncthreads();
  // CTA `rank` folds outputs [rank*256/S, (rank+1)*256/S) of the column block over the cluster in rank order
  const int c0 = rank * kT / p.S, c1 = (rank + 1) * kT / p.S;
  for (int i = threadIdx.x; i < p.M * (c1 - c0); i += kPaThreads) {
    const int m = i / (c1 - c0), c = c0 + (i - m * (c1 - c0));
    float s = 0.f;
    for (int q = 0; q < p.S; ++q) s += q == rank ? part[m * kT + c] : tc::ld_dsmem_f32(part + m * kT + c, (uint32_t)q);
    p.out[(int64_t)m * p.C + (int64_t)cb * kT + c] = f32_to_bf16_rn(s);
  }
  if (p.S > 1) tc::cluster_sync_all();  // no CTA leaves while a peer may still read its partial
}

template <int K, int L, int NT>
cudaError_t pa_launch(const PaParams& p0, cudaStream_t st) {
  PaParams p = p0;
  auto kern = pa_kernel<K, L, NT>;
  constexpr size_t kRed = (size_t)(kPaSlices + 1) * 8 * NT * kT * sizeof(float);
  constexpr size_t smem = pa_ring_bytes<K, NT>() > kRed ? pa_ring_bytes<K, NT>() : kRed;
  struct Fit {
    int clusters[9];  // most co-resident clusters of S CTAs, S = 1..8
  };
  static PerDevice<Fit> fit_of;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const Fit fit = fit_of.get(dev, [kern] {
    Fit f{};
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess) {
      cudaGetLastError();
      return f;
    }
    for (int s = 1; s <= 8; ++s) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(s);
      cfg.blockDim = dim3(kPaThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = s; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      f.clusters[s] = n;
    }
    return f;
  }, Fit{});
  if (fit.clusters[1] < 1) return cudaErrorInvalidConfiguration;
  // the widest cluster with which every column block's cluster is resident at once (one wave), and at least
  // one k-step of 16 rows per CTA
  int S = 1;
  for (int s = 8; s >= 2; --s)
    if (fit.clusters[s] >= p.nb && (int64_t)s * 16 <= p.R) {
      S = s;
      break;
    }
  p.S = S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.nb * S));
  cfg.blockDim = dim3(kPaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = S; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int K, int L>
cudaError_t pa_launch_nt(const PaParams& p, cudaStream_t st) {
  switch ((p.M + 7) / 8) {  // 8-token tiles
    case 1: return pa_launch<K, L, 1>(p, st);
    case 2: return pa_launch<K, L, 2>(p, st);
    case 3: return pa_launch<K, L, 3>(p, st);
    default: return pa_launch<K, L, 4>(p, st);
  }
}

}  // namespace

cudaError_t launch_prefill_axis0_small(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                       uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                       cudaStream_t st) {
  if (M < 1 || M > kPrefillSmallMaxM0 || rows % 8 != 0) return cudaErrorInvalidValue;
  PaParams p{};
  p.codes = codes; p.scales = scales; p.x = x; p.out = out;
  p.R = rows; p.C = cols; p.M = M; p.nb = (int)(cols / kT); p.S = 1;
  if (L == 16) {
    if (k == 2) return pa_launch_nt<2, 16>(p, st);
    if (k == 3) return pa_launch_nt<3, 16>(p, st);
    return pa_launch_nt<4, 16>(p, st);
  }
  if (k == 2) return pa_launch_nt<2, 12>(p, st);
  if (k == 3) return pa_launch_nt<3, 12>(p, st);
  return pa_launch_nt<4, 12>(p, st);
}

}  // namespace trellis
