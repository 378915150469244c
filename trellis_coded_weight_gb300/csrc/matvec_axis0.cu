// matvec_axis0.cu -- decode-fused matvec over an axis-0 trellis matrix (a
// stored W^T coded along the output dimension), M = 1..4.
//
// What is computed ("trellis-linear.ts" diff page: SCATTER_SOURCE and the
// partial fold of the scatter path; "trellis-balanced-scatter.ts"):
//   out[m][c] = bf16( sum_r (y(r,c)/d * scale[r]) * x[m][r] )
// The pages split the sum over stored rows into 128 slices, write every
// slice's partial vector and fold them with a separate reduction.
//
// GB300 design (a balanced, persistent split over the stored rows):
//   * the work is the list of (column block, stored row) pairs, column block
//     major; CTA c of G (one per SM) takes the contiguous range
//     [c*N/G, (c+1)*N/G) of it, so every SM decodes the same number of rows.
//     A range crosses at most a few column blocks; each piece is a segment.
//   * a warp takes two stored rows at a time, one per half-warp; lane j of a
//     half owns outputs 16j .. 16j+15 of the column block: per row it loads
//     the two or three words that cover its 16 windows (already word-aligned
//     for even k) and takes the windows with compile-time shifts, two 16-bit
//     windows per funnel shift when L = 16 and k is even.  The CTA's warps
//     take interleaved row pairs; the code words of the next group of rows
//     load while the current group decodes.
//   * x[m][r]*scale[r] of the segment's rows is staged in shared memory (in
//     pieces of at most kAx0StageRows rows) and read with a broadcast load per
//     row; 1/d is applied after the sum.
//   * at the end of a segment the CTA folds its warps in shared memory and
//     writes one fp32 partial per output to the workspace; the partials are
//     folded deterministically in one launch (axis0_split.cuh).
#include <cstdint>
#include <cuda_runtime.h>

#include "axis0_split.cuh"
#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "pdl.cuh"

namespace trellis {

constexpr int kAx0Chunk = 4;             // rows per lane per prefetch group
constexpr int64_t kAx0StageRows = 2048;  // rows of x*scale staged at once

// Warps per CTA: as many as the accumulators' registers allow with one CTA per SM.
template <int M>
__host__ __device__ constexpr int ax0_warps() { return M <= 2 ? 16 : 12; }

size_t axis0_workspace_bytes(int M, int64_t rows, int64_t cols) {
  (void)rows;
  const int64_t nb = cols / kT;
  const size_t part = (size_t)(kAx0MaxCtas + nb) * (size_t)M * kT * sizeof(float);
  return part + (((size_t)nb * sizeof(uint32_t) + 15) & ~(size_t)15);
}

template <int K, int L, int M, bool BW, bool IL>
__global__ void __launch_bounds__(32 * ax0_warps<M>(), 1) ax0_kernel(const Ax0Params p) {
  constexpr int W = ax0_warps<M>();
  constexpr int WPB = kT * K / 32;
  // Words of one lane's 16-position run: 15K + L bits, plus up to 16 bits of
  // misalignment when K is odd.
  constexpr bool kEven = (K % 2) == 0;
  constexpr int NR = (15 * K + L + (kEven ? 0 : 16) + 31) / 32;
  constexpr int G = kAx0Chunk;
  constexpr int RS = 2 * W;  // rows per CTA step
  extern __shared__ __align__(16) float smem[];
  pdl_enter();
  float* xs = smem;                                       // [stage][M]  x*scale of the staged rows
  float* red = smem + ((p.stage * M + 3) & ~3);           // [W][M][256], 16-byte aligned
  float* scs = red + W * M * kT;                          // [stage] row scales (bf16-weight numerics)
  __shared__ int pend[kAx0MaxPending];          // column blocks whose arrival is pending
  __shared__ uint32_t is_last[kAx0MaxPending];
  int npend = 0;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, j = lane & 15;
  const int rb = 2 * warp + half;  // this lane's first row of every staged piece
  // Half-warp `half` takes the odd or even row of each row pair; lane j of
  // the half owns block positions 16j .. 16j+15, whose windows start at
  // block bits (255-16j-i)*K, the lowest at lo = (240-16j)*K.
  const int lo = (kT - 16 * (j + 1)) * K;
  const int wa = lo >> 5, sh = lo & 31;
  const int64_t rowWords = IL ? 2 * WPB : (int64_t)p.nb * WPB;
  const float2 nmagic = make_float2(-kMagic, -kMagic);

  const int c = blockIdx.x;
  const int64_t f1 = (int64_t)(c + 1) * p.N / p.G;
  for (int64_t f = (int64_t)c * p.N / p.G; f < f1;) {
    const int cb = (int)(f / p.R);
    const int64_t sa = f - (int64_t)cb * p.R;
    const int64_t se = (f1 - (int64_t)cb * p.R < p.R) ? f1 - (int64_t)cb * p.R : p.R;
    f = (int64_t)cb * p.R + se;
    // first word of column block cb in either layout
    const uint32_t* base = IL ? p.codes + (int64_t)(cb >> 1) * p.R * (2 * WPB) + (cb & 1) * WPB
                              : p.codes + (int64_t)cb * WPB;

    float2 acc[M][8];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[m][i] = make_float2(0.f, 0.f);

    for (int64_t r0 = sa; r0 < se; r0 += p.stage) {
      const int nr = (int)((se - r0 < p.stage) ? se - r0 : p.stage);
      // This lane's rows of the piece are rb, rb + RS, ... in groups of G;
      // full groups run unguarded, a short last group repeats the lane's
      // first row for its missing rows and skips them.
      const int n = nr > rb ? (nr - rb + RS - 1) / RS : 0;
      const int nfull = n / G, tail = n - nfull * G;
      const uint32_t* wp[NR];  // this lane's words of row r0 + rb
#pragma unroll
      for (int i = 0; i < NR; ++i) wp[i] = base + (r0 + rb) * rowWords + ((wa + i >= WPB) ? wa + i - WPB : wa + i);
      const int64_t rstep = (int64_t)RS * rowWords;  // words between this lane's consecutive rows
      auto load_full = [&](uint32_t (&a)[G][NR], int64_t off) {
#pragma unroll
        for (int u = 0; u < G; ++u)
#pragma unroll
          for (int q = 0; q < NR; ++q) a[u][q] = __ldg(wp[q] + off + u * rstep);
      };
      auto load_tail = [&](uint32_t (&a)[G][NR], int64_t off) {
#pragma unroll
        for (int u = 0; u < G; ++u) {
          const int64_t o = u < tail ? off + u * rstep : 0;
#pragma unroll
          for (int q = 0; q < NR; ++q) a[u][q] = __ldg(wp[q] + o);
        }
      };
      uint32_t A[G][NR], B[G][NR];
      if (nfull > 0) load_full(A, 0);
      else if (tail > 0) load_tail(A, 0);

      // stage x*scale (or x and the scales) of the piece, four rows per thread in flight
      for (int rr = threadIdx.x; rr < nr; rr += 4 * blockDim.x) {
        float sv[4], xv[4][M];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rl = rr + u * (int)blockDim.x;
          const int64_t r = r0 + (rl < nr ? rl : 0);
          sv[u] = f16_to_f32(__ldg(p.scales + r));
#pragma unroll
          for (int m = 0; m < M; ++m) xv[u][m] = bf16_to_f32(__ldg(p.x + (int64_t)m * p.R + r));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rl = rr + u * (int)blockDim.x;
          if (rl < nr) {
            // default numerics fold the row scale into x; bf16 weights need it per weight
#pragma unroll
            for (int m = 0; m < M; ++m) xs[rl * M + m] = BW ? xv[u][m] : __fmul_rn(xv[u][m], sv[u]);
            if (BW) scs[rl] = sv[u];
          }
        }
      }
      __syncthreads();

    // one row: raw words, x of the row at xr[0..M), its scale at sc
    auto body = [&](const uint32_t (&raw)[NR], const float* xr, const float* sc) {
      uint32_t w[NR];
      if constexpr (kEven) {
#pragma unroll
        for (int i = 0; i < NR; ++i) w[i] = raw[i];
      } else {
#pragma unroll
        for (int i = 0; i + 1 < NR; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
        w[NR - 1] = raw[NR - 1] >> sh;
      }
      uint32_t s[16];
      run_states<K, L, 16, NR>(w, s);
      float xv[M];
      if constexpr (M == 4) {
        const float4 v = *reinterpret_cast<const float4*>(xr);
        xv[0] = v.x; xv[1] = v.y; xv[2] = v.z; xv[3] = v.w;
      } else {
#pragma unroll
        for (int m = 0; m < M; ++m) xv[m] = xr[m];
      }
      float sr = 0.f;
      if constexpr (BW) sr = *sc;
#pragma unroll
      for (int i2 = 0; i2 < 8; ++i2) {
        // y by an int-to-float conversion on the ALU pipe or by the float-bias subtraction on the FMA pipes (both
        // exact): the ALU form for every pair at K = 2 (L = 16) and three pairs in four at K = 4, where the window
        // extraction leaves the ALU pipe room; at K = 3 (and K = 2, L = 12) the window extraction fills the ALU
        // pipe and the FMA form stays
        constexpr bool kAluAll = K == 2 && L == 16, kAluMost = K == 4;
        const bool alu = kAluAll || (kAluMost && (i2 & 3) != 3);
        float2 y = alu ? code_y2_alu(s[2 * i2], s[2 * i2 + 1])
                       : __fadd2_rn(make_float2(__uint_as_float(code_magic(s[2 * i2])),
                                                __uint_as_float(code_magic(s[2 * i2 + 1]))),
                                    nmagic);
        if constexpr (BW) {  // bf16(value * scale), the expand weight
          const float2 wv = __fmul2_rn(value_rn2(y), make_float2(sr, sr));
          const uint32_t bb = pack_bf16x2(wv.x, wv.y);
          y = make_float2(bf16lo_to_f32(bb), bf16hi_to_f32(bb));
        }
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m][i2] = __ffma2_rn(y, make_float2(xv[m], xv[m]), acc[m][i2]);
      }
    };
      // group g covers this lane's rows g*G .. g*G+G-1
      auto run_full = [&](const uint32_t (&a)[G][NR], int g) {
        const float* xg = xs + (rb + g * G * RS) * M;
        const float* sg = scs + rb + g * G * RS;
#pragma unroll
        for (int u = 0; u < G; ++u) body(a[u], xg + u * RS * M, sg + u * RS);
      };
      auto run_tail = [&](const uint32_t (&a)[G][NR], int g) {
        const float* xg = xs + (rb + g * G * RS) * M;
        const float* sg = scs + rb + g * G * RS;
#pragma unroll
        for (int u = 0; u < G; ++u)
          if (u < tail) body(a[u], xg + u * RS * M, sg + u * RS);
      };
      // A holds group g at the top of each iteration
      int g = 0;
      for (; g + 1 < nfull; g += 2) {
        load_full(B, (int64_t)(g + 1) * G * rstep);
        run_full(A, g);
        if (g + 2 < nfull) load_full(A, (int64_t)(g + 2) * G * rstep);
        else if (g + 2 == nfull && tail > 0) load_tail(A, (int64_t)(g + 2) * G * rstep);
        run_full(B, g + 1);
      }
      if (g < nfull) {  // one full group left, then perhaps the tail
        if (tail > 0) load_tail(B, (int64_t)(g + 1) * G * rstep);
        run_full(A, g);
        if (tail > 0) run_tail(B, g + 1);
      } else if (tail > 0) {
        run_tail(A, g);
      }
      __syncthreads();  // the staged piece is no longer read
    }

    // fold the two halves of each warp, then the warps of this CTA
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[m][i].x += __shfl_xor_sync(0xFFFFFFFFu, acc[m][i].x, 16);
        acc[m][i].y += __shfl_xor_sync(0xFFFFFFFFu, acc[m][i].y, 16);
      }
    if (half == 0) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float4* dst = reinterpret_cast<float4*>(red + (warp * M + m) * kT + 16 * j);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_float4(acc[m][2 * q].x, acc[m][2 * q].y, acc[m][2 * q + 1].x, acc[m][2 * q + 1].y);
      }
    }
    __syncthreads();
    // red[w][m][t] holds block position t (output column cb*256 + t)
    float* slot = p.part + (int64_t)(c + cb) * M * kT;
    for (int i = threadIdx.x; i < M * kT; i += blockDim.x) {
      float v = red[i];
#pragma unroll
      for (int w = 1; w < W; ++w) v += red[w * M * kT + i];
      slot[i] = v;
    }
    ax0_publish<M, BW>(p, pend, is_last, npend, cb, f >= f1);
  }
}

template <int K, int L, int M, bool BW, bool IL>
static cudaError_t ax0_launch1(const Ax0Params& p, cudaStream_t st) {
  constexpr int W = ax0_warps<M>();
  const size_t smem = ((((size_t)p.stage * M + 3) & ~(size_t)3) + (size_t)W * M * kT + (BW ? (size_t)p.stage : 0)) *
                      sizeof(float);
  static PerDevice<cudaError_t> attr_of;  // function attributes are per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const cudaError_t attr_err = attr_of.get(dev, [] {
    const size_t most = ((kAx0StageRows * M + 3) & ~(size_t)3) * sizeof(float) + (size_t)W * M * kT * sizeof(float) +
                        (BW ? kAx0StageRows * sizeof(float) : 0);
    return cudaFuncSetAttribute(ax0_kernel<K, L, M, BW, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
  }, cudaErrorInvalidDevice);
  if (attr_err != cudaSuccess) return attr_err;
  const cudaError_t e = launch_pdl(ax0_kernel<K, L, M, BW, IL>, dim3(p.G), dim3(32 * W), smem, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int K, int L, bool BW, bool IL>
static cudaError_t ax0_launch_il(const Ax0Params& p, int M, cudaStream_t st) {
  switch (M) {
    case 1: return ax0_launch1<K, L, 1, BW, IL>(p, st);
    case 2: return ax0_launch1<K, L, 2, BW, IL>(p, st);
    case 3: return ax0_launch1<K, L, 3, BW, IL>(p, st);
    default: return ax0_launch1<K, L, 4, BW, IL>(p, st);
  }
}

template <int K, int L, bool BW>
static cudaError_t ax0_launch_m(const Ax0Params& p, int M, bool il, cudaStream_t st) {
  if constexpr (K == 3)  // the interleaved layout exists for k = 3 only
    if (il) return ax0_launch_il<K, L, BW, true>(p, M, st);
  return ax0_launch_il<K, L, BW, false>(p, M, st);
}

template <bool BW>
static cudaError_t ax0_dispatch(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                                int k, int L, int64_t rows, int64_t cols, int interleave, void* workspace,
                                cudaStream_t st) {
  Ax0Params p{};
  p.codes = codes; p.scales = scales; p.x = x; p.out = out;
  p.nb = (int)(cols / kT);
  p.part = static_cast<float*>(workspace);
  p.counter = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) +
                                          (size_t)(kAx0MaxCtas + p.nb) * (size_t)M * kT * sizeof(float));
  p.R = rows; p.C = cols; p.N = (int64_t)p.nb * rows;
  p.G = ax0_grid(p.N);
  const int64_t per = (p.N + p.G - 1) / p.G;  // longest range, hence longest segment
  p.stage = (int)(per < kAx0StageRows ? per : kAx0StageRows);
  const bool il = interleave != 0;
  if (L == 16) {
    if (k == 2) return ax0_launch_m<2, 16, BW>(p, M, il, st);
    if (k == 3) return ax0_launch_m<3, 16, BW>(p, M, il, st);
    return ax0_launch_m<4, 16, BW>(p, M, il, st);
  }
  if (k == 2) return ax0_launch_m<2, 12, BW>(p, M, il, st);
  if (k == 3) return ax0_launch_m<3, 12, BW>(p, M, il, st);
  return ax0_launch_m<4, 12, BW>(p, M, il, st);
}

cudaError_t launch_matvec_axis0_fma(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                    uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                    void* workspace, cudaStream_t st) {
  return ax0_dispatch<false>(codes, scales, x, out, M, k, L, rows, cols, interleave, workspace, st);
}

cudaError_t launch_matvec_axis0_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                      uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                      void* workspace, cudaStream_t st) {
  return ax0_dispatch<true>(codes, scales, x, out, M, k, L, rows, cols, interleave, workspace, st);
}

// M >= 3 on the tensor cores, M <= 2 on the CUDA cores: at 17408 x 5120 (k = 2 / 3 / 4) the tensor-core kernel
// costs about the same for every M (34.7-36.8 / 38.9-40.8 / 34.9-37.5 us) while this kernel grows with M
// (28.6, 32.8, 38.1, 40.6 us at k = 2), so they cross between M = 2 and M = 3.
cudaError_t launch_matvec_axis0(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                void* workspace, cudaStream_t st) {
  if (M >= 3) return launch_matvec_axis0_tc(codes, scales, x, out, M, k, L, rows, cols, interleave, workspace, st);
  return launch_matvec_axis0_fma(codes, scales, x, out, M, k, L, rows, cols, interleave, workspace, st);
}

}  // namespace trellis
