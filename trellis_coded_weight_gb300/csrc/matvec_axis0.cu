// matvec_axis0.cu -- decode-fused matvec over an axis-0 trellis matrix (a
// stored W^T coded along the output dimension), M = 1..4.
//
// What is computed ("trellis-linear.ts" diff page: SCATTER_SOURCE and the
// partial fold of the scatter path; "trellis-balanced-scatter.ts"):
//   out[m][c] = bf16( sum_r (y(r,c)/d * scale[r]) * x[m][r] )
// The pages split the sum over stored rows into 128 slices, write every
// slice's partial vector and fold them with a separate reduction.
//
// GB300 design:
//   * a CTA owns one column block (256 outputs) and one contiguous slice of
//     the stored rows; the number of slices is chosen so that all CTAs are
//     resident at once (about five per SM on 152 SMs).
//   * lane j of a warp owns outputs 8j .. 8j+7 of the column block (the
//     balanced assignment of the pages' k=3 kernel, used for every k): per
//     stored row it loads the two words that cover its 8 windows, aligns them
//     once and takes the windows with compile-time shifts.  The CTA's warps
//     take interleaved rows.
//   * x[m][r]*scale[r] is staged once per CTA in shared memory and read with
//     a broadcast load per row; 1/d is applied after the sum.
//   * the CTA folds its warps in shared memory, writes one fp32 partial per
//     output to the workspace, and the last CTA to arrive for a column block
//     (an atomic counter) folds all slices in slice order, stores bf16 and
//     resets the counter -- one launch, deterministic, no atomics on data.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace trellis {

constexpr int kAx0Warps = 4;
constexpr int kAx0Chunk = 8;  // rows per prefetch chunk
constexpr int64_t kAx0TargetCtas = 152 * 5;

struct Ax0Plan {
  int nb;       // column blocks
  int S;        // row slices
  int64_t rps;  // rows per slice
};

static Ax0Plan ax0_plan(int64_t rows, int64_t cols) {
  Ax0Plan p;
  p.nb = (int)(cols / kT);
  int64_t rps = (rows * p.nb + kAx0TargetCtas - 1) / kAx0TargetCtas;
  if (rps < 32) rps = 32;
  if (rps > 1600) rps = 1600;  // keeps the staged slice (and its scales) within 48 KB of shared memory
  p.S = (int)((rows + rps - 1) / rps);
  p.rps = (rows + p.S - 1) / p.S;
  return p;
}

size_t axis0_workspace_bytes(int M, int64_t rows, int64_t cols) {
  const Ax0Plan p = ax0_plan(rows, cols);
  const size_t part = (size_t)p.S * (size_t)M * (size_t)cols * sizeof(float);
  return part + (((size_t)p.nb * sizeof(uint32_t) + 15) & ~(size_t)15);
}

struct Ax0Params {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* out;
  float* part;        // [S][M][cols]
  uint32_t* counter;  // [nb]
  int64_t R, C, rps;
  int nb, S;
  int interleave;  // 2: codes in the [nb/2][R][2*WPB] layout
};

template <int K, int L, int M, bool BW>
__global__ void __launch_bounds__(32 * kAx0Warps) ax0_kernel(const Ax0Params p) {
  constexpr int WPB = kT * K / 32;
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                        // [rps][M]  x*scale of this slice's rows
  float* red = smem + ((p.rps * M + 3) & ~(int64_t)3);  // [warps][M][256], 16-byte aligned
  float* scs = red + kAx0Warps * M * kT;                 // [rps] row scales (bf16-weight numerics)
  __shared__ uint32_t last_flag;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cb = blockIdx.x, sl = blockIdx.y;
  const int64_t r0 = (int64_t)sl * p.rps;
  const int64_t r1 = (r0 + p.rps < p.R) ? r0 + p.rps : p.R;
  const int nr = (int)(r1 - r0);

  for (int i = threadIdx.x; i < nr * M; i += blockDim.x) {
    const int rl = i / M, m = i - rl * M;
    const int64_t r = r0 + rl;
    const float xv = bf16_to_f32(__ldg(p.x + (int64_t)m * p.R + r));
    // default numerics fold the row scale into x; bf16 weights need it per weight
    xs[i] = BW ? xv : __fmul_rn(xv, f16_to_f32(__ldg(p.scales + r)));
  }
  if (BW)
    for (int i = threadIdx.x; i < nr; i += blockDim.x) scs[i] = f16_to_f32(__ldg(p.scales + r0 + i));
  __syncthreads();

  const int lo = (kT - 8 * (lane + 1)) * K;
  const int wa = lo >> 5, sh = lo & 31;
  const int wb = (wa + 1 == WPB) ? 0 : wa + 1;
  // row stride and first word of column block cb in either layout
  const int64_t rowWords = p.interleave ? 2 * WPB : (int64_t)p.nb * WPB;
  const uint32_t* base = p.interleave ? p.codes + (int64_t)(cb >> 1) * p.R * (2 * WPB) + (cb & 1) * WPB
                                      : p.codes + (int64_t)cb * WPB;
  const float2 nmagic = make_float2(-kMagic, -kMagic);

  float2 acc[M][4];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = make_float2(0.f, 0.f);

  auto body = [&](uint32_t a, uint32_t b, int rl) {
    uint32_t w[2];
    w[0] = __funnelshift_r(a, b, sh);
    w[1] = b >> sh;
    float xr[M];
    if constexpr (M == 4) {
      const float4 v = *reinterpret_cast<const float4*>(xs + rl * 4);
      xr[0] = v.x; xr[1] = v.y; xr[2] = v.z; xr[3] = v.w;
    } else {
#pragma unroll
      for (int m = 0; m < M; ++m) xr[m] = xs[rl * M + m];
    }
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
      const uint32_t s0 = window_at<L, 2>(w, (7 - 2 * i2) * K);
      const uint32_t s1 = window_at<L, 2>(w, (6 - 2 * i2) * K);
      float2 y = __fadd2_rn(make_float2(__uint_as_float(code_magic(s0)), __uint_as_float(code_magic(s1))),
                            nmagic);
      if constexpr (BW) {  // bf16(value * scale), the expand weight
        const float sr = scs[rl];
        const float2 w = __fmul2_rn(value_rn2(y), make_float2(sr, sr));
        const uint32_t bb = pack_bf16x2(w.x, w.y);
        y = make_float2(bf16lo_to_f32(bb), bf16hi_to_f32(bb));
      }
#pragma unroll
      for (int m = 0; m < M; ++m) acc[m][i2] = __ffma2_rn(y, make_float2(xr[m], xr[m]), acc[m][i2]);
    }
  };

  // This warp's rows are warp, warp + W, ... (W warps per CTA).  They go in
  // chunks of kAx0Chunk rows; the code words of the next chunk load while the
  // current chunk decodes.  Rows past the slice load a valid row and are skipped.
  const int nw = nr > warp ? (nr - warp + kAx0Warps - 1) / kAx0Warps : 0;
  const int nch = (nw + kAx0Chunk - 1) / kAx0Chunk;
  auto load_chunk = [&](uint32_t (&a)[kAx0Chunk], uint32_t (&b)[kAx0Chunk], int ch) {
#pragma unroll
    for (int u = 0; u < kAx0Chunk; ++u) {
      int i = ch * kAx0Chunk + u;
      if (i >= nw) i = nw - 1;
      const uint32_t* rw = base + (r0 + warp + (int64_t)i * kAx0Warps) * rowWords;
      a[u] = __ldg(rw + wa);
      b[u] = __ldg(rw + wb);
    }
  };
  auto run_chunk = [&](const uint32_t (&a)[kAx0Chunk], const uint32_t (&b)[kAx0Chunk], int ch) {
#pragma unroll
    for (int u = 0; u < kAx0Chunk; ++u) {
      const int i = ch * kAx0Chunk + u;
      if (i < nw) body(a[u], b[u], warp + i * kAx0Warps);
    }
  };
  if (nch > 0) {
    uint32_t a0[kAx0Chunk], b0[kAx0Chunk], a1[kAx0Chunk], b1[kAx0Chunk];
    load_chunk(a0, b0, 0);
    for (int ch = 0; ch < nch; ch += 2) {
      if (ch + 1 < nch) load_chunk(a1, b1, ch + 1);
      run_chunk(a0, b0, ch);
      if (ch + 1 >= nch) break;
      if (ch + 2 < nch) load_chunk(a0, b0, ch + 2);
      run_chunk(a1, b1, ch + 1);
    }
  }

  // fold the warps of this CTA
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float4* dst = reinterpret_cast<float4*>(red + (warp * M + m) * kT + 8 * lane);
    dst[0] = make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
    dst[1] = make_float4(acc[m][2].x, acc[m][2].y, acc[m][3].x, acc[m][3].y);
  }
  __syncthreads();
  // red position 8j+i holds block position t = 8j+i, i.e. output column cb*256 + t
  for (int i = threadIdx.x; i < M * kT; i += blockDim.x) {
    const int m = i / kT, t = i - m * kT;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kAx0Warps; ++w) v += red[(w * M + m) * kT + t];
    p.part[((int64_t)sl * M + m) * p.C + (int64_t)cb * kT + t] = v;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_flag = (atomicAdd(p.counter + cb, 1u) == (uint32_t)(p.S - 1)) ? 1u : 0u;
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  for (int i = threadIdx.x; i < M * kT; i += blockDim.x) {
    const int m = i / kT, t = i - m * kT;
    float v = 0.f;
    for (int s = 0; s < p.S; ++s) v += __ldcg(p.part + ((int64_t)s * M + m) * p.C + (int64_t)cb * kT + t);
    uint16_t o;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(o) : "f"(BW ? v : __fmul_rn(v, kRcpD)));
    p.out[(int64_t)m * p.C + (int64_t)cb * kT + t] = o;
  }
  if (threadIdx.x == 0) p.counter[cb] = 0u;
}

template <int K, int L, bool BW>
static cudaError_t ax0_launch_m(const Ax0Params& p, int M, cudaStream_t st) {
  const dim3 grid((unsigned)p.nb, (unsigned)p.S), block(32 * kAx0Warps);
  const size_t sm = ((((size_t)p.rps * M + 3) & ~(size_t)3) + (size_t)kAx0Warps * M * kT + (BW ? (size_t)p.rps : 0)) *
                    sizeof(float);
  switch (M) {
    case 1: ax0_kernel<K, L, 1, BW><<<grid, block, sm, st>>>(p); break;
    case 2: ax0_kernel<K, L, 2, BW><<<grid, block, sm, st>>>(p); break;
    case 3: ax0_kernel<K, L, 3, BW><<<grid, block, sm, st>>>(p); break;
    default: ax0_kernel<K, L, 4, BW><<<grid, block, sm, st>>>(p); break;
  }
  return cudaGetLastError();
}

template <bool BW>
static cudaError_t ax0_dispatch(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                                int k, int L, int64_t rows, int64_t cols, int interleave, void* workspace,
                                cudaStream_t st) {
  const Ax0Plan pl = ax0_plan(rows, cols);
  Ax0Params p{};
  p.codes = codes; p.scales = scales; p.x = x; p.out = out;
  p.part = static_cast<float*>(workspace);
  p.counter = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) +
                                          (size_t)pl.S * (size_t)M * (size_t)cols * sizeof(float));
  p.R = rows; p.C = cols; p.rps = pl.rps; p.nb = pl.nb; p.S = pl.S; p.interleave = interleave;
  if (L == 16) {
    if (k == 2) return ax0_launch_m<2, 16, BW>(p, M, st);
    if (k == 3) return ax0_launch_m<3, 16, BW>(p, M, st);
    return ax0_launch_m<4, 16, BW>(p, M, st);
  }
  if (k == 2) return ax0_launch_m<2, 12, BW>(p, M, st);
  if (k == 3) return ax0_launch_m<3, 12, BW>(p, M, st);
  return ax0_launch_m<4, 12, BW>(p, M, st);
}

cudaError_t launch_matvec_axis0(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                void* workspace, cudaStream_t st) {
  return ax0_dispatch<false>(codes, scales, x, out, M, k, L, rows, cols, interleave, workspace, st);
}

cudaError_t launch_matvec_axis0_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                      uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols, int interleave,
                                      void* workspace, cudaStream_t st) {
  return ax0_dispatch<true>(codes, scales, x, out, M, k, L, rows, cols, interleave, workspace, st);
}

}  // namespace trellis
