// matvec_axis1.cu -- decode-fused matvec over axis-1 trellis matrices, M = 1..4,
// and the fused gate/up SwiGLU layer.
//
// What is computed ("trellis-linear.ts" diff page: REDUCE_SOURCE, GATEUP_SOURCE;
// "trellis-shared-m.ts": the shared-M variants):
//   out[m][r] = bf16( sum_c (y(r,c)/d * scale[r]) * x[m][c] )
// with the pages' default packed numerics (fp32 weight, no bf16 rounding), and
// for gate/up the bf16 cast chain gate -> up -> sigmoid -> silu -> product.
//
// GB300 design (differs from the pages' SIMD-group-per-row kernel):
//   * lane = output row.  A warp owns 32 consecutive rows; the CTA's S warps
//     split the row's blocks (the reduction axis) among themselves and fold
//     their partial sums through shared memory at the end.  No cross-lane
//     shuffle reduction is needed.
//   * every lane decodes runs of 32 consecutive positions held in K+1 registers
//     (the run's K words plus the spill word), so each window shift is a
//     compile-time constant; for L = 16 and K in {2,4} one funnel shift yields
//     two windows 16 bits apart.
//   * x is staged per block as fp32 in shared memory and read with broadcast
//     128-bit loads (every lane of the warp reads the same address), so the
//     x traffic costs one shared-memory wavefront per 4 positions x 32 rows.
//   * the 1MAD byte sum is one dp4a onto a float bias, y = float - bias with
//     packed f32x2 arithmetic, and y*x accumulates with packed f32x2 FMA; the
//     per-row factor scale/d is applied once after the reduction (the pages
//     apply it per weight; the difference is a few fp32 ulp per sum).
//   * each decoded weight is shared across the M input rows.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace trellis {

struct Mv1Params {
  const uint32_t* codes[2];
  const uint16_t* scales[2];
  const uint16_t* x;
  uint16_t* out;
  int64_t R;   // stored rows (= output features)
  int64_t C;   // coded columns (= input features)
  int nb;      // blocks per row (C / 256)
};

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

// The SwiGLU cast chain of GATEUP_SOURCE on fp32 gate/up sums.
__device__ __forceinline__ uint16_t swiglu_chain(float gate, float up) {
  const float g = bf16_to_f32(f32_to_bf16_rn(gate));
  const float u = bf16_to_f32(f32_to_bf16_rn(up));
  const float sig = bf16_to_f32(f32_to_bf16_rn(__fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)))));
  const float silu = bf16_to_f32(f32_to_bf16_rn(__fmul_rn(g, sig)));
  return f32_to_bf16_rn(__fmul_rn(silu, u));
}

template <int K, int L, int M, bool GU>
__global__ void __launch_bounds__(256) mv1_kernel(const Mv1Params p) {
  extern __shared__ __align__(16) float smem[];
  constexpr int NMAT = GU ? 2 : 1;
  constexpr int WPB = kT * K / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, S = blockDim.x >> 5;
  float* xs = smem + warp * (M * kT);
  float* red = smem + S * M * kT;

  const int64_t row = (int64_t)blockIdx.x * 32 + lane;
  const int64_t rr = row < p.R ? row : p.R - 1;  // clamped rows load valid memory and store nothing
  const int b0 = (int)((int64_t)warp * p.nb / S);
  const int b1 = (int)((int64_t)(warp + 1) * p.nb / S);

  const uint4* crow[NMAT];
#pragma unroll
  for (int t = 0; t < NMAT; ++t)
    crow[t] = reinterpret_cast<const uint4*>(p.codes[t] + rr * (int64_t)p.nb * WPB);

  float2 acc[NMAT][M][2];
#pragma unroll
  for (int t = 0; t < NMAT; ++t)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[t][m][0] = acc[t][m][1] = make_float2(0.f, 0.f);
  const float2 nmagic = make_float2(-kMagic, -kMagic);

  for (int b = b0; b < b1; ++b) {
    // codes of block b of this lane's row (issued first; x staging overlaps their latency)
    uint32_t cw[NMAT][WPB];
#pragma unroll
    for (int t = 0; t < NMAT; ++t)
#pragma unroll
      for (int i = 0; i < WPB / 4; ++i) {
        const uint4 v = __ldg(crow[t] + (int64_t)b * (WPB / 4) + i);
        cw[t][4 * i] = v.x; cw[t][4 * i + 1] = v.y; cw[t][4 * i + 2] = v.z; cw[t][4 * i + 3] = v.w;
      }
    // x[:, block b] as fp32 in this warp's shared tile
    __syncwarp();
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)m * p.C + (int64_t)b * kT) + lane);
      float4* dst = reinterpret_cast<float4*>(xs + m * kT + 8 * lane);
      dst[0] = make_float4(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x), bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
      dst[1] = make_float4(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z), bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
    }
    __syncwarp();
    // eight runs of 32 positions; run q holds positions 32q .. 32q+31 in
    // words (7-q)*K .. (7-q)*K+K-1, the spill word follows (wrapping for q = 0)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
#pragma unroll
      for (int t = 0; t < NMAT; ++t) {
        uint32_t w[K + 1];
#pragma unroll
        for (int i = 0; i < K; ++i) w[i] = cw[t][(7 - q) * K + i];
        w[K] = cw[t][((8 - q) * K) % WPB];
        uint32_t s[32];
        run_states<K, L>(w, s);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float2 ya = __fadd2_rn(make_float2(__uint_as_float(code_magic(s[4 * j4])),
                                                   __uint_as_float(code_magic(s[4 * j4 + 1]))), nmagic);
          const float2 yb = __fadd2_rn(make_float2(__uint_as_float(code_magic(s[4 * j4 + 2])),
                                                   __uint_as_float(code_magic(s[4 * j4 + 3]))), nmagic);
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const float4 xv = *reinterpret_cast<const float4*>(xs + m * kT + 32 * q + 4 * j4);
            acc[t][m][0] = __ffma2_rn(ya, make_float2(xv.x, xv.y), acc[t][m][0]);
            acc[t][m][1] = __ffma2_rn(yb, make_float2(xv.z, xv.w), acc[t][m][1]);
          }
        }
      }
    }
  }

  // fold the S warps' partial sums of each row in a fixed order
#pragma unroll
  for (int t = 0; t < NMAT; ++t)
#pragma unroll
    for (int m = 0; m < M; ++m)
      red[((t * S + warp) * M + m) * 32 + lane] =
          (acc[t][m][0].x + acc[t][m][0].y) + (acc[t][m][1].x + acc[t][m][1].y);
  __syncthreads();
  if (warp != 0 || row >= p.R) return;
  float f[NMAT];
#pragma unroll
  for (int t = 0; t < NMAT; ++t) f[t] = __fmul_rn(f16_to_f32(p.scales[t][row]), kRcpD);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float v[NMAT];
#pragma unroll
    for (int t = 0; t < NMAT; ++t) {
      float a = 0.f;
      for (int w = 0; w < S; ++w) a += red[((t * S + w) * M + m) * 32 + lane];
      v[t] = __fmul_rn(a, f[t]);
    }
    uint16_t o;
    if constexpr (GU) o = swiglu_chain(v[0], v[1]);
    else o = f32_to_bf16_rn(v[0]);
    p.out[(int64_t)m * p.R + row] = o;
  }
}

// Warps per CTA: the row's blocks are split S ways.
static int mv1_splits(int nb) { return nb < 4 ? nb : 4; }

template <int K, int L, bool GU>
static cudaError_t mv1_launch_m(const Mv1Params& p, int M, cudaStream_t st) {
  const int S = mv1_splits(p.nb);
  const int nmat = GU ? 2 : 1;
  const size_t sm = (size_t)S * M * kT * sizeof(float) + (size_t)nmat * S * M * 32 * sizeof(float);
  const dim3 grid((unsigned)((p.R + 31) / 32)), block(32 * S);
  switch (M) {
    case 1: mv1_kernel<K, L, 1, GU><<<grid, block, sm, st>>>(p); break;
    case 2: mv1_kernel<K, L, 2, GU><<<grid, block, sm, st>>>(p); break;
    case 3: mv1_kernel<K, L, 3, GU><<<grid, block, sm, st>>>(p); break;
    default: mv1_kernel<K, L, 4, GU><<<grid, block, sm, st>>>(p); break;
  }
  return cudaGetLastError();
}

template <bool GU>
static cudaError_t mv1_dispatch(const Mv1Params& p, int k, int L, int M, cudaStream_t st) {
  if (L == 16) {
    if (k == 2) return mv1_launch_m<2, 16, GU>(p, M, st);
    if (k == 3) return mv1_launch_m<3, 16, GU>(p, M, st);
    return mv1_launch_m<4, 16, GU>(p, M, st);
  }
  if (k == 2) return mv1_launch_m<2, 12, GU>(p, M, st);
  if (k == 3) return mv1_launch_m<3, 12, GU>(p, M, st);
  return mv1_launch_m<4, 12, GU>(p, M, st);
}

cudaError_t launch_matvec_axis1(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                cudaStream_t st) {
  Mv1Params p{};
  p.codes[0] = p.codes[1] = codes;
  p.scales[0] = p.scales[1] = scales;
  p.x = x; p.out = out; p.R = rows; p.C = cols; p.nb = (int)(cols / kT);
  return mv1_dispatch<false>(p, k, L, M, st);
}

cudaError_t launch_gateup_swiglu(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                                 const uint16_t* uscales, const uint16_t* x, uint16_t* out, int M, int k,
                                 int L, int64_t rows, int64_t cols, cudaStream_t st) {
  Mv1Params p{};
  p.codes[0] = gcodes; p.codes[1] = ucodes;
  p.scales[0] = gscales; p.scales[1] = uscales;
  p.x = x; p.out = out; p.R = rows; p.C = cols; p.nb = (int)(cols / kT);
  return mv1_dispatch<true>(p, k, L, M, st);
}

}  // namespace trellis
