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
//   * the 1MAD byte sum is one dp4a onto -510 and y an int-to-float
//     conversion (ALU pipe, leaving the FMA-heavy pipe to the multiply, the
//     byte sum and the FMAs; at k = 3 half of them take the float-bias
//     subtraction instead), and y*x accumulates with packed f32x2 FMA; the
//     per-row factor scale/d is applied once after the reduction (the pages
//     apply it per weight; the difference is a few fp32 ulp per sum).
//   * each decoded weight is shared across the M input rows.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "pdl.cuh"

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

// A half block: runs 7..4 (block words [0, 4K)) or runs 3..0 (words
// [4K, 8K)), plus the spill word of its last run (word 4K, or word 0 where
// the block wraps).
template <int K, int NMAT>
struct HalfBlock {
  uint32_t w[NMAT][4 * K + 1];
};

template <int K, int NMAT>
__device__ __forceinline__ void load_half(HalfBlock<K, NMAT>& hbk, const uint32_t* const (&crow)[NMAT], int ci) {
  constexpr int WPB = kT * K / 32;
  const int b = ci >> 1, hb = ci & 1;
#pragma unroll
  for (int t = 0; t < NMAT; ++t) {
    const uint32_t* blk = crow[t] + (int64_t)b * WPB;
    const uint4* v4 = reinterpret_cast<const uint4*>(blk + hb * 4 * K);
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const uint4 v = __ldg(v4 + i);
      hbk.w[t][4 * i] = v.x; hbk.w[t][4 * i + 1] = v.y; hbk.w[t][4 * i + 2] = v.z; hbk.w[t][4 * i + 3] = v.w;
    }
    hbk.w[t][4 * K] = __ldg(blk + (hb ? 0 : 4 * K));
  }
}

template <int K, int L, int M, bool GU, bool BW>
__global__ void __launch_bounds__(512) mv1_kernel(const Mv1Params p) {
  extern __shared__ __align__(16) float smem[];
  pdl_enter();
  constexpr int NMAT = GU ? 2 : 1;
  constexpr int WPB = kT * K / 32;
  constexpr int HB = kT / 2;  // positions per half block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, S = blockDim.x >> 5;
  float* xs = smem + warp * (M * HB);
  float* red = smem + S * M * HB;

  const int64_t row = (int64_t)blockIdx.x * 32 + lane;
  const int64_t rr = row < p.R ? row : p.R - 1;  // clamped rows load valid memory and store nothing
  const int c0 = (int)((int64_t)warp * 2 * p.nb / S);  // this warp's half blocks [c0, c1)
  const int c1 = (int)((int64_t)(warp + 1) * 2 * p.nb / S);

  const uint32_t* crow[NMAT];
#pragma unroll
  for (int t = 0; t < NMAT; ++t) crow[t] = p.codes[t] + rr * (int64_t)p.nb * WPB;

  float2 acc[NMAT][M][2];
#pragma unroll
  for (int t = 0; t < NMAT; ++t)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[t][m][0] = acc[t][m][1] = make_float2(0.f, 0.f);
  // bf16-weight numerics: each weight is bf16(value * scale) before the FMA
  float wsc[NMAT];
#pragma unroll
  for (int t = 0; t < NMAT; ++t) wsc[t] = BW ? f16_to_f32(__ldg(p.scales[t] + rr)) : 1.0f;
  auto bf16_weights = [&](float2 y, float sc) -> float2 {
    const float2 w = __fmul2_rn(value_rn2(y), make_float2(sc, sc));
    const uint32_t b = pack_bf16x2(w.x, w.y);
    return make_float2(bf16lo_to_f32(b), bf16hi_to_f32(b));
  };

  auto process = [&](const HalfBlock<K, NMAT>& hbk, int ci) {
    const int b = ci >> 1, hb = ci & 1;
    // x of this half block (positions 128*(1-hb) .. +127 of block b) as fp32
    const int pos0 = 128 * (1 - hb);
    __syncwarp();
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p.x + (int64_t)m * p.C + (int64_t)b * kT + pos0) + lane);
      *reinterpret_cast<float4*>(xs + m * HB + 4 * lane) =
          make_float4(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x), bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
    }
    __syncwarp();
    // runs r4 = 0..3 of the half: q = 7 - 4*hb - r4 holds positions 32q .. 32q+31
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const int xq = 32 * (3 - r4);  // offset of run q inside the half block's positions
#pragma unroll
      for (int t = 0; t < NMAT; ++t) {
        uint32_t w[K + 1];
#pragma unroll
        for (int i = 0; i <= K; ++i) w[i] = hbk.w[t][r4 * K + i];
        uint32_t s[32];
        run_states<K, L>(w, s);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          // y through the int-to-float conversion (ALU pipe); at K = 3, whose window extraction takes more
          // ALU work, every second pair through the float-bias subtraction on the FMA pipes instead (exact
          // either way)
          float2 ya = code_y2_alu(s[4 * j4], s[4 * j4 + 1]);
          float2 yb = K == 3 ? __fadd2_rn(make_float2(__uint_as_float(code_magic(s[4 * j4 + 2])),
                                                      __uint_as_float(code_magic(s[4 * j4 + 3]))),
                                          make_float2(-kMagic, -kMagic))
                             : code_y2_alu(s[4 * j4 + 2], s[4 * j4 + 3]);
          if constexpr (BW) {
            ya = bf16_weights(ya, wsc[t]);
            yb = bf16_weights(yb, wsc[t]);
          }
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const float4 xv = *reinterpret_cast<const float4*>(xs + m * HB + xq + 4 * j4);
            acc[t][m][0] = __ffma2_rn(ya, make_float2(xv.x, xv.y), acc[t][m][0]);
            acc[t][m][1] = __ffma2_rn(yb, make_float2(xv.z, xv.w), acc[t][m][1]);
          }
        }
      }
    }
  };

  // Half blocks in order; each lane's loads are issued at the top of the
  // half block and the warp's x staging overlaps their latency.  (Loading the
  // next half block ahead into a second register set measured slower.)
  for (int ci = c0; ci < c1; ++ci) {
    HalfBlock<K, NMAT> hbk;
    load_half<K, NMAT>(hbk, crow, ci);
    process(hbk, ci);
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
  for (int t = 0; t < NMAT; ++t) f[t] = BW ? 1.0f : __fmul_rn(f16_to_f32(p.scales[t][row]), kRcpD);
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

// Warps per CTA (the row's half blocks are split S ways): as many as keep
// four CTAs resident per SM with this instantiation's register count, so the
// R/32 CTAs of a large matrix run in a single wave; never more than the row
// has half blocks, and at most 16.  Registers are allocated per thread in
// units of 8, so the count is rounded up first.  Among the counts within a
// quarter of that bound, one that divides the half blocks evenly is taken, so
// that no warp of the CTA has a half block more than the others.
int mv1_splits(int nb, int regs) {
  const int r8 = ((regs > 0 ? regs : 64) + 7) & ~7;
  int s = 65536 / (4 * 32 * r8);
  if (s > 2 * nb) s = 2 * nb;
  if (s > 16) s = 16;
  if (s < 1) s = 1;
  for (int c = s; c * 4 >= s * 3; --c)
    if ((2 * nb) % c == 0) return c;
  return s;
}

template <int K, int L, int M, bool GU, bool BW>
static cudaError_t mv1_launch(const Mv1Params& p, cudaStream_t st) {
  static PerDevice<int> regs_of;  // per instantiation and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const int regs = regs_of.get(dev, [] {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, mv1_kernel<K, L, M, GU, BW>) != cudaSuccess) {
      cudaGetLastError();
      return 0;  // mv1_splits assumes 64 registers
    }
    return a.numRegs;
  }, 0);
  const int S = mv1_splits(p.nb, regs);
  const int nmat = GU ? 2 : 1;
  const size_t sm = (size_t)S * M * (kT / 2) * sizeof(float) + (size_t)nmat * S * M * 32 * sizeof(float);
  const dim3 grid((unsigned)((p.R + 31) / 32)), block(32 * S);
  const cudaError_t e = launch_pdl(mv1_kernel<K, L, M, GU, BW>, grid, block, sm, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int K, int L, bool GU, bool BW>
static cudaError_t mv1_launch_m(const Mv1Params& p, int M, cudaStream_t st) {
  switch (M) {
    case 1: return mv1_launch<K, L, 1, GU, BW>(p, st);
    case 2: return mv1_launch<K, L, 2, GU, BW>(p, st);
    case 3: return mv1_launch<K, L, 3, GU, BW>(p, st);
    default: return mv1_launch<K, L, 4, GU, BW>(p, st);
  }
}

template <bool GU, bool BW = false>
static cudaError_t mv1_dispatch(const Mv1Params& p, int k, int L, int M, cudaStream_t st) {
  if (L == 16) {
    if (k == 2) return mv1_launch_m<2, 16, GU, BW>(p, M, st);
    if (k == 3) return mv1_launch_m<3, 16, GU, BW>(p, M, st);
    return mv1_launch_m<4, 16, GU, BW>(p, M, st);
  }
  if (k == 2) return mv1_launch_m<2, 12, GU, BW>(p, M, st);
  if (k == 3) return mv1_launch_m<3, 12, GU, BW>(p, M, st);
  return mv1_launch_m<4, 12, GU, BW>(p, M, st);
}

// Load-only floor: the axis-1 matvec's access to the packed stream (lane =
// row, the row's half blocks split over the CTA's warps, K 16-byte loads and
// the spill word per half block) with no decode; every loaded word is folded
// by XOR so that the loads stay live, and the fold is stored per row.  Its
// bandwidth is what this access pattern can reach on HBM.
template <int K>
__global__ void __launch_bounds__(512) load_floor_kernel(const uint32_t* codes, uint32_t* out, int64_t R, int nb) {
  extern __shared__ uint32_t fold[];
  constexpr int WPB = kT * K / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, S = blockDim.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * 32 + lane;
  const int64_t rr = row < R ? row : R - 1;
  const int c0 = (int)((int64_t)warp * 2 * nb / S), c1 = (int)((int64_t)(warp + 1) * 2 * nb / S);
  const uint32_t* crow[1] = {codes + rr * (int64_t)nb * WPB};
  uint32_t acc = 0;
  for (int ci = c0; ci < c1; ++ci) {
    HalfBlock<K, 1> hbk;
    load_half<K, 1>(hbk, crow, ci);
#pragma unroll
    for (int i = 0; i <= 4 * K; ++i) acc ^= hbk.w[0][i];
  }
  fold[warp * 32 + lane] = acc;
  __syncthreads();
  if (warp != 0 || row >= R) return;
  uint32_t v = 0;
  for (int w = 0; w < S; ++w) v ^= fold[w * 32 + lane];
  out[row] = v;
}

cudaError_t launch_load_floor(const uint32_t* codes, uint32_t* out, int k, int64_t rows, int64_t cols,
                              cudaStream_t st) {
  const int nb = (int)(cols / kT);
  int S = 16;
  if (S > 2 * nb) S = 2 * nb;
  const dim3 grid((unsigned)((rows + 31) / 32)), block(32 * S);
  const size_t sm = (size_t)S * 32 * sizeof(uint32_t);
  if (k == 2) load_floor_kernel<2><<<grid, block, sm, st>>>(codes, out, rows, nb);
  else if (k == 3) load_floor_kernel<3><<<grid, block, sm, st>>>(codes, out, rows, nb);
  else load_floor_kernel<4><<<grid, block, sm, st>>>(codes, out, rows, nb);
  return cudaGetLastError();
}

// Coalesced load floor: a warp reads whole stored rows, its lanes on consecutive 16-byte chunks of the row
// (a row of 1280-2560 bytes in 3-5 requests), warps striding over the rows in a single wave; every word is
// folded by XOR so the loads stay live.  Its bandwidth is what a fully coalesced read of the same stream
// reaches at this size.
__global__ void __launch_bounds__(256) load_floor_rows_kernel(const uint4* codes, uint32_t* out, int64_t R,
                                                               int chunks) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < R; r += nwarps) {
    const uint4* row = codes + r * chunks;
    uint32_t acc = 0;
    for (int c = lane; c < chunks; c += 32) {
      const uint4 v = __ldg(row + c);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) out[r] = acc;
  }
}

cudaError_t launch_load_floor_rows(const uint32_t* codes, uint32_t* out, int k, int64_t rows, int64_t cols,
                                   cudaStream_t st) {
  static PerDevice<int> per_sm_of;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const int per_sm = per_sm_of.get(dev, [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, load_floor_rows_kernel, 256, 0) != cudaSuccess) {
      cudaGetLastError();
      n = 1;
    }
    return n < 1 ? 1 : n;
  }, 1);
  const int chunks = (int)(cols * k / 128);  // 16-byte chunks per row (cols is a multiple of 256)
  int64_t grid = (int64_t)device_sm_count() * per_sm;
  const int64_t need = (rows + 7) / 8;
  if (grid > need) grid = need;
  load_floor_rows_kernel<<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(codes), out, rows, chunks);
  return cudaGetLastError();
}

cudaError_t launch_matvec_axis1_fma(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                    uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                    cudaStream_t st) {
  Mv1Params p{};
  p.codes[0] = p.codes[1] = codes;
  p.scales[0] = p.scales[1] = scales;
  p.x = x; p.out = out; p.R = rows; p.C = cols; p.nb = (int)(cols / kT);
  return mv1_dispatch<false>(p, k, L, M, st);
}

cudaError_t launch_matvec_axis1_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                      uint16_t* out, int M, int k, int L, int64_t rows, int64_t cols,
                                      cudaStream_t st) {
  Mv1Params p{};
  p.codes[0] = p.codes[1] = codes;
  p.scales[0] = p.scales[1] = scales;
  p.x = x; p.out = out; p.R = rows; p.C = cols; p.nb = (int)(cols / kT);
  return mv1_dispatch<false, true>(p, k, L, M, st);
}

cudaError_t launch_gateup_swiglu_fma(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                                     const uint16_t* uscales, const uint16_t* x, uint16_t* out, int M, int k,
                                     int L, int64_t rows, int64_t cols, cudaStream_t st) {
  Mv1Params p{};
  p.codes[0] = gcodes; p.codes[1] = ucodes;
  p.scales[0] = gscales; p.scales[1] = uscales;
  p.x = x; p.out = out; p.R = rows; p.C = cols; p.nb = (int)(cols / kT);
  return mv1_dispatch<true>(p, k, L, M, st);
}

}  // namespace trellis
