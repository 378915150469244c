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
//   * a warp takes two stored rows at a time, one per half-warp; lane j of a
//     half owns outputs 16j .. 16j+15 of the column block: per row it loads
//     the two or three words that cover its 16 windows (already word-aligned
//     for even k) and takes the windows with compile-time shifts, two 16-bit
//     windows per funnel shift when L = 16 and k is even.  The CTA's warps
//     take interleaved row pairs.
//   * x[m][r]*scale[r] is staged once per CTA in shared memory and read with
//     a broadcast load per row; 1/d is applied after the sum.  The first code
//     words are requested before the staging so that their latency overlaps it.
//   * the CTA folds its warps in shared memory.  The slices of a column block
//     go in thread-block clusters of kAx0Cluster CTAs: each CTA of a cluster
//     folds its share of the outputs over the cluster's CTAs through
//     distributed shared memory and writes one fp32 partial per output to the
//     workspace.  The last CTA to arrive for a column block (an atomic
//     counter) folds the S / kAx0Cluster cluster partials in order, stores
//     bf16 and resets the counter -- one launch, deterministic, no atomics on
//     data.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace trellis {

constexpr int kAx0Warps = 4;
constexpr int kAx0Chunk = 4;    // row pairs per prefetch chunk
constexpr int kAx0Cluster = 8;  // CTAs (row slices) per thread-block cluster
constexpr int64_t kAx0TargetCtas = 152 * 5;

struct Ax0Plan {
  int nb;       // column blocks
  int S;        // row slices, a multiple of kAx0Cluster
  int64_t rps;  // rows per slice
};

static Ax0Plan ax0_plan(int64_t rows, int64_t cols) {
  Ax0Plan p;
  p.nb = (int)(cols / kT);
  int64_t rps = (rows * p.nb + kAx0TargetCtas - 1) / kAx0TargetCtas;
  if (rps < 32) rps = 32;
  if (rps > 1600) rps = 1600;  // keeps the staged slice (and its scales) within 48 KB of shared memory
  int64_t S = (rows + rps - 1) / rps;
  S = (S + kAx0Cluster - 1) / kAx0Cluster * kAx0Cluster;
  p.S = (int)S;
  p.rps = (rows + S - 1) / S;  // trailing slices may be short or empty
  return p;
}

size_t axis0_workspace_bytes(int M, int64_t rows, int64_t cols) {
  const Ax0Plan p = ax0_plan(rows, cols);
  const size_t part = (size_t)(p.S / kAx0Cluster) * (size_t)M * (size_t)cols * sizeof(float);
  return part + (((size_t)p.nb * sizeof(uint32_t) + 15) & ~(size_t)15);
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// fp32 at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), r;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

struct Ax0Params {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* out;
  float* part;        // [S / kAx0Cluster][M][cols]
  uint32_t* counter;  // [nb]
  int64_t R, C, rps;
  int nb, S;
  int interleave;  // 2: codes in the [nb/2][R][2*WPB] layout
};

template <int K, int L, int M, bool BW>
__global__ void __launch_bounds__(32 * kAx0Warps) ax0_kernel(const Ax0Params p) {
  constexpr int WPB = kT * K / 32;
  // Words of one lane's 16-position run: 15K + L bits, plus up to 16 bits of
  // misalignment when K is odd.
  constexpr bool kEven = (K % 2) == 0;
  constexpr int NR = (15 * K + L + (kEven ? 0 : 16) + 31) / 32;
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                        // [rps][M]  x*scale of this slice's rows
  float* red = smem + ((p.rps * M + 3) & ~(int64_t)3);  // [warps][M][256], 16-byte aligned
  float* scs = red + kAx0Warps * M * kT;                 // [rps] row scales (bf16-weight numerics)
  __shared__ uint32_t last_flag;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, j = lane & 15;
  const int cb = blockIdx.x, sl = blockIdx.y;
  const int64_t r0 = (int64_t)sl * p.rps;
  const int64_t r1 = (r0 + p.rps < p.R) ? r0 + p.rps : p.R;
  const int nr = r1 > r0 ? (int)(r1 - r0) : 0;

  // Half-warp `half` takes the odd or even row of each row pair; lane j of
  // the half owns block positions 16j .. 16j+15, whose windows start at
  // block bits (255-16j-i)*K, the lowest at lo = (240-16j)*K.
  const int lo = (kT - 16 * (j + 1)) * K;
  const int wa = lo >> 5, sh = lo & 31;
  int widx[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) widx[i] = (wa + i >= WPB) ? wa + i - WPB : wa + i;
  // row stride and first word of column block cb in either layout
  const int64_t rowWords = p.interleave ? 2 * WPB : (int64_t)p.nb * WPB;
  const uint32_t* base = p.interleave ? p.codes + (int64_t)(cb >> 1) * p.R * (2 * WPB) + (cb & 1) * WPB
                                      : p.codes + (int64_t)cb * WPB;

  // This warp's row pairs are warp, warp + W, ... (W warps per CTA); row
  // pair q holds rows 2q and 2q+1 of the slice.  They go in chunks of
  // kAx0Chunk pairs; the code words of the next chunk load while the current
  // chunk decodes.  Rows past the slice load a valid row and are skipped.
  const int np = (nr + 1) >> 1;
  const int nw = np > warp ? (np - warp + kAx0Warps - 1) / kAx0Warps : 0;
  const int nch = (nw + kAx0Chunk - 1) / kAx0Chunk;
  auto row_of = [&](int i) { return 2 * (warp + i * kAx0Warps) + half; };
  auto load_chunk = [&](uint32_t (&a)[kAx0Chunk][NR], int ch) {
#pragma unroll
    for (int u = 0; u < kAx0Chunk; ++u) {
      int i = ch * kAx0Chunk + u;
      if (i >= nw) i = nw - 1;
      int rl = row_of(i);
      if (rl >= nr) rl = nr - 1;
      const uint32_t* rw = base + (r0 + rl) * rowWords;
#pragma unroll
      for (int q = 0; q < NR; ++q) a[u][q] = __ldg(rw + widx[q]);
    }
  };
  uint32_t a0[kAx0Chunk][NR], a1[kAx0Chunk][NR];
  if (nch > 0) load_chunk(a0, 0);

  // stage x*scale (or x and the scales) of the slice, four rows per thread in flight
  for (int rb = threadIdx.x; rb < nr; rb += 4 * blockDim.x) {
    float sv[4], xv[4][M];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rl = rb + u * (int)blockDim.x;
      const int64_t r = r0 + (rl < nr ? rl : 0);
      sv[u] = f16_to_f32(__ldg(p.scales + r));
#pragma unroll
      for (int m = 0; m < M; ++m) xv[u][m] = bf16_to_f32(__ldg(p.x + (int64_t)m * p.R + r));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rl = rb + u * (int)blockDim.x;
      if (rl < nr) {
        // default numerics fold the row scale into x; bf16 weights need it per weight
#pragma unroll
        for (int m = 0; m < M; ++m) xs[rl * M + m] = BW ? xv[u][m] : __fmul_rn(xv[u][m], sv[u]);
        if (BW) scs[rl] = sv[u];
      }
    }
  }
  __syncthreads();

  const float2 nmagic = make_float2(-kMagic, -kMagic);
  float2 acc[M][8];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[m][i] = make_float2(0.f, 0.f);

  auto body = [&](const uint32_t (&raw)[NR], int rl) {
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
    float xr[M];
    if constexpr (M == 4) {
      const float4 v = *reinterpret_cast<const float4*>(xs + rl * 4);
      xr[0] = v.x; xr[1] = v.y; xr[2] = v.z; xr[3] = v.w;
    } else {
#pragma unroll
      for (int m = 0; m < M; ++m) xr[m] = xs[rl * M + m];
    }
    float sr = 0.f;
    if constexpr (BW) sr = scs[rl];
#pragma unroll
    for (int i2 = 0; i2 < 8; ++i2) {
      float2 y = __fadd2_rn(
          make_float2(__uint_as_float(code_magic(s[2 * i2])), __uint_as_float(code_magic(s[2 * i2 + 1]))), nmagic);
      if constexpr (BW) {  // bf16(value * scale), the expand weight
        const float2 wv = __fmul2_rn(value_rn2(y), make_float2(sr, sr));
        const uint32_t bb = pack_bf16x2(wv.x, wv.y);
        y = make_float2(bf16lo_to_f32(bb), bf16hi_to_f32(bb));
      }
#pragma unroll
      for (int m = 0; m < M; ++m) acc[m][i2] = __ffma2_rn(y, make_float2(xr[m], xr[m]), acc[m][i2]);
    }
  };
  auto run_chunk = [&](const uint32_t (&a)[kAx0Chunk][NR], int ch) {
#pragma unroll
    for (int u = 0; u < kAx0Chunk; ++u) {
      const int i = ch * kAx0Chunk + u;
      const int rl = row_of(i);
      if (i < nw && rl < nr) body(a[u], rl);
    }
  };
  for (int ch = 0; ch < nch; ch += 2) {
    if (ch + 1 < nch) load_chunk(a1, ch + 1);
    run_chunk(a0, ch);
    if (ch + 1 >= nch) break;
    if (ch + 2 < nch) load_chunk(a0, ch + 2);
    run_chunk(a1, ch + 1);
  }

  // fold the two halves of each warp, then the warps of this CTA into red[0 .. M*256)
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
  // red position m*256 + t holds block position t (output column cb*256 + t)
  for (int i = threadIdx.x; i < M * kT; i += blockDim.x) {
    float v = red[i];
#pragma unroll
    for (int w = 1; w < kAx0Warps; ++w) v += red[w * M * kT + i];
    red[i] = v;
  }
  // fold the cluster's CTAs (slices sl - rank .. sl - rank + kAx0Cluster - 1):
  // CTA `rank` takes outputs [rank, rank + 1) * M*256/kAx0Cluster
  cluster_sync();
  {
    constexpr int kShare = M * kT / kAx0Cluster;
    const uint32_t rank = cluster_rank();
    const int cl = sl / kAx0Cluster;
    for (int i = threadIdx.x; i < kShare; i += blockDim.x) {
      const int o = (int)rank * kShare + i;
      const int m = o / kT, t = o - m * kT;
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < kAx0Cluster; ++q) v += ld_dsmem(red + o, (uint32_t)q);
      p.part[((int64_t)cl * M + m) * p.C + (int64_t)cb * kT + t] = v;
    }
  }
  cluster_sync();  // no CTA leaves while another still reads its shared memory
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_flag = (atomicAdd(p.counter + cb, 1u) == (uint32_t)(p.S - 1)) ? 1u : 0u;
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const int ncl = p.S / kAx0Cluster;
  for (int i = threadIdx.x; i < M * kT; i += blockDim.x) {
    const int m = i / kT, t = i - m * kT;
    const float* pp = p.part + (int64_t)m * p.C + (int64_t)cb * kT + t;
    const int64_t stride = (int64_t)M * p.C;
    float v = 0.f;
    int s = 0;
    for (; s + 8 <= ncl; s += 8) {
      float q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) q[u] = __ldcg(pp + (s + u) * stride);
#pragma unroll
      for (int u = 0; u < 8; ++u) v += q[u];
    }
    for (; s < ncl; ++s) v += __ldcg(pp + s * stride);
    uint16_t o;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(o) : "f"(BW ? v : __fmul_rn(v, kRcpD)));
    p.out[(int64_t)m * p.C + (int64_t)cb * kT + t] = o;
  }
  if (threadIdx.x == 0) p.counter[cb] = 0u;
}

template <int K, int L, int M, bool BW>
static cudaError_t ax0_launch1(const Ax0Params& p, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)p.nb, (unsigned)p.S);
  cfg.blockDim = dim3(32 * kAx0Warps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kAx0Cluster;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ax0_kernel<K, L, M, BW>, p);
}

template <int K, int L, bool BW>
static cudaError_t ax0_launch_m(const Ax0Params& p, int M, cudaStream_t st) {
  const size_t sm = ((((size_t)p.rps * M + 3) & ~(size_t)3) + (size_t)kAx0Warps * M * kT + (BW ? (size_t)p.rps : 0)) *
                    sizeof(float);
  cudaError_t e;
  switch (M) {
    case 1: e = ax0_launch1<K, L, 1, BW>(p, sm, st); break;
    case 2: e = ax0_launch1<K, L, 2, BW>(p, sm, st); break;
    case 3: e = ax0_launch1<K, L, 3, BW>(p, sm, st); break;
    default: e = ax0_launch1<K, L, 4, BW>(p, sm, st); break;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool BW>
static cudaError_t ax0_dispatch(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                                int k, int L, int64_t rows, int64_t cols, int interleave, void* workspace,
                                cudaStream_t st) {
  const Ax0Plan pl = ax0_plan(rows, cols);
  if (pl.S > 65535) return cudaErrorInvalidConfiguration;  // grid y limit (more than 10^8 stored rows)
  Ax0Params p{};
  p.codes = codes; p.scales = scales; p.x = x; p.out = out;
  p.part = static_cast<float*>(workspace);
  p.counter = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + (size_t)(pl.S / kAx0Cluster) * (size_t)M *
                                                                              (size_t)cols * sizeof(float));
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
