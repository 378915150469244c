// matvec_axis0_tc.cu -- decode-fused matvec over an axis-0 trellis matrix (a stored W^T coded along the output
// dimension), M = 1..4, with the y * x*scale accumulation on the tensor cores.
//
// What is computed ("trellis-linear.ts" diff page: SCATTER_SOURCE and the partial fold of the scatter path;
// "trellis-balanced-scatter.ts"):
//   out[m][c] = bf16( sum_r (y(r,c)/d * scale[r]) * x[m][r] )
// with the pages' default packed numerics; 1/d multiplies the folded sum.
//
// GB300 design.  The split over the GPU and the fold of the partial sums are those of the CUDA-core kernel
// (axis0_split.cuh): CTA c takes an equal share of the (column block, stored row) pairs.  Within a CTA:
//   * the stored rows of a segment go through shared memory in pieces of 256 or 512 rows, in a ring of three:
//     while piece j is decoded, piece j+1 has landed and piece j+2 arrives -- its code words by 16-byte cp.async
//     (rows laid out so that the decoders' reads are free of bank conflicts), its x and scales by plain loads
//     held in registers and stored as B rows after the decode.  One barrier per piece.
//   * x[m][r]*scale[r] is exact in fp32 (bf16 times fp16: at most 19 significant bits).  It is split into a
//     tf32 high part (the top 11 significant bits) and the exact remainder (at most 8 bits), and the MMA's 8
//     token columns hold both: columns 0..3 the high parts of tokens 0..3, columns 4..7 the remainders.  y is an
//     integer in [-510, 510], so every product is exact and only the fp32 accumulation rounds.
//   * 16 warps: 4 column quarters (64 outputs, four 16-row MMA tiles) x 4 row slices (every fourth 8-row
//     k-step of a piece).  Lane (g, t) decodes stored rows t and t+4 of the k-step at the 8 outputs that the
//     tiles' A rows g and g+8 stand for.  Which outputs those are is chosen per k so that the windows come out
//     cheaply (axis0_windows.cuh).
//   * a tensor-core accumulation chain is at most kA0tChainSteps k-steps of a warp; longer runs are added into
//     fp32 sums.  The first two pieces of a CTA are a quarter and a half of a full one.
//   * measured at 17408 x 5120 (k = 2): 34.7-36.8 us for M = 1..4, against 28.6-40.6 us on the CUDA cores; the
//     matvec takes this kernel for M >= 3.  The steady state decodes a 512-row piece in about 5 us per CTA at
//     ~0.65 instructions per cycle per scheduler (16 warps a SM, 118-125 registers), about 6.9 instructions per
//     weight.
//   * at the end of a segment the lanes add the two token halves (a shuffle), the row slices fold through
//     shared memory in a fixed order and the CTA writes its partial (axis0_split.cuh).
#include <cstdint>
#include <cuda_runtime.h>

#include "axis0_split.cuh"
#include "axis0_windows.cuh"
#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "mma_tf32.cuh"
#include "pdl.cuh"

namespace trellis {
namespace {

constexpr int kA0tWarps = 16;
constexpr int kA0tSlices = kA0tWarps / 4;
constexpr int kA0tBufs = 3;        // pieces in flight: decoded, landed, arriving
constexpr int kA0tChainSteps = 64;  // k-steps of a warp per tensor-core accumulation chain (at most)

// Stored rows per staged piece: as many as three buffers of code words and B rows fit in shared memory.
template <int K>
constexpr int a0t_piece() { return K == 4 ? 256 : 512; }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A read-only 16-bit load issued where it stands: the asm is volatile, so the compiler keeps it ahead of the
// tensor-core loop (whose MMAs are volatile asm too) instead of sinking it next to its use after the loop.
__device__ __forceinline__ uint16_t ldg_u16_early(const uint16_t* ptr) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(ptr));
  return v;
}

// Staged words per row: rows t = 0..3 of a k-step (the four rows one load instruction reads) fall in distinct
// banks.  k = 2: 16 + 4; k = 3: 24, whose row offsets already fall 8 banks apart for the <= 8 words a lane set
// reads of each row; k = 4: 32 + 8.
template <int K>
constexpr int a0t_stride() { return K == 2 ? 20 : K == 3 ? 24 : 40; }

template <int K>
constexpr size_t a0t_smem(int M) {
  return ((size_t)kA0tBufs * a0t_piece<K>() * (a0t_stride<K>() + 8) + (size_t)kA0tSlices * M * kT) *
         sizeof(float);
}

template <int K, int L, int M, bool IL>
__global__ void __launch_bounds__(32 * kA0tWarps, 1) ax0tc_kernel(const Ax0Params p) {
  using Dec = A0Windows<K, L>;
  constexpr int WPB = kT * K / 32;
  constexpr int CH = WPB / 4;  // 16-byte chunks of a row's block
  constexpr int ST = a0t_stride<K>();
  constexpr int P = a0t_piece<K>();
  constexpr int kPieceSteps = P / 8 / kA0tSlices;  // k-steps of a warp in a full piece
  constexpr int kCopyRows = 32 * kA0tWarps / CH;  // rows one pass of the CTA's 16-byte copies covers
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_enter();
  uint32_t* cbuf = reinterpret_cast<uint32_t*>(smem);             // [kA0tBufs][P][ST] code words
  float* xsb = reinterpret_cast<float*>(cbuf + kA0tBufs * P * ST);  // [kA0tBufs][P/8][4][8][2] B operands
  float* red = xsb + kA0tBufs * P * 8;                             // [kA0tSlices][M][256]
  __shared__ int pend[kAx0MaxPending];
  __shared__ uint32_t is_last[kAx0MaxPending];
  int npend = 0;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int Q = warp & 3, slice = warp >> 2;
  const Dec dec(Q, g);
  const int64_t rowWords = IL ? 2 * WPB : (int64_t)p.nb * WPB;

  const int c = blockIdx.x;
  const int64_t f0 = (int64_t)c * p.N / p.G, f1 = (int64_t)(c + 1) * p.N / p.G;

  // A piece: up to P consecutive stored rows [r0, r0 + nr) of column block cb, inside this CTA's range
  // [f0, f1); `next` steps from piece j (starting at work item f) to piece j+1.  The first two pieces are a
  // quarter and a half of P, so that the first decode waits for a small copy rather than for two full pieces
  // requested by every CTA at once.
  struct Piece {
    int cb, nr, j;
    int64_t r0, f;
  };
  auto fit = [&](Piece& q) {
    const int cap = q.j == 0 ? P / 4 : (q.j == 1 ? P / 2 : P);
    int64_t n = p.R - q.r0;
    if (n > f1 - q.f) n = f1 - q.f;
    q.nr = (int)(n < cap ? n : cap);
  };
  auto next = [&](Piece q) {
    q.f += q.nr;
    q.r0 += q.nr;
    if (q.r0 == p.R) {
      ++q.cb;
      q.r0 = 0;
    }
    ++q.j;
    fit(q);
    return q;
  };
  // The piece's code words into buffer b: 16-byte copies, thread tid on chunk tid % CH of rows
  // tid / CH + kCopyRows*u; staged rows are ST words apart.
  const int cp_row = threadIdx.x / CH, cp_ch = threadIdx.x - cp_row * CH;
  auto issue_codes = [&](const Piece& q, int b) {
    if (cp_row >= kCopyRows) return;
    const uint32_t* src = (IL ? p.codes + (int64_t)(q.cb >> 1) * p.R * (2 * WPB) + (q.cb & 1) * WPB
                              : p.codes + (int64_t)q.cb * WPB) +
                          (q.r0 + cp_row) * rowWords + 4 * cp_ch;
    uint32_t* dst = cbuf + (b * P + cp_row) * ST + 4 * cp_ch;
#pragma unroll 4
    for (int r = cp_row; r < q.nr; r += kCopyRows, src += kCopyRows * rowWords, dst += kCopyRows * ST)
      cp_async16(dst, src);
  };
  // The piece's x and scales: thread r < P loads those of row r0 + r into registers ...
  struct XRow {
    float x[M], s;
  };
  auto load_x = [&](const Piece& q, XRow& v) {
    const int r = threadIdx.x;
    if (r < q.nr) {
      v.s = f16_to_f32(ldg_u16_early(p.scales + q.r0 + r));
#pragma unroll
      for (int m = 0; m < M; ++m) v.x[m] = bf16_to_f32(ldg_u16_early(p.x + (int64_t)m * p.R + q.r0 + r));
    }
  };
  // ... and stores its B operand row: the tf32 high parts of x*scale in token columns 0..3, the exact
  // remainders in 4..7 (zero for rows past the piece and for absent tokens).  Row r = 8ks + k of the piece goes
  // to k-step ks, pair slot (k mod 4, column n), half k / 4: lane (g, t) then reads its two B values (k-slots
  // t and t+4 of column g) with one 8-byte load.
  auto store_x = [&](const Piece& q, int b, const XRow& xr) {
    const int r = threadIdx.x;
    if (r >= P) return;
    float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < q.nr) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float v = __fmul_rn(xr.x[m], xr.s);  // exact
        hi[m] = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
        lo[m] = __fsub_rn(v, hi[m]);  // exact, at most 8 significant bits
      }
    }
    float* d = xsb + b * P * 8 + ((r >> 3) * 4 + (r & 3)) * 16 + ((r >> 2) & 1);
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      d[2 * n] = hi[n];
      d[2 * n + 8] = lo[n];
    }
  };

  float d[4][4], acc[4][4];
#pragma unroll
  for (int J = 0; J < 4; ++J)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[J][i] = acc[J][i] = 0.f;
  int chain = 0;  // k-steps of this warp (at most, counted per piece) in the current accumulation chain

  // Ring of kA0tBufs pieces: piece j sits in buffer j % kA0tBufs.  Iteration j waits for piece j, passes one
  // barrier (after which every warp is done with piece j-1, whose buffer piece j+2 takes) and issues piece j+2.
  Piece cur;
  cur.cb = (int)(f0 / p.R);
  cur.r0 = f0 - (int64_t)cur.cb * p.R;
  cur.f = f0;
  cur.j = 0;
  fit(cur);
  Piece q1 = next(cur), q2 = cur;
  XRow xr, xr1;  // x of a piece two ahead; in the prologue, of pieces 0 and 1 together
  issue_codes(cur, 0);
  cp_async_commit();
  if (q1.f < f1) issue_codes(q1, 1);
  cp_async_commit();
  load_x(cur, xr);
  if (q1.f < f1) load_x(q1, xr1);
  store_x(cur, 0, xr);
  if (q1.f < f1) store_x(q1, 1, xr1);
  for (int buf = 0; cur.f < f1; buf = (buf + 1 == kA0tBufs) ? 0 : buf + 1) {
    cp_async_wait<1>();  // this thread's copies of piece j have landed
    __syncthreads();     // ... and every thread's, with its B rows; piece j-1 is no longer read
    const int buf2 = (buf + 2) % kA0tBufs;
    q2 = next(q1);
    const bool has2 = q1.f < f1 && q2.f < f1;
    if (has2) {
      issue_codes(q2, buf2);
      load_x(q2, xr);
    }
    cp_async_commit();

    // this warp's k-steps of the piece: slice, slice + 4, ...; rows past the piece hold stale words (finite y)
    // against zero B rows
    const uint32_t* cw = cbuf + (buf * P + 8 * slice + t) * ST;
    const float* xb = xsb + buf * P * 8 + (slice * 4 + t) * 16 + 2 * g;
    const int nks = (cur.nr + 7) >> 3;
#pragma unroll 2
    for (int ks = slice; ks < nks; ks += kA0tSlices, cw += 8 * kA0tSlices * ST, xb += 64 * kA0tSlices) {
      uint32_t sa[4][2], sb[4][2];
      dec.states(cw, sa);           // stored row 8ks + t
      dec.states(cw + 4 * ST, sb);  // stored row 8ks + t + 4
      const float2 bv = *reinterpret_cast<const float2*>(xb);
      const uint32_t b0 = __float_as_uint(bv.x), b1 = __float_as_uint(bv.y);
#pragma unroll
      for (int J = 0; J < 4; ++J)
        mma_tf32(d[J], code_f32<true>(sa[J][0]), code_f32<false>(sa[J][1]), code_f32<true>(sb[J][0]),
                 code_f32<false>(sb[J][1]), b0, b1);
    }
    if (has2) store_x(q2, buf2, xr);  // its buffer's last readers finished before the barrier above
    chain += kPieceSteps;
    if (chain + kPieceSteps > kA0tChainSteps) {
#pragma unroll
      for (int J = 0; J < 4; ++J)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[J][i] += d[J][i];
          d[J][i] = 0.f;
        }
      chain = 0;
    }

    const bool last = q1.f >= f1;
    if (cur.r0 + cur.nr == p.R || last) {  // end of a segment: fold and publish its partial
      float v[4][4];
#pragma unroll
      for (int J = 0; J < 4; ++J)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[J][i] = acc[J][i] + d[J][i];
          v[J][i] += __shfl_xor_sync(0xFFFFFFFFu, v[J][i], 2);  // high part + remainder of the same token
          acc[J][i] = d[J][i] = 0.f;
        }
      chain = 0;
      if (t < 2) {  // lanes t = 0, 1 hold tokens 2t and 2t+1
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int m = 2 * t + e;
          if (m < M) {
#pragma unroll
            for (int J = 0; J < 4; ++J) {
              red[(slice * M + m) * kT + dec.col(J, 0)] = v[J][e];
              red[(slice * M + m) * kT + dec.col(J, 1)] = v[J][2 + e];
            }
          }
        }
      }
      __syncthreads();
      float* slot = p.part + (int64_t)(c + cur.cb) * M * kT;
      for (int i = threadIdx.x; i < M * kT; i += blockDim.x) {
        float sum = red[i];
#pragma unroll
        for (int sl = 1; sl < kA0tSlices; ++sl) sum += red[sl * M * kT + i];
        slot[i] = sum;
      }
      ax0_publish<M, false>(p, pend, is_last, npend, cur.cb, last);
    }
    cur = q1;
    q1 = q2;
  }
  cp_async_wait<0>();
}

template <int K, int L, int M, bool IL>
cudaError_t a0t_launch1(const Ax0Params& p, cudaStream_t st) {
  const size_t smem = a0t_smem<K>(M);
  static PerDevice<cudaError_t> attr_of;  // function attributes are per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const cudaError_t attr_err = attr_of.get(dev, [smem] {
    return cudaFuncSetAttribute(ax0tc_kernel<K, L, M, IL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  }, cudaErrorInvalidDevice);
  if (attr_err != cudaSuccess) return attr_err;
  const cudaError_t e = launch_pdl(ax0tc_kernel<K, L, M, IL>, dim3(p.G), dim3(32 * kA0tWarps), smem, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int K, int L, bool IL>
cudaError_t a0t_launch_m(const Ax0Params& p, int M, cudaStream_t st) {
  switch (M) {
    case 1: return a0t_launch1<K, L, 1, IL>(p, st);
    case 2: return a0t_launch1<K, L, 2, IL>(p, st);
    case 3: return a0t_launch1<K, L, 3, IL>(p, st);
    default: return a0t_launch1<K, L, 4, IL>(p, st);
  }
}

template <int L>
cudaError_t a0t_launch_k(const Ax0Params& p, int M, int k, bool il, cudaStream_t st) {
  if (k == 2) return a0t_launch_m<2, L, false>(p, M, st);
  if (k == 3) return il ? a0t_launch_m<3, L, true>(p, M, st) : a0t_launch_m<3, L, false>(p, M, st);
  return a0t_launch_m<4, L, false>(p, M, st);
}

}  // namespace

cudaError_t launch_matvec_axis0_tc(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                                   int M, int k, int L, int64_t rows, int64_t cols, int interleave, void* workspace,
                                   cudaStream_t st) {
  Ax0Params p{};
  p.codes = codes; p.scales = scales; p.x = x; p.out = out;
  p.nb = (int)(cols / kT);
  p.part = static_cast<float*>(workspace);
  p.counter = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) +
                                          (size_t)(kAx0MaxCtas + p.nb) * (size_t)M * kT * sizeof(float));
  p.R = rows; p.C = cols; p.N = (int64_t)p.nb * rows;
  p.G = ax0_grid(p.N);
  if (L == 16) return a0t_launch_k<16>(p, M, k, interleave != 0, st);
  return a0t_launch_k<12>(p, M, k, interleave != 0, st);
}

}  // namespace trellis
