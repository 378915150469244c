// axis0_windows.cuh -- where a lane of the axis-0 tensor-core kernels finds its windows in one stored row of a
// 256-position column block (matvec_axis0_tc.cu, prefill_axis0_small.cu).  Lane (g, t) of column quarter Q
// stands for the 8 outputs that A rows g and g+8 of the quarter's four 16-row MMA tiles J = 0..3 represent;
// states(row) returns their states (s[J][0] for row g, s[J][1] for row g+8) from the row's staged words, and
// col(J, h) their block positions.  Position p's window starts at block bit (255 - p)*K ("trellis-linear.ts"
// diff page, header comment: the state of position t of a T-long block, wrapping inside the block).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace trellis {

// The L-bit window at bit o of the 64-bit pair (hi:lo), o < 32 a compile-time constant after unrolling.
template <int L>
__device__ __forceinline__ uint32_t window64(uint32_t lo, uint32_t hi, int o) {
  const uint32_t v = (o + L <= 32) ? (lo >> o) : __funnelshift_r(lo, hi, o);
  return (o + L == 32) ? v : (v & ((1u << L) - 1u));
}

// Window layout of one staged row for lane (g, t) of column quarter Q: the states of the 8 outputs that A rows
// g and g+8 of the quarter's four MMA tiles J = 0..3 stand for, s[J][0] for row g and s[J][1] for row g+8, and
// the block position of each (col).  Position p's window starts at block bit (255 - p)*K.
template <int K, int L>
struct A0Windows;

// K = 2: tile J, A row i <-> position 64Q + 16J + i.  The windows of positions p and p+8 are 16 bits apart, so
// one funnel shift (by 14 - 2g, the same for all tiles) from words 15-4Q-J and 16-4Q-J gives both.
template <int L>
struct A0Windows<2, L> {
  int q4, sh, g, Q;
  __device__ A0Windows(int Q_, int g_) : q4(12 - 4 * Q_), sh(14 - 2 * g_), g(g_), Q(Q_) {}
  __device__ __forceinline__ void states(const uint32_t* row, uint32_t (&s)[4][2]) const {
    const uint4 v = *reinterpret_cast<const uint4*>(row + q4);
    const uint32_t w[5] = {v.x, v.y, v.z, v.w, row[(q4 + 4) & 15]};
#pragma unroll
    for (int J = 0; J < 4; ++J) {
      const uint32_t F = __funnelshift_r(w[3 - J], w[4 - J], sh);
      s[J][0] = (L == 16) ? (F >> 16) : ((F >> 16) & ((1u << L) - 1u));
      s[J][1] = F & ((1u << L) - 1u);
    }
  }
  __device__ __forceinline__ int col(int J, int h) const { return 64 * Q + 16 * J + g + 8 * h; }
};

// K = 3: tile J, A row g <-> position P + 2J, row g+8 <-> P + 2J + 1, with P = 64Q + 8g, so the lane owns the
// 8 consecutive positions P..P+7.  Their windows span 37 bits from bit base = 3*(248 - P); two funnel shifts by
// base mod 32 align them, and each window then sits at the compile-time offset 3*(7 - j).  The block is 24
// words; indices wrap inside it.
template <int L>
struct A0Windows<3, L> {
  int i0, i1, i2, sh, g, Q;
  __device__ A0Windows(int Q_, int g_) : g(g_), Q(Q_) {
    const int base = 744 - 192 * Q_ - 24 * g_;
    i0 = base >> 5;
    i1 = i0 + 1 >= 24 ? i0 + 1 - 24 : i0 + 1;
    i2 = i0 + 2 >= 24 ? i0 + 2 - 24 : i0 + 2;
    sh = base & 31;
  }
  __device__ __forceinline__ void states(const uint32_t* row, uint32_t (&s)[4][2]) const {
    const uint32_t r0 = row[i0], r1 = row[i1], r2 = row[i2];
    const uint32_t a = __funnelshift_r(r0, r1, sh), b = __funnelshift_r(r1, r2, sh);
#pragma unroll
    for (int J = 0; J < 4; ++J) {
      s[J][0] = window64<L>(a, b, 21 - 6 * J);  // position P + 2J
      s[J][1] = window64<L>(a, b, 18 - 6 * J);  // position P + 2J + 1
    }
  }
  __device__ __forceinline__ int col(int J, int h) const { return 64 * Q + 8 * g + 2 * J + h; }
};

// K = 4: the same consecutive ownership as K = 3.  Here base = 4*(248 - P) is word aligned (word 31 - 8Q - g),
// and positions P+j and P+j+4 are 16 bits apart: F_j = (w1:w0) >> (12 - 4j) holds P+j in its high half and
// P+j+4 in its low half.
template <int L>
struct A0Windows<4, L> {
  int i0, i1, g, Q;
  __device__ A0Windows(int Q_, int g_) : i0(31 - 8 * Q_ - g_), i1((32 - 8 * Q_ - g_) & 31), g(g_), Q(Q_) {}
  __device__ __forceinline__ void states(const uint32_t* row, uint32_t (&s)[4][2]) const {
    const uint32_t w0 = row[i0], w1 = row[i1];
    constexpr uint32_t mask = (1u << L) - 1u;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t F = (j == 3) ? w0 : __funnelshift_r(w0, w1, 12 - 4 * j);
      hi[j] = (L == 16) ? (F >> 16) : ((F >> 16) & mask);  // position P + j
      lo[j] = F & mask;                                    // position P + j + 4
    }
    s[0][0] = hi[0]; s[0][1] = hi[1];
    s[1][0] = hi[2]; s[1][1] = hi[3];
    s[2][0] = lo[0]; s[2][1] = lo[1];
    s[3][0] = lo[2]; s[3][1] = lo[3];
  }
  __device__ __forceinline__ int col(int J, int h) const { return 64 * Q + 8 * g + 2 * J + h; }
};

}  // namespace trellis
