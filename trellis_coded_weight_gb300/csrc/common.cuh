// common.cuh -- device primitives of the trellis (QTIP 1MAD) decode for sm_103a.
//
// Format and code: "trellis-linear.ts" diff page (mlx-bun 0.2.0 -> 0.4.0),
// header comment and HEADER source (trellis_state, trellis_y, trellis_val,
// trellis_val_rcp).  The state of position t of a T-long block is the L-bit
// window that starts at bit (T-1-t)*k of the block (LSB-first inside
// little-endian uint32 words, wrapping inside the block); the code of state s
// is y = bytesum(s*34038481 + 76625530 mod 2^32) - 510.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace trellis {

constexpr uint32_t kMulA = 34038481u;
constexpr uint32_t kAddB = 76625530u;
constexpr float kD = 147.800537109375f;
constexpr float kRcpD = 1.0f / 147.800537109375f;  // fp32 nearest to 1/d (folded at compile time)
constexpr int kT = 256;                             // positions per block (the only supported T)

// The fp32 pattern 0x4B400000 is 1.5*2^23, whose ulp is 1: adding an integer
// n with |n| < 2^22 to the pattern adds n to the value.  The byte-sum
// instruction adds the four bytes onto this bias, so its result, read as a
// float, is exactly 1.5*2^23 + y.
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kMagic = 12582912.0f;

// 1MAD of a zero-extended L-bit state: bit pattern of the float 1.5*2^23 + y.
__device__ __forceinline__ uint32_t code_magic(uint32_t s) {
  const uint32_t x = s * kMulA + kAddB;
  return __dp4a(x, 0x01010101u, kMagicBits - 510u);
}

// y as an exact float.
__device__ __forceinline__ float code_y(uint32_t s) {
  return __fsub_rn(__uint_as_float(code_magic(s)), kMagic);
}

// y as an integer (the byte sum onto -510), and as an exact float through an
// int-to-float conversion.  The conversion runs on the ALU pipe, the bias
// subtraction of code_magic on the FMA pipe that also carries the 1MAD
// multiply and the byte sum, so kernels bound by that pipe use this form.
__device__ __forceinline__ int code_int(uint32_t s) {
  return (int)__dp4a(s * kMulA + kAddB, 0x01010101u, (uint32_t)-510);
}
__device__ __forceinline__ float2 code_y2_alu(uint32_t s0, uint32_t s1) {
  return make_float2(__int2float_rn(code_int(s0)), __int2float_rn(code_int(s1)));
}

// Correctly rounded y / d: the reciprocal product refined by one residual
// step ("trellis_val_rcp" in the HEADER source).  The pages state, and the
// oracle pins check exhaustively, that this equals the IEEE quotient for
// every y in [-510, 510].
__device__ __forceinline__ float value_rn(float y) {
  const float q = __fmul_rn(y, kRcpD);
  const float e = __fmaf_rn(-q, kD, y);
  return __fmaf_rn(e, kRcpD, q);
}

// fp32 split of 1/d: kRcpHi = kRcpD is the nearest fp32, kRcpLo the nearest
// fp32 to the remainder (1/d in double minus kRcpHi).  fma(y, kRcpHi,
// y * kRcpLo) is the correctly rounded y/d for every y in [-510, 510]: one
// rounding of a 48-bit-accurate product (checked exhaustively against exact
// rational arithmetic by the oracle pin tests).
constexpr float kRcpHi = kRcpD;
constexpr float kRcpLo = (float)(1.0 / 147.800537109375 - (double)(1.0f / 147.800537109375f));

// Correctly rounded (y0/d, y1/d) for exact integer-valued y, packed f32x2.
__device__ __forceinline__ float2 value_rn2(float2 y) {
  return __ffma2_rn(y, make_float2(kRcpHi, kRcpHi), __fmul2_rn(y, make_float2(kRcpLo, kRcpLo)));
}

// Round two floats to bf16 (nearest even) and pack them, a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

__device__ __forceinline__ float f16_to_f32(uint16_t h) {
  float f;
  asm("{ .reg .f16 t; mov.b16 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "h"(h));
  return f;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

// The SwiGLU cast chain of GATEUP_SOURCE ("trellis-linear.ts" diff page) on
// fp32 gate/up sums: each intermediate is rounded to bf16.
__device__ __forceinline__ uint16_t swiglu_chain(float gate, float up) {
  const float g = bf16_to_f32(f32_to_bf16_rn(gate));
  const float u = bf16_to_f32(f32_to_bf16_rn(up));
  const float sig = bf16_to_f32(f32_to_bf16_rn(__fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)))));
  const float silu = bf16_to_f32(f32_to_bf16_rn(__fmul_rn(g, sig)));
  return f32_to_bf16_rn(__fmul_rn(silu, u));
}

// The L-bit window starting at run-relative bit O of the words w[] (w[0]
// holds run bits 0..31).  O is a compile-time constant after unrolling.
template <int L, int NW>
__device__ __forceinline__ uint32_t window_at(const uint32_t (&w)[NW], int O) {
  const int wi = O >> 5, off = O & 31;
  uint32_t v;
  if (off == 0) v = w[wi];
  else if (off + L <= 32) v = w[wi] >> off;
  else v = __funnelshift_r(w[wi], w[wi + 1], off);
  return (off + L == 32) ? v : (v & ((1u << L) - 1u));
}

// States of the N positions t0 .. t0+N-1 of a run.  Position t0+j starts at
// run bit (N-1-j)*K; w[] holds the run's words, aligned so that w[0] bit 0 is
// run bit 0, followed by the spill word.  For L = 16 and K in {2, 4}, windows
// 16 bits apart come from one 32-bit funnel shift: the low half is one state
// and the high half the other.
template <int K, int L, int N = 32, int NW = K + 1>
__device__ __forceinline__ void run_states(const uint32_t (&w)[NW], uint32_t (&s)[N]) {
  constexpr bool kPair = (L == 16) && (K == 2 || K == 4);
  constexpr int kPartner = 16 / K;  // j - kPartner starts 16 bits above j
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int o = (N - 1 - j) * K;
    if (kPair) {
      if ((o & 31) < 16) {
        const uint32_t F = (o & 31) ? __funnelshift_r(w[o >> 5], w[(o >> 5) + 1], o & 31) : w[o >> 5];
        s[j] = F & 0xFFFFu;
        s[j - kPartner] = F >> 16;
      }
    } else {
      s[j] = window_at<L, NW>(w, o);
    }
  }
}

}  // namespace trellis
