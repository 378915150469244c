// mma_tf32.cuh -- the warp-level tensor-core step of the decode-fused matvecs: decoded y (exact in tf32) times
// x (bf16, or a split of x*scale into two tf32 parts) through mma.sync m16n8k8 with fp32 accumulation.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace trellis {

// D += A * B for one m16n8k8 tile.  Lane (g, t) = (lane / 4, lane % 4) holds A rows g and g+8 at k-slots t and
// t+4 (a0 = (g, t), a1 = (g+8, t), a2 = (g, t+4), a3 = (g+8, t+4)), B k-slots t and t+4 of column g, and D rows g
// and g+8 at columns 2t and 2t+1 (d0, d1 for row g; d2, d3 for row g+8).
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// y of state s as fp32 bits (exact): through an int-to-float conversion (ALU pipe) or through the float bias
// 1.5*2^23 and its subtraction (FMA pipe).  The kernels take one A row of a lane each way, which balances the
// two pipes (the window extraction also runs on the ALU pipe).
template <bool ALU>
__device__ __forceinline__ uint32_t code_f32(uint32_t s) {
  return __float_as_uint(ALU ? __int2float_rn(code_int(s)) : code_y(s));
}

}  // namespace trellis
