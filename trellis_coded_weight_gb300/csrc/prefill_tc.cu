// prefill_tc.cu -- prefill GEMM over an axis-1 trellis matrix on the 5th-
// generation tensor cores (tcgen05), any M >= 1 (intended for M > 4).
//
// What is computed ("trellis-tiled-prefill.ts" diff page: tiledTrellisPrefill;
// "trellis-linear.ts": the expand + matmul path of TrellisLinear.forward):
//   out[m][r] = bf16( sum_c e(r,c) * x[m][c] ),
// e(r,c) = bf16( fl32( value(s(r,c)) * scale[r] ) ), value correctly rounded
// -- the expand numerics -- with fp32 accumulation.  The pages decode each
// weight tile into threadgroup memory and run 8x8 SIMD-group MMAs.
//
// GB300 design: a persistent kernel, one CTA per SM, walking output tiles of
// 128 weight rows x BN tokens (tile t -> row tile t % nRT, token tile t / nRT,
// so the CTAs running together share one token tile of x in L2).
//   warp 0      TMA producer: x tiles [BN tokens][64 columns] land in shared
//               memory in the 128-byte swizzled K-major layout.
//   warp 1      allocates 2*BN tensor-memory columns (two accumulators); one
//               lane issues tcgen05.mma (M=128, N=BN, K=16, bf16 -> fp32)
//               four times per 64-column stage and commits each stage back to
//               the ring and each finished tile to the epilogue.
//   warps 2-5   epilogue: tcgen05.ld of a finished accumulator (each warp
//               reads its own 32-lane sub-partition), bf16 conversion and
//               coalesced stores of out[m][r]; the accumulator is released
//               while the MMA already fills the other one.
//   warps 6-21  decoders in two groups of eight, taking alternate stages:
//               each thread decodes a run of 32 positions of one of the
//               tile's 128 weight rows straight into the swizzled A tile
//               (generic-proxy stores, then fence.proxy.async).  The code
//               words of a run are loaded two stages ahead.
// A ring of NS stages (A 16 KB + B BN*128 bytes each) decouples producer,
// decoders and MMA; every mbarrier wait is bounded.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace trellis {

// Device-side error word: set when a bounded wait in a tensor-core kernel
// gives up (read through trellis_device_error in the C ABI).
__device__ int g_device_error = 0;

namespace {

constexpr int kBM = 128;               // weight rows per tile (MMA M)
constexpr int kBK = 64;                // columns per stage (one 128-byte swizzle row of bf16)
constexpr int kATile = kBM * kBK * 2;  // 16 KB
constexpr int kProdWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4, kDecWarp0 = 6;
constexpr int kGroupWarps = 8, kGroups = 2;
constexpr int kThreads = 32 * (kDecWarp0 + kGroups * kGroupWarps);  // 704
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct PrefillParams {
  const uint32_t* codes;
  const uint16_t* scales;
  uint16_t* out;
  int64_t R, C;
  int M, nb;
  int nRT, nTiles;  // row tiles, total tiles
};

template <int BN>
struct Cfg {
  static constexpr int NS = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);  // ring stages
  static constexpr int BTile = BN * kBK * 2;
  static constexpr int Stage = kATile + BTile;
  static constexpr int TmemCols = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
  static constexpr size_t Smem = 1024 + (size_t)NS * Stage + 256;
};

// The words of one run (K words of positions 32q .. 32q+31 plus the spill
// word, which wraps to word 0 for the block's last run).
template <int K>
struct RunWords {
  uint32_t w[K + 1];
  float scale;
};

template <int K>
__device__ __forceinline__ void load_run(RunWords<K>& rw, const uint32_t* __restrict__ blk, int q,
                                         const uint16_t* __restrict__ sc) {
  constexpr int WPB = kT * K / 32;
#pragma unroll
  for (int i = 0; i < K; ++i) rw.w[i] = __ldg(blk + (7 - q) * K + i);
  rw.w[K] = __ldg(blk + ((8 - q) * K) % WPB);
  rw.scale = f16_to_f32(__ldg(sc));
}

// Decode one run into the A tile: bf16(value*scale) in the 128-byte swizzled
// K-major layout, where 16-byte chunk q of row rl sits at chunk q ^ (rl & 7).
template <int K, int L>
__device__ __forceinline__ void decode_run_to_tile(const RunWords<K>& rw, uint8_t* a_tile, int rl, int chunk0) {
  uint32_t s[32];
  run_states<K, L>(rw.w, s);
  const float2 nmagic = make_float2(-kMagic, -kMagic);
  const float2 rcp = make_float2(kRcpD, kRcpD), nd = make_float2(-kD, -kD);
  const float2 sc = make_float2(rw.scale, rw.scale);
  uint32_t packed[16];
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 y = __fadd2_rn(make_float2(__uint_as_float(code_magic(s[j])), __uint_as_float(code_magic(s[j + 1]))),
                                nmagic);
    // correctly rounded y/d by one residual step, then * scale, all per element
    const float2 qv = __fmul2_rn(y, rcp);
    const float2 e = __ffma2_rn(qv, nd, y);  // y - q*d, exact residual
    const float2 v = __ffma2_rn(e, rcp, qv);
    const float2 wv = __fmul2_rn(v, sc);
    packed[j / 2] = pack_bf16x2(wv.x, wv.y);
  }
  uint8_t* row = a_tile + rl * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int chunk = (chunk0 + c) ^ (rl & 7);
    *reinterpret_cast<uint4*>(row + chunk * 16) =
        make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
  }
}

__device__ __forceinline__ void report(int code) { atomicCAS(&g_device_error, 0, code); }

template <int K, int L, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_x, const PrefillParams p) {
  using C_ = Cfg<BN>;
  constexpr int NS = C_::NS;
  constexpr int WPB = kT * K / 32;
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kBM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* a_tiles = smem;                          // NS x 16 KB
  uint8_t* b_tiles = smem + (size_t)NS * kATile;    // NS x BN*128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)NS * C_::Stage);
  uint64_t* full_a = bars;             // decoder group -> MMA (8 warp arrivals)
  uint64_t* full_b = bars + NS;        // TMA -> MMA (1 arrival + tx bytes)
  uint64_t* empty = bars + 2 * NS;     // MMA commit -> producer and decoders
  uint64_t* acc_full = bars + 3 * NS;  // [2] MMA commit -> epilogue
  uint64_t* acc_empty = bars + 3 * NS + 2;  // [2] epilogue warps -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * NS + 4);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int n_local = (p.nTiles - (int)blockIdx.x + G - 1) / G;
  const int nk = (int)(p.C / kBK);
  const int64_t total = (int64_t)n_local * nk;  // stages this CTA runs
  const uint64_t deadline = kWaitNs;  // per wait

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(full_a + s, kGroupWarps);
      tc::mbar_init(full_b + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full + b, 1);
      tc::mbar_init(acc_empty + b, kEpiWarps);
    }
    *fail = 0;
    tc::fence_mbar_init();
  }
  if (warp == kProdWarp && lane == 0) tc::prefetch_tmap(&tmap_x);
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, C_::TmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProdWarp) {
    if (lane == 0) {
      int64_t g = 0;
      int64_t issued = 0;
      for (int lt = 0; lt < n_local && !*fail; ++lt) {
        const int t = (int)blockIdx.x + lt * G;
        const int m0 = (t / p.nRT) * BN;
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int s = (int)(g % NS);
          if (g >= NS && !tc::mbar_wait(empty + s, (uint32_t)((g / NS) & 1) ^ 1u, deadline)) { *fail = 1; break; }
          tc::mbar_arrive_expect_tx(full_b + s, (uint32_t)C_::BTile);
          tc::tma_load_2d(b_tiles + (size_t)s * C_::BTile, &tmap_x, full_b + s, ks * kBK, m0);
          ++issued;
        }
      }
      if (*fail) {  // let copies already in flight land before the CTA exits
        for (int64_t j = (issued > NS ? issued - NS : 0); j < issued; ++j)
          tc::mbar_wait(full_b + j % NS, (uint32_t)((j / NS) & 1), kWaitNs);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t a0 = tc::smem_u32(a_tiles), b0 = tc::smem_u32(b_tiles);
      int64_t g = 0;
      for (int lt = 0; lt < n_local && !*fail; ++lt) {
        const int buf = lt & 1;
        if (lt >= 2 && !tc::mbar_wait(acc_empty + buf, (uint32_t)((lt >> 1) & 1) ^ 1u, deadline)) {
          *fail = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int s = (int)(g % NS);
          const uint32_t ph = (uint32_t)((g / NS) & 1);
          if (!tc::mbar_wait(full_a + s, ph, deadline) || !tc::mbar_wait(full_b + s, ph, deadline)) {
            *fail = 1;
            break;
          }
          tc::fence_after_sync();
          const uint64_t ad = tc::desc_sw128(a0 + s * kATile), bd = tc::desc_sw128(b0 + s * C_::BTile);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // +32 bytes along K per MMA: +2 in the address field
            tc::mma_bf16(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (ks | kk) != 0 ? 1u : 0u);
          tc::mma_commit(empty + s);
        }
        tc::mma_commit(acc_full + buf);
      }
    }
  } else if (warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue ----------------
    const int sp = warp & 3;  // TMEM sub-partition this warp may read
    for (int lt = 0; lt < n_local; ++lt) {
      const int buf = lt & 1;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(acc_full + buf, (uint32_t)((lt >> 1) & 1), deadline));
      tc::fence_after_sync();
      if (!ok) { *fail = 1; break; }
      const int t = (int)blockIdx.x + lt * G;
      const int64_t row = (int64_t)(t % p.nRT) * kBM + 32 * sp + lane;
      const int m0 = (t / p.nRT) * BN;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(buf * BN + c0), v);
        tc::tmem_ld_wait();
        if (row < p.R) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int m = m0 + c0 + i;
            if (m < p.M) {
              uint16_t o;
              asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(o) : "f"(__uint_as_float(v[i])));
              p.out[(int64_t)m * p.R + row] = o;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty + buf);
    }
  } else {
    // ---------------- decoders ----------------
    const int dw = warp - kDecWarp0;       // 0..15
    const int grp = dw / kGroupWarps;      // stages g with g % 2 == grp
    const int gw = dw % kGroupWarps;
    const int rl = (gw & 3) * 32 + lane;   // tile row of this thread
    const int h = gw >> 2;                 // which 32-column half of a stage
    auto fetch = [&](RunWords<K>& rw, int64_t g) {
      if (g >= total) return;
      const int lt = (int)(g / nk), ks = (int)(g % nk);
      const int t = (int)blockIdx.x + lt * G;
      int64_t r = (int64_t)(t % p.nRT) * kBM + rl;
      if (r >= p.R) r = p.R - 1;  // rows past the end decode row R-1 and are never stored
      const uint32_t* blk = p.codes + (r * p.nb + (ks >> 2)) * WPB;
      load_run<K>(rw, blk, 2 * (ks & 3) + h, p.scales + r);
    };
    auto process = [&](const RunWords<K>& rw, int64_t g) -> bool {
      const int s = (int)(g % NS);
      if (g >= NS && !tc::mbar_wait(empty + s, (uint32_t)((g / NS) & 1) ^ 1u, deadline)) return false;
      decode_run_to_tile<K, L>(rw, a_tiles + (size_t)s * kATile, rl, 4 * h);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(full_a + s);
      return true;
    };
    RunWords<K> ra, rb;
    int64_t g = grp;
    fetch(ra, g);
    fetch(rb, g + 2);
    while (g < total) {
      if (!process(ra, g)) { *fail = 1; break; }
      fetch(ra, g + 4);
      g += 2;
      if (g >= total) break;
      if (!process(rb, g)) { *fail = 1; break; }
      fetch(rb, g + 4);
      g += 2;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *fail) report(1);
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C_::TmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 148;
  return n;
}

template <int K, int L, int BN>
cudaError_t prefill_launch(PrefillParams p, const uint16_t* x, cudaStream_t st) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)p.C, (cuuint64_t)p.M};
  const cuuint64_t strides[1] = {(cuuint64_t)p.C * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)BN};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  auto kern = prefill_kernel<K, L, BN>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<BN>::Smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  p.nRT = (int)((p.R + kBM - 1) / kBM);
  p.nTiles = p.nRT * ((p.M + BN - 1) / BN);
  const int sms = sm_count();
  const int grid = p.nTiles < sms ? p.nTiles : sms;
  kern<<<grid, kThreads, Cfg<BN>::Smem, st>>>(map, p);
  return cudaGetLastError();
}

template <int K, int L>
cudaError_t prefill_bn(const PrefillParams& p, const uint16_t* x, cudaStream_t st) {
  if (p.M <= 32) return prefill_launch<K, L, 32>(p, x, st);
  if (p.M <= 64) return prefill_launch<K, L, 64>(p, x, st);
  if (p.M <= 128) return prefill_launch<K, L, 128>(p, x, st);
  return prefill_launch<K, L, 256>(p, x, st);
}

}  // namespace

cudaError_t launch_gemm_prefill(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                                int M, int k, int L, int64_t rows, int64_t cols, cudaStream_t st) {
  PrefillParams p{};
  p.codes = codes; p.scales = scales; p.out = out;
  p.R = rows; p.C = cols; p.M = M; p.nb = (int)(cols / kT);
  if (L == 16) {
    if (k == 2) return prefill_bn<2, 16>(p, x, st);
    if (k == 3) return prefill_bn<3, 16>(p, x, st);
    return prefill_bn<4, 16>(p, x, st);
  }
  if (k == 2) return prefill_bn<2, 12>(p, x, st);
  if (k == 3) return prefill_bn<3, 12>(p, x, st);
  return prefill_bn<4, 12>(p, x, st);
}

// Read (and optionally clear) the device error word.
int read_device_error(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (reset && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace trellis
