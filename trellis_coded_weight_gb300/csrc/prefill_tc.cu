// prefill_tc.cu -- prefill GEMM over a trellis matrix (axis 1, and the
// stored-transposed axis 0) on the 5th-generation tensor cores (tcgen05),
// any M >= 1 (intended for M > 4).
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
//   warp 0      TMA producer: x tiles [BN tokens][BK columns] land in shared
//               memory in the swizzled K-major layout (128-byte swizzle for
//               BK = 64, 64-byte swizzle for BK = 32).
//   warp 1      allocates the accumulators in tensor memory; one lane issues
//               tcgen05.mma (M=128, N<=256, K=16, bf16 -> fp32) for every
//               16 columns of a stage and every 256-token half of the tile,
//               commits each stage back to the ring and each finished tile
//               to the epilogue.
//   warps 2-5   epilogue: tcgen05.ld of a finished accumulator (each warp
//               reads its own 32-lane sub-partition), bf16 conversion and
//               coalesced stores of out[m][r].  With two accumulators (BN <=
//               256) the epilogue of one tile overlaps the next tile's MMAs.
//   warps 6-21  decoders in groups that take turns on the ring's stages
//               (axis 1: on half blocks of 128 columns, each thread loading
//               its row's half block once with 16-byte loads):
//               each thread decodes a run of 32 positions of one of the
//               tile's 128 weight rows straight into the swizzled A tile
//               (generic-proxy stores, then fence.proxy.async).  The code
//               words of the next turn load while the current turn decodes.
// Tile shapes: BN = 512 tokens for M > 256 (a 512-column accumulator, so each
// decoded weight feeds 512 tokens -- decoding, not the tensor core, is the
// costly part of this GEMM), else the smallest of 32..256 that covers M (on axis 1 128 rather than 64).
// Axis 0 (stored W^T, coded along the output features;
// "trellis-splitk-prefill.ts" diff page): the A tile is 128 output features
// x BK stored rows.  A decoder warp decodes a run of 32 features along each of
// 32 stored rows (the coding direction) and stores the weights transposed
// into the K-major A tile with stmatrix .trans (decode_runs_transposed).
// With fewer output tiles than SMs, a thread-block cluster of S CTAs splits
// each tile's reduction and sums the partial accumulators through
// distributed shared memory (epilogue, split reduction); with more, the full
// waves run unsplit and the leftover tiles run split in a second launch.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "devcache.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace trellis {

// Device-side error word: set when a bounded wait in a tensor-core kernel
// gives up (read through trellis_device_error in the C ABI).
__device__ int g_device_error = 0;

namespace {

constexpr int kBM = 128;  // weight rows per tile (MMA M)
constexpr int kProdWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4, kDecWarp0 = 6, kDecWarps = 16;
constexpr int kThreads = 32 * (kDecWarp0 + kDecWarps);  // 704
constexpr uint64_t kWaitNs = 2000000000ull;  // default limit per wait: 2 s, far beyond any legitimate wait
// Waits for work already issued (TMA copies in flight, committed MMAs) before a CTA exits after a failure
// always use this limit: those operations finish by themselves, and the CTA must not leave before they do.
constexpr uint64_t kDrainNs = 2000000000ull;
// The limit given to launches (host side); a diagnostic setter changes it for tests of the error path.
std::atomic<uint64_t> g_wait_ns{kWaitNs};


struct PrefillParams {
  const uint32_t* codes;
  const uint16_t* scales;
  uint16_t* out;
  int64_t R, C;     // stored rows and coded columns
  int64_t nOut;     // output features: R for axis 1, C for axis 0
  int64_t Kd;       // reduction length: C for axis 1, R for axis 0
  int M, nb;
  int nRT, nTiles;  // output-feature tiles, total tiles
  int tma_out;      // 1: out written by TMA tensor stores (nOut % 8 == 0)
  int S;            // axis 0: CTAs (a cluster) splitting each tile's reduction; 1 = no split
  int t0;           // first tile of this launch: it runs tiles t0 .. t0 + nTiles - 1
  uint64_t wait_ns; // limit of each pipeline wait (%globaltimer ns); a wait that runs out sets the error word
};

constexpr int kMaxChunks = 16;  // 32-column chunks of the widest accumulator (BN = 512)
// Split reduction slots (in the owner's stage ring): 128 rows x 32 fp32, rows padded to 144 bytes so that
// the owner's 16-byte row reads of a warp spread over the banks.
constexpr int kSlotRow = 144;
constexpr int kSlotBytes = kBM * kSlotRow;
constexpr int kMaxSplit = 8;  // the plan's largest cluster

// AX0: axis-0 kernel (reserves the split reduction's chunk buffer).
template <int BN, int BK, bool AX0 = false>
struct Cfg {
  static constexpr int NACC = 2 * BN <= 512 ? 2 : 1;  // accumulators in tensor memory
  static constexpr int NMMA = BN > 256 ? 256 : BN;    // MMA N
  static constexpr int NH = BN / NMMA;                 // MMAs along N per 16 columns
  static constexpr int ATile = kBM * BK * 2;
  static constexpr int BTile = BN * BK * 2;
  static constexpr int Stage = ATile + BTile;
  static constexpr int EpiBytes = kEpiWarps * 2 * 32 * 32 * 2;  // per warp: two 32x32 bf16 sub-tiles
  static constexpr int NS0 = (220 * 1024 - EpiBytes) / Stage;
  static constexpr int NS = NS0 > 8 ? 8 : NS0;         // ring stages
  static constexpr int TmemCols = NACC * BN < 32 ? 32 : NACC * BN;
  static constexpr int RunsPerRow = BK / 32;            // runs of 32 positions per row and stage
  static constexpr int GroupWarps = 4 * RunsPerRow;     // decoder warps that fill one stage
  static constexpr int Groups = kDecWarps / GroupWarps;
  static constexpr uint32_t SBO = 8u * BK * 2u;         // bytes between 8-row groups
  static constexpr uint32_t SwMode = BK == 64 ? 2u : 4u;  // descriptor swizzle: 128B or 64B
  static constexpr CUtensorMapSwizzle TmaSw = BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr size_t Smem = 1024 + (size_t)NS * Stage + EpiBytes + 1024;
  // axis 0 split: the slots of every sender of the largest cluster fit in the idle stage ring
  static_assert(!AX0 || kMaxSplit * kSlotBytes <= NS * Stage, "split reduction slots exceed the stage ring");
  static_assert(BK == 64 || BK == 32, "stage width");
  static_assert(NS >= 2, "ring too small");
  // a decoder group's consecutive stages are Groups apart: within one lap of the ring, so that an
  // mbarrier parity never stands for a phase two laps old
  static_assert(Groups <= NS, "decoder groups must not outnumber the ring's stages");
};

// The words of one run (K words of positions 32q .. 32q+31 plus the spill
// word, which wraps to word 0 for the block's last run) and the row scale, kept
// as its fp16 bits so that the scale's load is waited for only where it is used.
template <int K>
struct RunWords {
  uint32_t w[K + 1];
  uint16_t scale;
};

template <int K>
__device__ __forceinline__ void load_run(RunWords<K>& rw, const uint32_t* __restrict__ blk, int q,
                                         const uint16_t* __restrict__ sc) {
  constexpr int WPB = kT * K / 32;
#pragma unroll
  for (int i = 0; i < K; ++i) rw.w[i] = __ldg(blk + (7 - q) * K + i);
  rw.w[K] = __ldg(blk + ((8 - q) * K) % WPB);
  rw.scale = __ldg(sc);
}

// Decode one run into the A tile as bf16(value*scale): 16-byte chunk c of the
// row goes to chunk position c ^ sw, the swizzle of the row (row & 7 for the
// 128-byte pattern, (row >> 1) & 3 for the 64-byte one).
template <int K, int L>
__device__ __forceinline__ void decode_run_to_tile(const RunWords<K>& rw, uint8_t* row, int sw, int chunk0) {
  uint32_t s[32];
  run_states<K, L>(rw.w, s);
  const float2 nmagic = make_float2(-kMagic, -kMagic);
  const float scale = f16_to_f32(rw.scale);
  const float2 sc = make_float2(scale, scale);
  uint32_t packed[16];
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 y = __fadd2_rn(make_float2(__uint_as_float(code_magic(s[j])), __uint_as_float(code_magic(s[j + 1]))),
                                nmagic);
    const float2 v = value_rn2(y);  // correctly rounded y/d
    const float2 wv = __fmul2_rn(v, sc);
    packed[j / 2] = pack_bf16x2(wv.x, wv.y);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(row + (((chunk0 + c) ^ sw) << 4)) =
        make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
}

// Axis 0: one warp decodes run q (32 output features) of 32 consecutive stored
// rows (K positions 8*kc0 .. 8*kc0+31) and stores the weights transposed into
// the K-major A tile with stmatrix .trans.  In each 8x8 block of that store,
// lane t holds stored row t/4 and the feature pair 2(t%4), 2(t%4)+1, so lane t
// decodes, for each of its four rows 8*kc0 + 8n + t/4, the features
// 8i + 2(t%4) + {0,1} (i = 0..3).  Its run words are first shifted left by
// 2(t%4)*K bits, which puts all eight windows at compile-time offsets.  Lane t
// gives the address of A row t (feature t of the run) for K block n.
template <int K, int L, int BK>
__device__ __forceinline__ void decode_runs_transposed(const RunWords<K> (&rw)[4], uint8_t* a, int kc0, int lane) {
  constexpr int RowBytes = BK * 2;
  const int sh = 2 * (lane & 3) * K;  // < 32 for K <= 5
  const float2 nmagic = make_float2(-kMagic, -kMagic);
  const int swz = BK == 64 ? (lane & 7) : ((lane >> 1) & 3);  // swizzle of A row t (runs start at multiples of 32)
  const uint32_t row_addr = tc::smem_u32(a + lane * RowBytes);
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    uint32_t w[K + 1];
    w[0] = rw[n].w[0] << sh;
#pragma unroll
    for (int i = 1; i <= K; ++i) w[i] = __funnelshift_l(rw[n].w[i - 1], rw[n].w[i], sh);
    const float scale = f16_to_f32(rw[n].scale);
    const float2 sc = make_float2(scale, scale);
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // features 8i + 2(t%4) (window at (31-8i)K after the shift) and the next
      const uint32_t s0 = window_at<L, K + 1>(w, (31 - 8 * i) * K);
      const uint32_t s1 = window_at<L, K + 1>(w, (30 - 8 * i) * K);
      const float2 y = __fadd2_rn(make_float2(__uint_as_float(code_magic(s0)), __uint_as_float(code_magic(s1))), nmagic);
      const float2 wv = __fmul2_rn(value_rn2(y), sc);
      pk[i] = pack_bf16x2(wv.x, wv.y);
    }
    const uint32_t addr = row_addr + ((uint32_t)((kc0 + n) ^ swz) << 4);
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                 : "memory");
  }
}

__device__ __forceinline__ void report(int code) { atomicCAS(&g_device_error, 0, code); }

// Axis 1: the K order of a tile's nk stages.  Half blocks of 128 columns
// (SPH stages each) go to the NG decoder groups in turn; within a round of NG
// half blocks the stages interleave the groups (stage = round base + r*NG +
// group, r = the run index of the half block), so a decoder thread loads a
// half block once and every group's next stage is at most NG stages after
// its last -- never a full lap of the stage ring ahead of the MMAs.  The
// half blocks past the last full round go stage by stage to the groups in
// turn.  Returns the first column of stage ks.
template <int SPH, int NG, int BK>
__device__ __forceinline__ int ax1_stage_col(int ks, int nk) {
  const int full = (nk / SPH / NG) * NG * SPH;
  if (ks < full) {
    const int T = ks / (NG * SPH), rem = ks % (NG * SPH);
    return (T * NG + rem % NG) * 128 + (rem / NG) * BK;
  }
  return (full / SPH + (ks - full) / SPH) * 128 + ((ks - full) % SPH) * BK;
}

template <int K, int L, int BN, int BK, int AX>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_out,
                   const PrefillParams p) {
  using C_ = Cfg<BN, BK, AX == 0>;
  constexpr int NS = C_::NS, NACC = C_::NACC, NMMA = C_::NMMA, NH = C_::NH;
  constexpr int WPB = kT * K / 32;
  constexpr int RowBytes = BK * 2;
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kBM, NMMA);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* a_tiles = smem;                                // NS x ATile
  uint8_t* b_tiles = smem + (size_t)NS * C_::ATile;       // NS x BTile
  uint8_t* epi_stage = smem + (size_t)NS * C_::Stage;     // kEpiWarps x 2 x [32 tokens][32 rows] bf16
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + C_::EpiBytes);
  uint64_t* full_a = bars;                 // decoder group -> MMA
  uint64_t* full_b = bars + NS;            // TMA -> MMA (1 arrival + tx bytes)
  uint64_t* empty = bars + 2 * NS;         // MMA commit -> producer and decoders
  uint64_t* acc_full = bars + 3 * NS;      // [NACC] MMA commit -> epilogue
  uint64_t* acc_empty = bars + 3 * NS + 2; // [NACC] epilogue warps -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * NS + 4);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* ready = bars + 3 * NS + 5;                  // [kMaxChunks] split: partials of a round -> its owner
  uint64_t* done = bars + 3 * NS + 5 + kMaxChunks;      // [kMaxChunks] split: the owners have read a round
  uint64_t* ringfree = bars + 3 * NS + 5 + 2 * kMaxChunks;  // split: every other CTA's MMAs are done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Without a split a CTA walks tiles cid, cid + G, ... over all nk stages.  With a split (axis 0), the S
  // CTAs of a cluster share one tile and CTA `rank` runs stages [kbeg, kbeg + kcnt) of its reduction.
  const bool split = AX == 0 && p.S > 1;
  const int S = split ? p.S : 1;
  const int G = gridDim.x / S;
  const int cid = (int)blockIdx.x / S, rank = (int)blockIdx.x % S;
  const int n_local = (p.nTiles - cid + G - 1) / G;
  const int nk = (int)((p.Kd + BK - 1) / BK);  // the last stage may run past Kd: TMA fills zeros
  const int kbeg = (int)((int64_t)rank * nk / S);
  const int kcnt = (int)((int64_t)(rank + 1) * nk / S) - kbeg;
  const int64_t total = (int64_t)n_local * kcnt;  // stages this CTA runs

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(full_a + s, C_::GroupWarps);
      tc::mbar_init(full_b + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < NACC; ++b) {
      tc::mbar_init(acc_full + b, 1);
      tc::mbar_init(acc_empty + b, kEpiWarps);
    }
    if (split) {
      // ready[rd]: the owner's expect_tx arrival (plus the senders' bytes); done[rd]: one arrival per
      // epilogue warp of every owner of round rd this CTA sent to; ringfree: one from every other CTA
      constexpr int NCH = BN / 32;
      for (int rd = 0; rd < kMaxChunks; ++rd) {
        const int nown = NCH - rd * S < S ? NCH - rd * S : S;
        const int others = nown > 0 ? nown - (rank < nown ? 1 : 0) : 0;
        tc::mbar_init(ready + rd, 1);
        tc::mbar_init(done + rd, others > 0 ? kEpiWarps * others : 1);
      }
      tc::mbar_init(ringfree, S - 1);
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
  if (split) tc::cluster_sync_all();  // every CTA's barriers exist before any remote arrival
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProdWarp) {
    if (lane == 0) {
      int64_t g = 0, issued = 0;
      for (int lt = 0; lt < n_local && !*fail; ++lt) {
        const int t = p.t0 + cid + lt * G;
        const int m0 = (t / p.nRT) * BN;
        for (int ks = 0; ks < kcnt; ++ks, ++g) {
          const int s = (int)(g % NS);
          if (g >= NS && !tc::mbar_wait(empty + s, (uint32_t)((g / NS) & 1) ^ 1u, p.wait_ns)) { *fail = 1; break; }
          tc::mbar_arrive_expect_tx(full_b + s, (uint32_t)C_::BTile);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tc::tma_load_2d(b_tiles + (size_t)s * C_::BTile + (size_t)h * NMMA * RowBytes, &tmap_x, full_b + s,
                            AX == 1 ? ax1_stage_col<128 / BK, C_::Groups, BK>(ks, nk) : (kbeg + ks) * BK,
                            m0 + h * NMMA);
          ++issued;
        }
      }
      // every copy issued has landed before the CTA exits (the MMA warp waited for all but the last NS of
      // them; after a failure elsewhere it may not have waited for those)
      for (int64_t j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        tc::mbar_wait(full_b + j % NS, (uint32_t)((j / NS) & 1), kDrainNs);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t a0 = tc::smem_u32(a_tiles), b0 = tc::smem_u32(b_tiles);
      int64_t g = 0, last = -1;  // last: the latest stage whose MMAs were committed
      for (int lt = 0; lt < n_local && !*fail; ++lt) {
        const int buf = lt % NACC, use = lt / NACC;
        if (use >= 1 && !tc::mbar_wait(acc_empty + buf, (uint32_t)((use - 1) & 1), p.wait_ns)) { *fail = 1; break; }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        bool ok = true;
        for (int ks = 0; ks < kcnt; ++ks, ++g) {
          const int s = (int)(g % NS);
          const uint32_t ph = (uint32_t)((g / NS) & 1);
          if (!tc::mbar_wait(full_a + s, ph, p.wait_ns) || !tc::mbar_wait(full_b + s, ph, p.wait_ns)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t ad = tc::desc_kmajor(a0 + s * C_::ATile, C_::SBO, C_::SwMode);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const uint64_t bd = tc::desc_kmajor(b0 + s * C_::BTile + h * NMMA * RowBytes, C_::SBO, C_::SwMode);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes along K per MMA: +2 in the address field
              tc::mma_bf16(d + h * NMMA, ad + 2 * kk, bd + 2 * kk, kIdesc, (ks | kk) != 0 ? 1u : 0u);
          }
          tc::mma_commit(empty + s);
          last = g;
        }
        if (!ok) { *fail = 1; break; }  // no commit without MMAs behind it
        tc::mma_commit(acc_full + buf);
      }
      // the MMAs issued have finished (their last commit arrived) before this CTA frees its tensor memory
      // and exits: normally the epilogue waited for them, but not if one of its waits ran out
      if (last >= 0) tc::mbar_wait(empty + last % NS, (uint32_t)((last / NS) & 1), kDrainNs);
    }
  } else if (warp < kEpiWarp0 + kEpiWarps && split) {
    // ---------------- epilogue, split reduction (axis 0) ----------------
    // The cluster's S CTAs hold partial accumulators of one tile.  The tile's
    // 32-column chunks go round by round to owners: in round rd, chunk
    // rd*S + q belongs to CTA q.  Every CTA reads each chunk of the round
    // from tensor memory; a non-owner pushes its fp32 rows with st.async
    // into slot [its rank] of the owner's stage ring (idle once the owner's
    // MMAs are done), completing bytes on the owner's ready[rd]; the owner
    // sums the S partials in rank order (its own from registers), stores
    // bf16 and tells every sender (done[rd]) that the slots are free again.
    // No CTA writes into another's ring before that CTA's MMAs are done
    // (ringfree).  All barriers are single-use and every wait is bounded;
    // after a failure an owner still waits (with the drain limit) for the
    // bytes it was promised, so nothing lands in a CTA that has left.
    const int sp = warp & 3;
    const int t = p.t0 + cid;
    const int64_t row = (int64_t)(t % p.nRT) * kBM + 32 * sp + lane;
    const int m0 = (t / p.nRT) * BN;
    constexpr int NCH = BN / 32;
    constexpr uint32_t kRoundBytes = kBM * 32 * 4;  // one sender's rows of one chunk
    const int rounds = (NCH + S - 1) / S;
    auto owners = [&](int rd) { return NCH - rd * S < S ? NCH - rd * S : S; };  // ranks 0 .. owners-1
    // the four epilogue warps take every branch together (named barrier 1, an AND over their waits)
    auto all_ok = [&](bool v) { return tc::bar_and(v, 1, kEpiWarps * 32); };
    int invited = -1;     // a round whose partials the others may be sending to this owner, not yet received
    int registered = -1;  // the last round whose bytes this owner has announced on ready[]
    bool ok = all_ok(tc::mbar_wait(acc_full, 0u, p.wait_ns));
    tc::fence_after_sync();
    if (ok) {
      if (sp == 0 && lane == 0)
        for (int r = 0; r < S; ++r)
          if (r != rank) tc::mbar_arrive_cluster(ringfree, (uint32_t)r);
      if (rank < owners(0)) invited = 0;
      ok = all_ok(tc::mbar_wait_cluster(ringfree, 0u, p.wait_ns));
    }
    for (int rd = 0; rd < rounds && ok; ++rd) {
      // every round before the last has S owners: all of them got this CTA's partials of that round
      if (rd > 0 && !(ok = all_ok(tc::mbar_wait_cluster(done + rd - 1, 0u, p.wait_ns)))) break;
      const bool owner = rank < owners(rd);
      if (owner) {
        if (sp == 0 && lane == 0) tc::mbar_arrive_expect_tx(ready + rd, (uint32_t)(S - 1) * kRoundBytes);
        registered = rd;
      }
      for (int q = 0; q < owners(rd); ++q) {  // this CTA's partials of the other owners' chunks
        if (q == rank) continue;
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(32 * (rd * S + q)), v);
        tc::tmem_ld_wait();
        const uint32_t dst =
            tc::mapa_shared(a_tiles + (size_t)rank * kSlotBytes + (32 * sp + lane) * kSlotRow, (uint32_t)q);
        const uint32_t bar = tc::mapa_shared(ready + rd, (uint32_t)q);
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4)
          tc::st_async_v4(dst + 16 * k4, __uint_as_float(v[4 * k4]), __uint_as_float(v[4 * k4 + 1]),
                          __uint_as_float(v[4 * k4 + 2]), __uint_as_float(v[4 * k4 + 3]), bar);
      }
      if (!owner) continue;
      if (!(ok = all_ok(tc::mbar_wait_cluster(ready + rd, 0u, p.wait_ns)))) break;
      invited = -1;
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0.f;
      for (int r = 0; r < S; ++r) {  // rank order: the sum does not depend on arrival order
        if (r == rank) {             // this CTA's own partial, straight from tensor memory
          uint32_t v[32];
          tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(32 * (rd * S + rank)), v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] += __uint_as_float(v[j]);
        } else {
          const float4* src =
              reinterpret_cast<const float4*>(a_tiles + (size_t)r * kSlotBytes + (32 * sp + lane) * kSlotRow);
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 f = src[k4];
            acc[4 * k4] += f.x; acc[4 * k4 + 1] += f.y; acc[4 * k4 + 2] += f.z; acc[4 * k4 + 3] += f.w;
          }
        }
      }
      if (row < p.nOut) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int m = m0 + 32 * (rd * S + rank) + j;
          if (m < p.M) {
            uint16_t o;
            asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(o) : "f"(acc[j]));
            p.out[(int64_t)m * p.nOut + row] = o;
          }
        }
      }
      tc::fence_acq_rel_cluster();  // the slot reads above complete before the senders may refill them
      __syncwarp();
      if (lane == 0)
        for (int r = 0; r < S; ++r)
          if (r != rank) tc::mbar_arrive_cluster(done + rd, (uint32_t)r);
      if (rd + 1 < rounds && rank < owners(rd + 1)) invited = rd + 1;
    }
    // after a failure: partials the others may be sending this owner land before the CTA may leave (the
    // wait ends at once if they arrived, after the drain limit if no sender got that far)
    if (invited >= 0) {
      if (registered != invited && sp == 0 && lane == 0)
        tc::mbar_arrive_expect_tx(ready + invited, (uint32_t)(S - 1) * kRoundBytes);
      tc::mbar_wait_cluster(ready + invited, 0u, kDrainNs);
    }
    if (!ok) *fail = 1;
  } else if (warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue ----------------
    const int sp = warp & 3;  // TMEM sub-partition this warp may read
    int ec = 0;               // staging buffers alternate per stored chunk
    for (int lt = 0; lt < n_local; ++lt) {
      const int buf = lt % NACC, use = lt / NACC;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(acc_full + buf, (uint32_t)(use & 1), p.wait_ns));
      tc::fence_after_sync();
      if (!ok) { *fail = 1; break; }
      const int t = p.t0 + cid + lt * G;
      const int64_t rbase = (int64_t)(t % p.nRT) * kBM + 32 * sp;  // first row of this warp's 32
      const int64_t row = rbase + lane;
      const int m0 = (t / p.nRT) * BN;
      uint16_t* my_stage = reinterpret_cast<uint16_t*>(epi_stage) + (size_t)(warp - kEpiWarp0) * 2 * 32 * 32;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(buf * BN + c0), v);
        tc::tmem_ld_wait();
        if (p.tma_out) {
          // stage [32 tokens][32 rows] bf16, then one lane stores the box with TMA
          uint16_t* st = my_stage + (ec++ & 1) * 32 * 32;
          if (lane == 0) tc::bulk_wait_read<1>();  // the previous use of this buffer has been read
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            uint16_t o;
            asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(o) : "f"(__uint_as_float(v[i])));
            st[i * 32 + lane] = o;
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && m0 + c0 < p.M && rbase < p.nOut) {
            tc::tma_store_2d(&tmap_out, st, (int)rbase, m0 + c0);
            tc::bulk_commit();
          }
        } else if (row < p.nOut) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int m = m0 + c0 + i;
            if (m < p.M) {
              uint16_t o;
              asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(o) : "f"(__uint_as_float(v[i])));
              p.out[(int64_t)m * p.nOut + row] = o;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty + buf);
    }
    if (lane == 0) tc::bulk_wait<0>();  // all tensor stores of this warp complete before exit
    __syncwarp();
  } else {
    // ---------------- decoders ----------------
    constexpr int GW = C_::GroupWarps, NG = C_::Groups;
    const int dw = warp - kDecWarp0;       // 0..15
    const int grp = dw / GW;               // this group fills stages g with g % NG == grp
    const int gw = dw % GW;
    const int rl = (gw & 3) * 32 + lane;   // tile row of this thread
    const int h = gw >> 2;                 // which run of the stage
    const int sw = BK == 64 ? (rl & 7) : ((rl >> 1) & 3);
    if constexpr (AX == 0) {
      // Row direction: warp gw of the group takes run q of the tile's 128 output features for 32 stored
      // rows of the stage (K positions kr0 .. kr0+31); each lane decodes two adjacent features of four of
      // those rows, and the warp stores them transposed (decode_runs_transposed).  The run words and
      // row scales are requested before the wait for the stage's ring slot, which hides their latency.
      const int q = gw & 3;                  // run of the tile's features: 32q .. 32q+31
      const int kr0 = (gw >> 2) * 32;        // first stored row of the warp in the stage
      const int ntot = (int)total;           // stages of this CTA (n_local * kcnt, far below 2^31)
      int lt = grp / kcnt, ks = grp % kcnt;  // tile and stage of g, advanced incrementally
      for (int g = grp; g < ntot; g += NG) {
        const int s = g % NS;
        RunWords<K> rw[4];
        {
          const int tb = (p.t0 + cid + lt * G) % p.nRT;  // 128-feature tile: block tb >> 1, half tb & 1
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            int64_t r = (int64_t)(kbeg + ks) * BK + kr0 + 8 * n + (lane >> 2);
            if (r >= p.R) r = p.R - 1;  // past the reduction's end the x tile is zero
            load_run<K>(rw[n], p.codes + (r * p.nb + (tb >> 1)) * WPB, 4 * (tb & 1) + q, p.scales + r);
          }
        }
        // warp-uniform outcome: the transposing store below is a whole-warp instruction
        if (g >= NS && !__all_sync(0xffffffffu, tc::mbar_wait(empty + s, (uint32_t)((g / NS) & 1) ^ 1u, p.wait_ns))) {
          *fail = 1;
          break;
        }
        decode_runs_transposed<K, L, BK>(rw, a_tiles + (size_t)s * C_::ATile + 32 * q * RowBytes, kr0 >> 3, lane);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(full_a + s);
        ks += NG;
        while (ks >= kcnt) { ks -= kcnt; ++lt; }
      }
    } else {
      // Stage order of ax1_stage_col: a turn of this group is a half block of
      // a full round (SPH stages, NG apart) or one stage past the last full
      // round.  Each thread loads its row's half block once per turn with
      // 16-byte loads, a turn ahead, and decodes its run of each stage from
      // registers.  Words [4K, 8K) of a block hold runs 3..0 (positions
      // 0..127) with the spill word 0; words [0, 4K) hold runs 7..4 with the
      // spill word 4K.
      constexpr int SPH = 128 / BK;  // stages per half block
      constexpr int RPR = C_::RunsPerRow;
      static_assert(NG <= NS, "a group's consecutive stages must stay within one lap of the ring");
      const int F = nk / SPH / NG, full = F * NG * SPH;
      const int tail = nk - full > grp ? (nk - full - grp + NG - 1) / NG : 0;  // this group's stages past the rounds
      const int per_tile = F + tail;
      const int nturn = n_local * per_tile;  // turns of this group (a few thousand at most)
      struct HalfWords {
        uint32_t w[4 * K + 1];
        uint16_t scale;  // fp16 bits, converted where used
      };
      // A turn cursor (tile lt, turn v of the tile), advanced without division.
      struct Cursor {
        int lt, v;
      };
      auto advance = [&](Cursor& c) {
        if (++c.v == per_tile) { c.v = 0; ++c.lt; }
      };
      // turn v of a tile: half block hbk and first stage ks0 (full turns: SPH stages NG apart; tail: one
      // stage of run r0)
      auto turn = [&](int v, int& hbk, int& ks0, int& r0) -> bool {
        if (v < F) {
          hbk = v * NG + grp; ks0 = v * NG * SPH + grp; r0 = -1;
          return true;
        }
        ks0 = full + grp + (v - F) * NG;
        hbk = F * NG + (ks0 - full) / SPH; r0 = (ks0 - full) % SPH;
        return false;
      };
      auto fetch = [&](HalfWords& hw, const Cursor& c) {
        if (c.lt >= n_local || c.v >= per_tile) return;  // past the last turn (or a group without turns)
        int hbk, ks0, r0;
        turn(c.v, hbk, ks0, r0);
        const int t = p.t0 + cid + c.lt * G;
        int64_t r = (int64_t)(t % p.nRT) * kBM + rl;
        if (r >= p.R) r = p.R - 1;  // rows past the end decode row R-1 and are never stored
        const int c0 = hbk * 128;   // first column of the half block
        const int hb = (c0 % kT) < 128 ? 1 : 0;
        const uint32_t* blk = p.codes + (r * p.nb + c0 / kT) * WPB;
        const uint4* v4 = reinterpret_cast<const uint4*>(blk + hb * 4 * K);
#pragma unroll
        for (int i = 0; i < K; ++i) {
          const uint4 v = __ldg(v4 + i);
          hw.w[4 * i] = v.x; hw.w[4 * i + 1] = v.y; hw.w[4 * i + 2] = v.z; hw.w[4 * i + 3] = v.w;
        }
        hw.w[4 * K] = __ldg(blk + (hb ? 0 : 4 * K));
        hw.scale = __ldg(p.scales + r);
      };
      // one stage: decode run qh (of the half block) into slot g % NS
      auto stage = [&](const RunWords<K>& rw, int g) -> bool {
        const int s = g % NS;
        if (g >= NS && !tc::mbar_wait(empty + s, (uint32_t)((g / NS) & 1) ^ 1u, p.wait_ns)) return false;
        decode_run_to_tile<K, L>(rw, a_tiles + (size_t)s * C_::ATile + rl * RowBytes, sw, 4 * h);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(full_a + s);
        return true;
      };
      auto process = [&](const HalfWords& hw, const Cursor& c) -> bool {
        int hbk, ks0, r0;
        const bool round = turn(c.v, hbk, ks0, r0);
        const int gbase = c.lt * nk + ks0;  // this CTA's stage index
        if (round) {
#pragma unroll
          for (int ss = 0; ss < SPH; ++ss) {  // run qh = ss*RPR + h, at words (3-qh)*K
            RunWords<K> rw;
#pragma unroll
            for (int i = 0; i <= K; ++i) {
              if constexpr (RPR > 1) rw.w[i] = h ? hw.w[(2 - ss * RPR) * K + i] : hw.w[(3 - ss * RPR) * K + i];
              else rw.w[i] = hw.w[(3 - ss) * K + i];
            }
            rw.scale = hw.scale;
            if (!stage(rw, gbase + ss * NG)) return false;
          }
          return true;
        }
        RunWords<K> rw;  // one stage of run r0: select its words
#pragma unroll
        for (int i = 0; i <= K; ++i) {
          uint32_t v = 0;
#pragma unroll
          for (int rr = 0; rr < SPH; ++rr)
#pragma unroll
            for (int hh = 0; hh < RPR; ++hh)
              if (rr == r0 && hh == h) v = hw.w[(3 - rr * RPR - hh) * K + i];
          rw.w[i] = v;
        }
        rw.scale = hw.scale;
        return stage(rw, gbase);
      };
      // two turns in flight: the words of turn u + 2 load while turn u decodes
      HalfWords ha, hb2;
      Cursor cu{0, 0}, cf{0, 0};  // the turn being decoded, the turn being fetched
      fetch(ha, cf);
      advance(cf);
      fetch(hb2, cf);
      advance(cf);
      for (int u = 0; u < nturn;) {
        if (!process(ha, cu)) { *fail = 1; break; }
        advance(cu);
        fetch(ha, cf);
        advance(cf);
        if (++u >= nturn) break;
        if (!process(hb2, cu)) { *fail = 1; break; }
        advance(cu);
        fetch(hb2, cf);
        advance(cf);
        ++u;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  // split: no CTA of the cluster leaves while a peer may still read its chunk buffers or arrive on its
  // barriers (every wait is bounded, so every CTA gets here)
  if (split) tc::cluster_sync_all();
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
  static PerDevice<int> sms_of;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  return sms_of.get(dev, [dev] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 148;
    }
    return n;
  }, 148);
}

template <int K, int L, int BN, int BK, int AX>
cudaError_t prefill_launch(PrefillParams p, const uint16_t* x, cudaStream_t st, const PrefillLaunch* plan,
                           int nplan) {
  using C_ = Cfg<BN, BK, AX == 0>;
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap map, omap;
  memset(&omap, 0, sizeof(omap));
  {  // x [M][Kd] bf16, boxes of [NMMA tokens][BK columns], swizzled
    const cuuint64_t dims[2] = {(cuuint64_t)p.Kd, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.Kd * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)C_::NMMA};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, C_::TmaSw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.tma_out = 0;
  if (p.nOut % 8 == 0) {  // out rows are 16-byte multiples: tensor stores of [32 tokens][32 features] boxes
    const cuuint64_t dims[2] = {(cuuint64_t)p.nOut, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.nOut * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
        CUDA_SUCCESS)
      p.tma_out = 1;
  }
  auto kern = prefill_kernel<K, L, BN, BK, AX>;
  static PerDevice<cudaError_t> attr_of;  // per instantiation; function attributes are per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const cudaError_t attr_err = attr_of.get(dev, [kern] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_::Smem);
  }, cudaErrorInvalidDevice);
  if (attr_err != cudaSuccess) return attr_err;
  p.nRT = (int)((p.nOut + kBM - 1) / kBM);
  p.nTiles = p.nRT * ((p.M + BN - 1) / BN);
  // Axis 1: a decoder group's stages are C_::Groups apart within a tile; with nk a multiple of the group
  // count they stay so across the tiles of a persistent CTA (the stage ring relies on it).  Coded widths
  // are multiples of 256 columns, so this always holds.
  if (AX == 1 && ((p.Kd + BK - 1) / BK) % C_::Groups != 0) return cudaErrorInvalidValue;
  const int sms = sm_count();
  // one launch over tiles [t0, t0 + count): persistent CTAs (S = 1) or one tile per cluster of S CTAs
  auto launch_part = [&](int t0, int count, int S) -> cudaError_t {
    PrefillParams q = p;
    q.t0 = t0;
    q.nTiles = count;
    q.S = S;
    if (S > 1) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3((unsigned)(count * S));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = C_::Smem;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)S;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, omap, q);
      return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int grid = count < sms ? count : sms;
    kern<<<grid, kThreads, C_::Smem, st>>>(map, omap, q);
    return cudaGetLastError();
  };
  for (int i = 0; i < nplan; ++i) {
    const cudaError_t e = launch_part(plan[i].t0, plan[i].count, plan[i].S);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int K, int L, int AX>
cudaError_t prefill_bn(const PrefillParams& p, const uint16_t* x, cudaStream_t st, int BN, const PrefillLaunch* plan,
                       int nplan) {
  if (BN == 32) return prefill_launch<K, L, 32, 64, AX>(p, x, st, plan, nplan);
  if (BN == 64) return prefill_launch<K, L, 64, 64, AX>(p, x, st, plan, nplan);
  if (BN == 128) return prefill_launch<K, L, 128, 64, AX>(p, x, st, plan, nplan);
  if (BN == 256) return prefill_launch<K, L, 256, 64, AX>(p, x, st, plan, nplan);
  return prefill_launch<K, L, 512, 32, AX>(p, x, st, plan, nplan);
}

template <int AX>
cudaError_t prefill_axis(const PrefillParams& p, const uint16_t* x, int k, int L, cudaStream_t st) {
  PrefillLaunch plan[2];
  int BN = 0;
  const int nplan = prefill_plan(p.M, AX, p.nOut, p.Kd, sm_count(), &BN, plan);
  if (L == 16) {
    if (k == 2) return prefill_bn<2, 16, AX>(p, x, st, BN, plan, nplan);
    if (k == 3) return prefill_bn<3, 16, AX>(p, x, st, BN, plan, nplan);
    return prefill_bn<4, 16, AX>(p, x, st, BN, plan, nplan);
  }
  if (k == 2) return prefill_bn<2, 12, AX>(p, x, st, BN, plan, nplan);
  if (k == 3) return prefill_bn<3, 12, AX>(p, x, st, BN, plan, nplan);
  return prefill_bn<4, 12, AX>(p, x, st, BN, plan, nplan);
}

}  // namespace

// Tiles: 128 output features x BN tokens, BN = 512 for M > 256 (stages of 32 columns), else the smallest
// of 32..256 covering M (stages of 64 columns), except 128 rather than 64 on axis 1.  Axis 1 runs one persistent launch.  Axis 0 has few
// output tiles (one per 128 features), each with a long reduction:
//   - when they leave SMs idle, a cluster of S CTAs splits each tile's reduction (S * tiles <= SMs);
//   - when they overrun whole waves, the full waves run unsplit and the tiles left over run split in a
//     second launch, instead of as a nearly empty wave.
// The split reduction pushes each CTA's partial rows into the owners' shared memory with st.async, a few
// microseconds per tile whatever S is, so S goes up to the portable cluster size 8 (whose senders' slots
// fit in the idle stage ring) and at most the reduction's stage count.
int device_sm_count() { return sm_count(); }

int prefill_plan(int M, int axis, int64_t nOut, int64_t Kd, int sms, int* tokens_per_tile, PrefillLaunch* launches) {
  if (M <= prefill_small_max_m(axis)) {  // no tiles: the register-decode kernels (prefill_small.cu, prefill_axis0_small.cu)
    *tokens_per_tile = 0;
    return 0;
  }
  // axis 1 skips 64-token tiles: 128-token tiles measured 51.3 against 53.3 us at 40 and 64 tokens (17408 x
  // 5120, k = 2, the same bits); on axis 0 they measured slower (90.4 against 84.6 us, k = 3)
  const int BN = M <= 32 ? 32 : M <= 64 ? (axis == 1 ? 128 : 64) : M <= 128 ? 128 : M <= 256 ? 256 : 512;
  const int BK = BN == 512 ? 32 : 64;
  const int nk = (int)((Kd + BK - 1) / BK);
  const int nTiles = (int)((nOut + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  const int cap = kMaxSplit;
  if (sms < 1) sms = 1;
  auto split_of = [&](int count) {
    int S = sms / count;
    if (S > cap) S = cap;
    if (S > nk) S = nk;
    return S < 1 ? 1 : S;
  };
  *tokens_per_tile = BN;
  if (axis == 0 && nTiles > sms && nTiles % sms != 0) {
    const int rem = nTiles % sms;
    launches[0] = PrefillLaunch{0, nTiles - rem, 1};
    launches[1] = PrefillLaunch{nTiles - rem, rem, split_of(rem)};
    return 2;
  }
  launches[0] = PrefillLaunch{0, nTiles, axis == 0 ? split_of(nTiles) : 1};
  return 1;
}

cudaError_t launch_gemm_prefill(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                                int M, int k, int L, int axis, int64_t rows, int64_t cols, cudaStream_t st) {
  if (M <= prefill_small_max_m(axis))
    return axis == 1 ? launch_prefill_small(codes, scales, x, out, M, k, L, rows, cols, st)
                     : launch_prefill_axis0_small(codes, scales, x, out, M, k, L, rows, cols, st);
  PrefillParams p{};
  p.codes = codes; p.scales = scales; p.out = out;
  p.R = rows; p.C = cols; p.M = M; p.nb = (int)(cols / kT);
  p.nOut = axis == 1 ? rows : cols;
  p.Kd = axis == 1 ? cols : rows;
  p.wait_ns = g_wait_ns.load();
  return axis == 1 ? prefill_axis<1>(p, x, k, L, st) : prefill_axis<0>(p, x, k, L, st);
}

// Limit of each pipeline wait of the tensor-core kernels (ns); 0 restores the default.
void set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : kWaitNs); }

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
