/*
 * trellis.h -- C ABI of libtrellis.so: linear layers over packed trellis-coded
 * (QTIP "1MAD") weights on NVIDIA GB300 (sm_103a).
 *
 * Format (from the "trellis-linear.ts" diff page, mlx-bun 0.2.0 -> 0.4.0, the
 * file's header comment): a weight matrix is stored as a uint32 bitstream
 * codes[rows][cols*k/32] plus one fp16 scale per stored row.  Each stored row
 * is a sequence of blocks of T positions (T*k/32 words per block).  The state
 * of position t of a block is the L-bit window starting at bit (T-1-t)*k of
 * the block, bits read least-significant first inside little-endian words and
 * wrapping to the block's first word.  A state s decodes with the 1MAD code:
 * x = s*34038481 + 76625530 (mod 2^32), y = (sum of the four bytes of x) - 510,
 * value = y / 147.800537109375, weight = value * scale[row].
 *
 * axis = 1: coded along the input dimension; the stored matrix is W [out, in]
 *           (rows = out features, cols = in features).
 * axis = 0: coded along the output dimension; the stored matrix is W^T
 *           [in, out] (rows = in features, cols = out features).
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers to memory the caller allocated
 *     and owns; the library never allocates, frees or retains them.  Inputs
 *     are read only.  Every pointer must be 16-byte aligned.
 *   - bf16 and fp16 values travel as their 16-bit storage patterns (uint16_t).
 *   - Arrays are dense and row-major in the shapes given below.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and return after the launch.  The library keeps no
 *     state between calls except a per-device cache of launch attributes;
 *     calls are thread-safe.
 *   - The return value is TRELLIS_OK or a negative trellis_status.  On every
 *     error except TRELLIS_ECUDA nothing was launched and no memory touched;
 *     TRELLIS_ECUDA reports the CUDA error seen at launch.
 *
 * Supported geometry of the GPU kernels: k in {2, 3, 4}, L = 16 or 12,
 * T = 256, rows >= 1, cols a positive multiple of T.  (The pages' own fast
 * paths assume L = 12 and T = 256; the measured workloads use L = 16.)
 */
#ifndef TRELLIS_H
#define TRELLIS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Geometry of one packed matrix (TrellisGeometry on the "trellis-linear.ts"
 * page: {k, L, T, axis, rows, cols}; rows/cols are the STORED matrix's). */
typedef struct trellis_geom {
  int32_t k;          /* bits per weight */
  int32_t L;          /* window (trellis state) length in bits */
  int32_t T;          /* positions per block */
  int32_t axis;       /* 1 or 0, see above */
  int64_t rows;       /* stored rows */
  int64_t cols;       /* coded positions per stored row */
  int32_t interleave; /* 0: row-major codes [rows][cols*k/32].
                         2: the k=3 axis-0 layout [cols/512][rows][48] of the
                         "trellis-linear.ts" format comment: two coded blocks
                         of a row side by side (words 0..23 and 24..47), the
                         rows of one 512-column group contiguous.  Supported
                         by trellis_expand_bf16 and the axis-0 matvecs. */
  int32_t reserved;   /* must be 0 */
} trellis_geom_t;

typedef void *trellis_stream_t; /* a cudaStream_t */

enum trellis_status {
  TRELLIS_OK = 0,
  TRELLIS_EGEOM = -1,      /* unsupported or inconsistent geometry */
  TRELLIS_EM = -2,         /* M outside the call's range */
  TRELLIS_EALIGN = -3,     /* a pointer is not 16-byte aligned */
  TRELLIS_EAXIS = -4,      /* geometry axis does not fit the call */
  TRELLIS_EWORKSPACE = -5, /* workspace missing, misaligned or too small */
  TRELLIS_ECUDA = -6,      /* CUDA reported an error at launch */
  TRELLIS_ENULL = -7,      /* a required pointer is NULL */
  TRELLIS_EDEVICE = -8     /* no usable sm_103 device is current */
};

/* Version of this interface (major*100 + minor): 101. */
int trellis_abi_version(void);

/* Static description of a status code; never NULL. */
const char *trellis_status_string(int status);

/* 0 if the GPU kernels support the geometry, else TRELLIS_EGEOM.  Pure host
 * check (trellisGeometry's rules plus the kernels' supported set). */
int trellis_check_geom(const trellis_geom_t *g);

/*
 * trellis_expand_bf16 -- decode the whole stored matrix
 * ("trellis-linear.ts": expandTrellis / EXPAND_SOURCE; "trellis-vector-
 * expand.ts").  out[r][c] = bf16(value(s(r,c)) * scale[r]), where value is
 * the correctly rounded fp32 quotient y / 147.800537109375, the product is
 * rounded to fp32 and then to bf16 (nearest, ties to even).  Bit-exact.
 *   codes  [rows][cols*k/32] uint32     scales [rows] fp16
 *   out    [rows][cols] bf16, in STORED order (for axis 0 this is W^T).
 * Any axis.  Writes every element of out.
 */
int trellis_expand_bf16(const uint32_t *codes, const uint16_t *scales, uint16_t *out,
                        const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_matvec_axis1 -- decode-fused matvec for M = 1..4 input rows over
 * an axis-1 matrix ("trellis-linear.ts": TrellisLinear.forward for M <= 4,
 * REDUCE_SOURCE; "trellis-shared-m.ts" for M = 2..4).
 *   out[m][r] = bf16( sum_c w(r,c) * x[m][c] ),  w = fp32 value * scale[r]
 * (the pages' default packed numerics: no bf16 rounding of the weight),
 * accumulated in fp32 in any order.
 *   codes [rows][cols*k/32]   scales [rows]   x [M][cols] bf16   out [M][rows] bf16
 * Requires g->axis == 1 and 1 <= M <= 4.
 */
int trellis_matvec_axis1(const uint32_t *codes, const uint16_t *scales, const uint16_t *x,
                         uint16_t *out, int M, const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_matvec_axis1_host -- trellis_matvec_axis1 with x and out in host
 * memory: one call queues, in order on `stream`, the copy of x_host
 * [M][cols] bf16 into the caller's device buffer x_dev, the matvec, and the
 * transfer of its output [M][rows] into out_host.  It returns once they are
 * queued; out_host holds the result when the stream has reached that point
 * (synchronize the stream or an event recorded after the call).  The pages'
 * decode call does the same for one token: its input arrives from the host
 * and its output goes back.
 *   x_host, out_host: host memory, no alignment rule.  Pinned memory
 *   (cudaHostAlloc / cudaHostRegister) mapped into the device's address space
 *   and 16-byte aligned is reached through that mapping: a small kernel copies
 *   x_host into x_dev and the matvec stores its output straight into out_host
 *   (out_dev is then not written).  Other host memory goes through the copy
 *   engines: x_host into x_dev, the matvec into out_dev, out_dev into
 *   out_host; pageable memory is copied through a driver staging buffer and
 *   the call may block.
 *   x_dev, out_dev: device memory, 16-byte aligned, owned by the caller; they
 *   must not be in use by other work until the stream has passed the call.
 *   codes, scales, M, g: as for trellis_matvec_axis1.
 * Errors: as for trellis_matvec_axis1 (TRELLIS_ENULL also for a NULL host or
 * staging pointer, TRELLIS_EALIGN for a staging buffer); TRELLIS_ECUDA if a
 * copy or the launch could not be queued.
 */
int trellis_matvec_axis1_host(const uint32_t *codes, const uint16_t *scales, const uint16_t *x_host,
                              uint16_t *out_host, int M, const trellis_geom_t *g, uint16_t *x_dev,
                              uint16_t *out_dev, trellis_stream_t stream);

/*
 * trellis_matvec_axis0 -- decode-fused matvec for M = 1..4 input rows over
 * an axis-0 matrix, i.e. a stored W^T ("trellis-linear.ts": the scatter path
 * of TrellisLinear.forward, SCATTER_SOURCE and its partial fold;
 * "trellis-balanced-scatter.ts" and "trellis-shared-scatter.ts").
 *   out[m][c] = bf16( sum_r w(r,c) * x[m][r] ),  w = fp32 value * scale[r]
 * The sum over stored rows is split across thread blocks; each block writes
 * fp32 partial sums to `workspace` and the last block to finish a column
 * block folds the partials in a fixed order (deterministic) and stores bf16.
 *   codes [rows][cols*k/32]   scales [rows]   x [M][rows] bf16   out [M][cols] bf16
 *   workspace: device memory of at least trellis_workspace_bytes(M, g) bytes,
 *   16-byte aligned, ZERO-FILLED before its first use; every call leaves it
 *   ready for the next one.  Calls that share a workspace must not overlap
 *   in time (put them on one stream).
 * Requires g->axis == 0 and 1 <= M <= 4.
 */
int trellis_matvec_axis0(const uint32_t *codes, const uint16_t *scales, const uint16_t *x,
                         uint16_t *out, int M, const trellis_geom_t *g, void *workspace,
                         size_t workspace_bytes, trellis_stream_t stream);

/*
 * trellis_matvec_axis1_bf16w, trellis_matvec_axis0_bf16w -- the two matvecs
 * with the pages' bf16-rounded weight numerics (decoder variants 0-3 of the
 * HEADER source in "trellis-linear.ts", TRELLIS_ROUND): every weight is
 * bf16(fl32(value * scale)) with the correctly rounded value -- exactly the
 * trellis_expand_bf16 weight -- before the fp32 multiply-add.  Arguments,
 * shapes, workspace and errors as for trellis_matvec_axis1 / _axis0.
 */
int trellis_matvec_axis1_bf16w(const uint32_t *codes, const uint16_t *scales, const uint16_t *x,
                               uint16_t *out, int M, const trellis_geom_t *g, trellis_stream_t stream);
int trellis_matvec_axis0_bf16w(const uint32_t *codes, const uint16_t *scales, const uint16_t *x,
                               uint16_t *out, int M, const trellis_geom_t *g, void *workspace,
                               size_t workspace_bytes, trellis_stream_t stream);

/* Bytes of workspace trellis_matvec_axis0 needs for (M, g); 0 if the
 * geometry or M is unsupported. */
size_t trellis_workspace_bytes(int M, const trellis_geom_t *g);

/*
 * trellis_matvec_axis0_noalloc -- the same axis-0 matvec as
 * trellis_matvec_axis0, for callers that cannot allocate device memory: a
 * custom-operator slot in an inference engine that passes a kernel only its
 * input and output tensors, or a serving runtime that plans all device
 * memory before it starts and forbids cudaMalloc afterwards.  The pages have
 * no counterpart; this call is an addition of this library.
 *
 * It takes no workspace argument.  The split-row partial sums live in a
 * fixed array of TRELLIS_NOALLOC_SCRATCH_BYTES bytes of device memory that
 * the library defines; every GPU that loads the library holds that array
 * until the process exits.  The call allocates nothing: it clears the
 * array's arrival counters with cudaMemsetAsync on `stream` and launches the
 * axis-0 kernel.  Each call looks up the array's device address
 * (cudaGetSymbolAddress, with the caller's device current) and keeps it per
 * device; a call whose stream is being captured into a CUDA graph uses the
 * kept address, so make the first call on each device before any stream
 * capture (a capture-time call with no kept address returns TRELLIS_ECUDA).
 * The fresh lookup keeps ordinary calls valid after cudaDeviceReset.  All
 * calls share the one array, so calls whose executions overlap on the GPU
 * race: issue them on one stream or otherwise serialise them.
 *
 * Arguments, shapes and results are those of trellis_matvec_axis0.  Returns
 * TRELLIS_EWORKSPACE when trellis_workspace_bytes(M, g) exceeds
 * TRELLIS_NOALLOC_SCRATCH_BYTES (the problem needs more scratch than the
 * fixed array holds; use trellis_matvec_axis0 with a larger workspace).
 */
#define TRELLIS_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20) /* 4 MiB */
int trellis_matvec_axis0_noalloc(const uint32_t *codes, const uint16_t *scales, const uint16_t *x,
                                 uint16_t *out, int M, const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_gateup_swiglu -- fused gate/up projections with the SwiGLU
 * activation for M = 1..4 ("trellis-linear.ts": fusedGateUpSwiglu /
 * GATEUP_SOURCE; "trellis-shared-m.ts": GATEUP_SHARED_M_SOURCE).  Both
 * matrices are decoded once per call, x is read once, and the gate and up
 * vectors are never stored:
 *   g = bf16(sum_c wg(r,c) x[m][c]),  u = bf16(sum_c wu(r,c) x[m][c])
 *   sig = bf16(1 / (1 + exp(-g))),  silu = bf16(g * sig),
 *   out[m][r] = bf16(silu * u)      (fp32 arithmetic between the casts)
 * Both matrices share the geometry g (axis 1; same k, L, T, rows, cols).
 *   gcodes, ucodes [rows][cols*k/32]   gscales, uscales [rows]
 *   x [M][cols] bf16   out [M][rows] bf16
 */
int trellis_gateup_swiglu(const uint32_t *gcodes, const uint16_t *gscales, const uint32_t *ucodes,
                          const uint16_t *uscales, const uint16_t *x, uint16_t *out, int M,
                          const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_mlp_decode -- the decode-time MLP block of the pages' Qwen3MLP
 * ("qwen3_5.ts" diff page, Qwen3MLP.forward for M <= 4: the fused gate/up
 * SwiGLU kernel followed by the down projection):
 *   hidden = trellis_gateup_swiglu(gate, up, x)        [M][I] bf16
 *   out    = trellis_matvec_axis0(down, hidden)        [M][H] bf16
 * Two kernel launches on `stream`, no allocation and no synchronisation, so
 * the call can be captured into a CUDA graph.
 *   g_up    axis-1 geometry of gate and up: rows = I (intermediate), cols = H
 *   g_down  axis-0 geometry of down (stored W^T): rows = I, cols = H
 *   x [M][H]   hidden [M][I] (caller-owned, written)   out [M][H]
 *   workspace: as for trellis_matvec_axis0 with (M, g_down).
 * Requires 1 <= M <= 4; k may differ between the two geometries.
 */
int trellis_mlp_decode(const uint32_t *gcodes, const uint16_t *gscales, const uint32_t *ucodes,
                       const uint16_t *uscales, const uint32_t *dcodes, const uint16_t *dscales,
                       const uint16_t *x, uint16_t *hidden, uint16_t *out, int M,
                       const trellis_geom_t *g_up, const trellis_geom_t *g_down, void *workspace,
                       size_t workspace_bytes, trellis_stream_t stream);

/*
 * trellis_gemm_prefill -- prefill GEMM over an axis-1 or axis-0 matrix for any
 * M >= 1 (intended for M > 4) ("trellis-tiled-prefill.ts": tiledTrellisPrefill
 * and the expand + matmul path of TrellisLinear.forward;
 * "trellis-splitk-prefill.ts" for axis 0).  Weight tiles are
 * decoded into shared memory as bf16 (the expand numerics: bf16 of the
 * correctly rounded value times the scale), x tiles arrive by TMA, and the
 * 5th-generation tensor cores (tcgen05, accumulators in tensor memory)
 * compute
 *   out[m][r] = bf16( sum_c e(r,c) * x[m][c] ),  e = the bf16 expand weight,
 * accumulated in fp32.
 *   codes [rows][cols*k/32]   scales [rows]   x [M][cols] bf16   out [M][rows] bf16
 * Axis 0 (stored W^T, the down projection): out[m][c] = bf16( sum_r e(r,c) *
 * x[m][r] ), x [M][rows], out [M][cols]; weights are decoded along the stored
 * rows and stored transposed into the tile, and the long reduction over rows
 * is split across thread-block clusters where tiles alone would leave SMs
 * idle (possibly as a second launch on `stream` for the tiles left after
 * whole waves).  With M <= 24 on axis 1 and M <= 32 on axis 0 the decoded
 * weights stay in registers instead and warp-level MMAs (mma.sync bf16, one
 * to four 8-token tiles) multiply them: the same numerics, no shared-memory weight tiles; on axis 0 a
 * thread-block cluster splits each 256-output block's reduction and folds
 * it through distributed shared memory.  Results
 * are deterministic: repeated calls give equal bits.
 * Requires M >= 1, no interleaved layout, and for axis 0 rows % 8 == 0.
 */
int trellis_gemm_prefill(const uint32_t *codes, const uint16_t *scales, const uint16_t *x,
                         uint16_t *out, int M, const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_load_floor -- measurement aid with no counterpart in the pages'
 * operations: reads an axis-1 bitstream with exactly the access pattern of
 * trellis_matvec_axis1 at M = 1 (one lane per stored row, 16-byte loads of
 * half blocks) and decodes nothing; out[r] = XOR of every word it loads for
 * stored row r: each block's words plus the spill reads of its words 4k and
 * 0, i.e. the XOR of the row's words other than words 0 and 4k of each block.
 * Its bandwidth is the HBM rate that access pattern can reach, the floor
 * the decode-fused matvec is compared with.
 *   codes [rows][cols*k/32] (device, 16-byte aligned)   out [rows] uint32 (device)
 * Requires a valid axis-1 geometry without the interleaved layout.  Errors:
 * EGEOM, EAXIS, ENULL, EALIGN, EDEVICE, ECUDA (launch).
 */
int trellis_load_floor(const uint32_t *codes, uint32_t *out, const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_load_floor_rows -- measurement aid with no counterpart in the
 * pages' operations: reads the same axis-1 bitstream fully coalesced (one
 * warp per stored row, its lanes on consecutive 16-byte chunks of the row,
 * warps striding over the rows in one wave) and decodes nothing;
 * out[r] = XOR of all words of stored row r.  Its bandwidth is what the best
 * access pattern reaches on HBM for a stream of this size.
 *   codes [rows][cols*k/32] (device, 16-byte aligned)   out [rows] uint32 (device)
 * Requires a valid axis-1 geometry without the interleaved layout.  Errors:
 * EGEOM, EAXIS, ENULL, EALIGN, EDEVICE, ECUDA (launch).
 */
int trellis_load_floor_rows(const uint32_t *codes, uint32_t *out, const trellis_geom_t *g, trellis_stream_t stream);

/*
 * trellis_prefill_plan -- the tile plan trellis_gemm_prefill follows for
 * (M, g) on a GPU with `sms` SMs (sms < 1: the current device's).  Host
 * arithmetic only: no CUDA call unless sms < 1, nothing launched.  Writes
 * the tokens per tile to *tokens_per_tile and, per launch, three ints to
 * launches[3*i ..]: first tile, tile count, and CTAs per tile (a thread-
 * block cluster splitting each tile's reduction when > 1).  Tiles are 128
 * output features x tokens_per_tile tokens; tile t is feature tile
 * t % ceil(features/128), token tile t / ceil(features/128).
 *   launches: caller-owned, room for 2 launches (6 ints).
 * Returns the number of launches (1 or 2); 0, with *tokens_per_tile = 0,
 * when the call has no tiles: with M <= 24 (axis 1) or M <= 32 (axis 0)
 * trellis_gemm_prefill decodes
 * into registers and multiplies with warp-level MMAs instead (axis 1: 64
 * rows per thread block; axis 0: a thread-block cluster per 256 outputs).  Or a negative status: the geometry and M checks
 * of trellis_gemm_prefill, ENULL, or EDEVICE when sms < 1 and no usable
 * device is current.
 */
int trellis_prefill_plan(int M, const trellis_geom_t *g, int sms, int *tokens_per_tile, int *launches);

/*
 * trellis_device_error -- diagnostic of the tensor-core kernel.  Every wait on
 * an mbarrier inside trellis_gemm_prefill is bounded (2 s); a wait that gives
 * up records a non-zero code in a device word instead of hanging the GPU.
 * Returns that code (0 = none), reading it synchronously from the current
 * device; reset != 0 clears it.  Negative values are trellis_status errors.
 */
int trellis_device_error(int reset);

/*
 * trellis_set_wait_limit -- diagnostic with no counterpart in the pages:
 * sets the limit of each bounded wait in the tensor-core kernel
 * (trellis_gemm_prefill) for launches issued after the call, in
 * nanoseconds of the GPU's global timer; 0 restores the default (2 s).
 * It exists so that tests can make the waits run out on an ordinary
 * problem and check the error path: the kernel then records a non-zero
 * code (trellis_device_error), lets its copies and MMAs already issued
 * finish, and returns with the context intact; its output is undefined.
 * The setting is process-wide and applies to every device.  Returns
 * TRELLIS_OK.
 */
int trellis_set_wait_limit(uint64_t nanoseconds);

#ifdef __cplusplus
}
#endif

#endif /* TRELLIS_H */
