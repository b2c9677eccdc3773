/*
 * bsp.h - bitmap-encoded unstructured sparse matmul on one GB300 (sm_103a).
 *
 * Computes Y = W * X for an unstructured-pruned weight W (M x K, any zero
 * pattern) held in a bitmap-indexed tile format, and a dense activation
 * block X (K x N).
 *
 * Format (TCA-BME, from "SpInfer: How bitmaps make sparse LLMs actually
 * fast", sections "How TCA-BME addresses the indexing overhead" and "The
 * Values array and why it's confusing at first"):
 *   - BitmapTile (BT): 8x8 elements, one uint64 bitmap, bit set <=> the
 *     element's raw bits are nonzero; bit p = 8*row + col inside the BT.
 *   - TCTile: 16x16 = 2x2 BTs, stored in mma A-register order
 *     (rows 0-7/cols 0-7, rows 8-15/cols 0-7, rows 0-7/cols 8-15,
 *      rows 8-15/cols 8-15).
 *   - GroupTile (GT): 64x64 = 4x4 TCTiles, row-major; GTs row-major over the
 *     ceil(M/64) x ceil(K/64) grid.  BT g = (t*16 + tc)*4 + b for GT t,
 *     TCTile tc.  When M or K is not a multiple of 64 the edge GTs are
 *     padded with zeros (their bits are 0 and nothing is stored for them).
 *   - values: the nonzeros only, packed in GT -> TCTile -> BT -> bit order.
 *   - offsets: uint32 [NGT+1], offsets[t] = nonzeros stored before GT t.
 *   A value's index is offsets[t] + (nonzeros of the earlier BTs of its GT)
 *   + popcount(bitmap & ((1 << p) - 1)) (the masked popcount of the
 *   section "Shared Memory Bitmap Decoding (SMBD)").
 *
 * Layouts: W is row-major [M][K].  X is [N][K] and Y is [N][M] with K and M
 * contiguous (PyTorch's [tokens, features]); that is the column-major view
 * of the pages' K x N and M x N, so row n of Y is W times row n of X.
 *
 * Pointers: arguments documented "device" must be device memory of the
 * current device (or managed memory); "host" arguments are ordinary host
 * memory.  No call keeps a pointer to caller memory after it returns,
 * except that kernels launched on `stream` read and write it until they
 * complete.
 *
 * Errors: every entry point returns a bsp_status_t and never aborts or
 * throws.  A launch failure reports BSP_ERR_CUDA (the CUDA error is also
 * left for cudaGetLastError()).  Calls that launch work are asynchronous
 * with respect to the host unless stated otherwise.
 *
 * Threading: a handle is immutable after bsp_encode except for its split-K
 * workspace; calls that compute with one handle must be serialised on one
 * stream (as with a cuBLAS handle).  Distinct handles are independent.
 */
#ifndef BSP_H
#define BSP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *bsp_stream_t;

typedef struct bsp_handle *bsp_handle_t;

typedef enum {
    BSP_OK = 0,
    BSP_ERR_INVALID_ARG = 1, /* null pointer, N out of range, bad handle   */
    BSP_ERR_SHAPE = 2,       /* M, K < 1, or K not a multiple of 8 (fp16) / 16 (int8) */
    BSP_ERR_DTYPE = 3,       /* call does not match the handle's dtype     */
    BSP_ERR_ALIGN = 4,       /* X / Y / W not 16-byte aligned              */
    BSP_ERR_OOM = 5,         /* device or host allocation failed           */
    BSP_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed       */
    BSP_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up         */
    BSP_ERR_INTERNAL = 8     /* an invariant of the format was violated    */
} bsp_status_t;

typedef enum {
    BSP_FP16 = 0, /* IEEE binary16 values, fp32 accumulation, fp16 output */
    BSP_INT8 = 1  /* int8 values, int32 accumulation (exact)             */
} bsp_dtype_t;

/* Largest N of the decode path (the skinny product, N <= 16): split-K
 * workspaces are sized for it.  Larger N run the prefill kernel (fp16) or
 * the decode kernels over blocks of 16 columns (int8). */
#define BSP_DECODE_MAX_N 16

typedef struct {
    int64_t M, K;
    int32_t dtype;        /* bsp_dtype_t                                   */
    int32_t gt_m, gt_k;   /* GroupTile shape: 64, 64                        */
    int32_t device;       /* CUDA device the arrays live on                */
    int64_t NGT, NBT;     /* GroupTiles, BitmapTiles of the padded grid     */
    uint64_t NNZ;         /* stored nonzeros                                */
    const uint64_t *bitmaps; /* device, [NBT]                              */
    const uint32_t *offsets; /* device, [NGT + 1]                          */
    const void *values;      /* device, [NNZ] (+16 B tail slack, not counted) */
} bsp_info_t;

/* Short static description of a status code (never NULL). */
const char *bsp_status_string(bsp_status_t s);

/*
 * Encode a dense weight into the format, on the device.
 *   W      device, row-major [M][K] fp16 or int8 (raw bits are examined:
 *          an element is stored iff its bits are nonzero, so -0.0 / NaN /
 *          Inf are kept as payload); 16-byte aligned.  Not retained.
 *   M, K   M >= 1; K a multiple of 8 for fp16 or of 16 for int8, so that
 *          every row of W and of X starts on a 16-byte boundary
 *          (BSP_ERR_SHAPE otherwise); the total nonzero count must fit in
 *          uint32.  M and K need not be multiples of 64 (zero-padded edge
 *          GTs; NGT and NBT count the padded grid).
 *   stream work is ordered on it; the call synchronises `stream` once (to
 *          learn NNZ and size the values array), so W may be freed when it
 *          returns.
 *   out    receives the new handle, which owns every device array it uses.
 * Encoding is an offline step; the pages exclude it from kernel timings
 * (UnionSparse, "Baselines and Fairness").
 */
bsp_status_t bsp_encode(const void *W, bsp_dtype_t dtype, int64_t M, int64_t K,
                        bsp_stream_t stream, bsp_handle_t *out);

/* Free a handle and its device arrays (synchronises the device first). */
bsp_status_t bsp_destroy(bsp_handle_t h);

/*
 * Y = W * X.  ("Unified Static-Dynamic Pruning for Efficient LLM
 * Inference", section 3.1: W in R^{MxK}, X in R^{KxN}.)
 *   X  device [N][K], fp16 (BSP_FP16 handle) or int8 (BSP_INT8), 16-B aligned.
 *   Y  device [N][M], fp16 (BSP_FP16) or int32 (BSP_INT8), 16-B aligned.
 *   N  >= 1.  Kernels, by dtype and N (the crossovers are the tuning
 *      knobs BSP_TUNE_NARROW_MIN_N, default 3, and BSP_TUNE_NARROW_MIN_N_I8,
 *      default 3):
 *        fp16, N <= 2: the GT-per-warp CUDA-core decode kernel (split-K
 *          over GroupTiles, fp32 accumulation);
 *        fp16, 3 <= N <= 16: the narrow tcgen05 kernel (decoded tiles in
 *          tensor memory, MMAs of N = 16, fp32 accumulation, persistent
 *          CTAs; tiles split between CTAs are finished by a second kernel);
 *        fp16, N > 16: the tcgen05 prefill kernel (decoded tiles in shared
 *          memory, fp32 accumulation in tensor memory);
 *        int8, N <= 2: the CUDA-core team decode kernel (dp4a);
 *        int8, 3 <= N <= 16: the same narrow tcgen05 kernel on exact fp16
 *          copies of the int8 weights and activations (fp32 accumulation in
 *          runs of at most 16 GroupTile columns, each an exact integer below
 *          2^24, added as int32);
 *        int8, N > 16: the team decode kernel over blocks of 16 columns.
 * fp16: Y = fp16(round-to-nearest of an fp32 sum in unspecified order).
 * int8: Y is the exact int32 sum.
 */
bsp_status_t bsp_spmm(bsp_handle_t h, const void *X, int64_t N, void *Y,
                      bsp_stream_t stream);

/*
 * Deterministic split-K (on = 1) or the default atomic one (on = 0).
 * The decode kernels (bsp_spmm with N <= BSP_DECODE_MAX_N, bsp_spmspv) split
 * the K range of a row strip or tile over several CTAs.  By default the
 * fp16 partial sums meet through fp32 atomic adds, so the rounding order,
 * and with it the last bit of an fp16 output, may change from call to
 * call.  With on = 1 each split stores its partial sums to a slot of its
 * own and the slots are added in split order (by the last CTA of the strip
 * in the CUDA-core kernels, by the finishing kernel after the tcgen05 and
 * column-index kernels): the same inputs give bit-identical outputs on
 * every call on the same GPU model (the split count depends on the SM
 * count).  int8 is exact either way; the prefill kernel (fp16,
 * N > BSP_DECODE_MAX_N) adds its two K halves in a fixed order and is
 * deterministic either way.  The first switch-on
 * allocates the slots (splits x BSP_DECODE_MAX_N x M fp32) on the handle's
 * device; later calls do not allocate.  Not safe to call while another
 * thread uses the handle.  BSP_ERR_INVALID_ARG for a bad handle or an `on`
 * other than 0 or 1; BSP_ERR_OOM if the slots cannot be allocated (the
 * mode is then unchanged).
 */
bsp_status_t bsp_set_deterministic(bsp_handle_t h, int on);

/*
 * Process-wide tuning of the dispatch (the pages fix none of these; they
 * are launch choices of this library).  Each knob starts from the
 * environment variable named beside it, read once, at the first product
 * call or bsp_get_tuning / bsp_set_tuning of the process; afterwards only
 * bsp_set_tuning changes it.  A change applies to calls made after it
 * returns; it is not synchronised with calls other threads make meanwhile.
 *   BSP_TUNE_SPLITK          (BSP_SPLITK)        split-K count of the
 *                            CUDA-core decode kernels; 0 = automatic
 *   BSP_TUNE_NARROW_CTAS     (BSP_NARROW_CTAS)   CTAs the tcgen05 decode
 *                            kernel's steps are balanced over; 0 = automatic
 *                            (every resident slot)
 *   BSP_TUNE_UNION_SPLITK    (BSP_UNION_SPLITK)  split-K count of the IE-BME
 *                            product; 0 = automatic
 *   BSP_TUNE_NARROW_MIN_N    (BSP_NARROW_MIN_N)  smallest fp16 N <= 16 that
 *                            runs the tcgen05 decode kernel; larger than 16:
 *                            never; default 3
 *   BSP_TUNE_PREFILL_KSPLIT  (BSP_PF_KSPLIT)     prefill split-K over a CTA
 *                            pair: -1 automatic, 0 off, 1 on (N <= 256)
 *   BSP_TUNE_PREFILL_CSTAGES (BSP_PF_SC)         compressed-ring depth of the
 *                            prefill kernel; 0 = as many as fit
 *   BSP_TUNE_NARROW_MIN_N_I8 (BSP_NARROW_MIN_N_I8) smallest int8 N <= 16
 *                            that runs the tcgen05 decode kernel; larger
 *                            than 16: never; default 3
 * Split counts are clamped to the problem (at most one per GroupTile
 * column).  BSP_ERR_INVALID_ARG for an unknown knob or a value out of range
 * (split counts and stages 0..4096, NARROW_CTAS 0..2^20, NARROW_MIN_N and
 * NARROW_MIN_N_I8 1..1024, KSPLIT -1..1).
 */
typedef enum {
    BSP_TUNE_SPLITK = 0,
    BSP_TUNE_NARROW_CTAS = 1,
    BSP_TUNE_UNION_SPLITK = 2,
    BSP_TUNE_NARROW_MIN_N = 3,
    BSP_TUNE_PREFILL_KSPLIT = 4,
    BSP_TUNE_PREFILL_CSTAGES = 5,
    BSP_TUNE_NARROW_MIN_N_I8 = 6
} bsp_tune_t;

bsp_status_t bsp_set_tuning(bsp_tune_t knob, int64_t value);
bsp_status_t bsp_get_tuning(bsp_tune_t knob, int64_t *value);

/*
 * INT8 with per-row dequantisation: Y[n][m] = fp32(acc[n][m]) * row_scale[m],
 * one round-to-nearest int->float conversion and one fp32 multiply (on the
 * CUDA-core team decode kernel at every N).
 *   X device int8 [N][K]; row_scale device fp32 [M]; Y device fp32 [N][M].
 *   1 <= N <= BSP_DECODE_MAX_N.  BSP_ERR_DTYPE on an fp16 handle.
 */
bsp_status_t bsp_spmm_scaled(bsp_handle_t h, const int8_t *X, int64_t N,
                             const float *row_scale, float *Y,
                             bsp_stream_t stream);

/*
 * Sparse-matrix times sparse-vector: y = W * x for one activation vector,
 * skipping the weight columns whose activation is exactly zero ("Unified
 * Static-Dynamic Pruning for Efficient LLM Inference", sections 4.2-4.2.1:
 * inactive columns are neither loaded nor decoded).  The result equals
 * bsp_spmm with N = 1.
 *   x device [K] (fp16 or int8), y device [M] (fp16 or int32), 16-B aligned.
 * With a column index (bsp_build_column_index) the skip unit is the column
 * for both the fetch and the arithmetic: only the active columns' bitmaps
 * and values are read.  Without one it runs on the row-wise format: fp16
 * skips the multiply-adds per column and the fetch per K-octet (a BT column
 * of 8 activations, fetched only when one of them survives, and fetched by
 * the octet only in GroupTiles where at most two of the eight octets
 * survive); int8 skips per K-octet.
 */
bsp_status_t bsp_spmspv(bsp_handle_t h, const void *x, void *y,
                        bsp_stream_t stream);

/*
 * spMspV with magnitude pruning of the activations, the dynamic pruning of
 * "Unified Static-Dynamic Pruning for Efficient LLM Inference" (section
 * 3.2 and 4.2, a TEAL-style magnitude criterion):
 *   y = W * x',  x'_k = 0 if |x_k| <= threshold, else x_k.
 * Pruned columns are skipped as in bsp_spmspv (with a column index, per
 * column; without, per K-octet); threshold = 0 is exactly bsp_spmspv.  NaN activations are
 * never pruned.  threshold must be >= 0 (BSP_ERR_INVALID_ARG otherwise).
 * The comparison is |x| <= threshold with x widened exactly to fp32.
 */
bsp_status_t bsp_spmspv_threshold(bsp_handle_t h, const void *x, float threshold,
                                  void *y, bsp_stream_t stream);

/*
 * Tiled-CBC column index ("Unified Static-Dynamic Pruning for Efficient LLM
 * Inference", section 4.1, "Tiled-CBC: Unified Compression Format"): a
 * column-major copy of the encoded weight that lets bsp_spmspv and
 * bsp_spmspv_threshold fetch only the columns whose activation survives
 * (section 4.2, step (3)).  GTiles of 256 x 64 elements tile W row-major (M
 * and K zero-padded to multiples of 256 and 64); each 256 x 1 column tile
 * has four uint64 bitmaps (rows 0-63, 64-127, 128-191, 192-255; bit r % 64
 * of word r / 64 <=> element r is nonzero); the GTile's nonzeros follow in
 * column order, top to bottom.  Arrays: TileOffset u32 [NGT + 1] (values
 * before each GTile), ColInfo u32 [NGT * 64] (column's first value inside
 * its GTile << 16 | its nonzero count), bitmaps u64 [NGT * 64 * 4], values
 * [NNZ].  Storage, the page's closed form with TILE_K = 64:
 *   4 (NGT + 1) + 4 NGT 64 + 8 NBM + B_v NNZ,  NBM = (M, K padded) / 64.
 *
 * bsp_build_column_index builds it on the handle's device from the handle's
 * arrays (allocates the index and a dense scratch copy of W, synchronises
 * `stream`); from then on the handle's spMspV calls use it (and allocate
 * nothing).  Building again replaces it.  BSP_ERR_OOM if it does not fit.
 */
bsp_status_t bsp_build_column_index(bsp_handle_t h, bsp_stream_t stream);

/* Bytes of the column index (the closed form above); BSP_ERR_INVALID_ARG
 * when the handle has none. */
bsp_status_t bsp_column_index_bytes(bsp_handle_t h, uint64_t *bytes);

/* Copies of the index arrays (device or host memory, any pointer may be
 * NULL), ordered on `stream`; BSP_ERR_INVALID_ARG without an index. */
bsp_status_t bsp_column_index_export(bsp_handle_t h, uint32_t *offsets, uint32_t *colinfo,
                                     uint64_t *bitmaps, void *values, bsp_stream_t stream);

/*
 * Same product as bsp_spmm, from and to HOST memory: copies X in, runs the
 * product and copies Y out on `stream`, then synchronises `stream`.  Uses a
 * device staging buffer owned by the handle (grown on demand, so this call
 * may allocate).  X host [N][K]; Y host [N][M]; pinned memory is fastest.
 */
bsp_status_t bsp_spmm_host(bsp_handle_t h, const void *X_host, int64_t N,
                           void *Y_host, bsp_stream_t stream);

/*
 * bsp_spmm_host without the final synchronisation: the copies and the
 * product are only enqueued on `stream`, so calls on several handles
 * overlap their transfers and kernels.  Y_host holds the result once
 * `stream` has been synchronised (or an event recorded after the call has
 * completed); X_host and Y_host must stay valid until then and should be
 * pinned (pageable memory makes the copies synchronous with the host).
 * Successive calls on one handle reuse its staging buffers in stream order,
 * so they must use the same stream; a call that needs larger staging
 * buffers than the handle holds replaces them, which synchronises the
 * device (cudaFree).  Errors as bsp_spmm_host; an error of the enqueued
 * work is reported by the synchronisation or by bsp_check.
 */
bsp_status_t bsp_spmm_host_async(bsp_handle_t h, const void *X_host, int64_t N,
                                 void *Y_host, bsp_stream_t stream);

/*
 * Footprint of the encoded weight in bytes, exactly
 *   Stor = 4*(NGT+1) + 8*NBT + B_v*NNZ   (B_v = 2 fp16, 1 int8),
 * the closed form on the SpInfer page ("How TCA-BME addresses the indexing
 * overhead").  The 16 B of tail slack of the values allocation is not
 * counted.
 */
bsp_status_t bsp_storage_bytes(bsp_handle_t h, uint64_t *bytes);

/*
 * Compression ratio CR = B_v*M*K / Stor ("Unified Static-Dynamic Pruning
 * for Efficient LLM Inference", eq. (1), which is written for fp16 with
 * B_v = 2; int8 handles use B_v = 1, the same-dtype dense size).
 */
bsp_status_t bsp_cr(bsp_handle_t h, double *cr);

/* Shapes, counts and device pointers of the encoded arrays (read only):
 * the bitmaps, offsets and values of the format of "SpInfer: How bitmaps
 * make sparse LLMs actually fast", section "How TCA-BME addresses the
 * indexing overhead". */
bsp_status_t bsp_info(bsp_handle_t h, bsp_info_t *out);

/*
 * Copy the three encoded arrays into caller buffers (device memory, or any
 * memory cudaMemcpyAsync with cudaMemcpyDefault accepts): bitmaps u64
 * [NBT], offsets u32 [NGT+1], values [NNZ] elements.  Any pointer may be
 * NULL to skip that array.  Ordered on `stream`; does not synchronise.
 */
bsp_status_t bsp_export(bsp_handle_t h, uint64_t *bitmaps, uint32_t *offsets,
                        void *values, bsp_stream_t stream);

/*
 * Build a handle from an existing encoding (for instance one cached on disk
 * after bsp_export): copies bitmaps u64 [Mp*Kp/64], offsets u32
 * [Mp/64 * Kp/64 + 1] and values [nnz] elements (Mp, Kp: M, K rounded up
 * to multiples of 64) from device or host memory (anything cudaMemcpyAsync
 * with cudaMemcpyDefault accepts) into arrays the new handle owns.  The
 * copy is validated on the device (offsets[0] == 0, each GroupTile's
 * offset step == the popcount of its bitmaps, no bit set in the zero
 * padding, last offset == nnz) before any kernel can read it; an
 * inconsistent encoding returns
 * BSP_ERR_INVALID_ARG and no handle.  Synchronises `stream`; the caller's
 * arrays may be freed when it returns.
 */
bsp_status_t bsp_import(const uint64_t *bitmaps, const uint32_t *offsets,
                        const void *values, bsp_dtype_t dtype, int64_t M,
                        int64_t K, uint64_t nnz, bsp_stream_t stream,
                        bsp_handle_t *out);

/*
 * Synchronise `stream` and report device-side failures of earlier calls on
 * this handle: every wait inside the kernels is bounded, and a wait that
 * gives up makes its kernel store BSP_ERR_TIMEOUT in the handle's error
 * word and return early (its output is then incomplete).  Returns that
 * status (and clears it), or BSP_OK.
 */
bsp_status_t bsp_check(bsp_handle_t h, bsp_stream_t stream);

/*
 * Decode back to dense: W_out device row-major [M][K] (fp16 or int8 bits),
 * 16-B aligned.  Each element is the value at offsets[t] + (values of the
 * earlier BTs of its GT) + the masked popcount of its BT's bitmap, or 0
 * when its bit is clear ("SpInfer: How bitmaps make sparse LLMs actually
 * fast", sections "How TCA-BME addresses the indexing overhead" and "Shared
 * Memory Bitmap Decoding (SMBD)").  decode(encode(W)) == W bit for bit.
 */
bsp_status_t bsp_decode(bsp_handle_t h, void *W_out, bsp_stream_t stream);

/*
 * Largest M that bsp_spmm_noalloc accepts.  Its scratch is a fixed
 * [BSP_DECODE_MAX_N][BSP_NOALLOC_MAX_M] fp32 workspace plus one counter
 * per 64 rows: about 2 MiB that every GPU which loads the library keeps
 * until the process exits.
 */
#define BSP_NOALLOC_MAX_M 32768

/*
 * bsp_spmm_noalloc: Y = W * X on the decode path (1 <= N <= 16) without
 * allocating anything.  The pages have no counterpart: this exists for
 * callers that cannot call cudaMalloc, such as an operator that a host
 * framework gives only its input and output buffers, a real-time loop in
 * which allocation (and the device synchronisation of cudaFree) is not
 * allowed, or code whose device memory must all come from an arena that a
 * direct cudaMalloc would bypass.  Such a caller encodes once (bsp_encode)
 * and keeps copies of the encoded arrays in its own memory (bsp_export), or
 * receives them already encoded.
 *   bitmaps  device u64 [M*K/64], 16-B aligned.
 *   offsets  device u32 [M/64 * K/64 + 1], 4-B aligned.
 *   values   device [NNZ] fp16 or int8, 16-B aligned, and readable for at
 *            least 16 bytes past the last value (bulk copies read whole
 *            16-B chunks); the slack bytes' contents do not matter.
 *   X, Y     device [N][K] and [N][M] as for bsp_spmm (fp16 -> fp16,
 *            int8 -> int32), 16-B aligned.
 *   M, K     multiples of 64, M <= BSP_NOALLOC_MAX_M; N in 1..16.  Larger
 *            M or N returns BSP_ERR_SHAPE before any device work.
 * The split-K scratch is one array compiled into the library, shared by
 * every call on a device; each call first clears the part it uses (on
 * `stream`), so calls that overlap on the GPU (different streams, or other
 * threads) race and must not be issued.  The first call on a device, with
 * that device current, looks up the array's device address and zeroes it
 * synchronously: make that first call before any stream capture.  The call
 * runs the kernels bsp_spmm runs for the same dtype and N (fp16 N <= 2:
 * GT-per-warp CUDA-core kernel; N >= BSP_TUNE_NARROW_MIN_N (fp16) or
 * BSP_TUNE_NARROW_MIN_N_I8 (int8): the narrow tcgen05 kernel and its
 * finishing kernel; the N between: the CUDA-core team kernel), with
 * GroupTile stages sized for dense GroupTiles
 * (it does not inspect the arrays), so the results equal bsp_spmm's within
 * the fp16 rounding bound (int8: exactly).  A device-side wait that gives
 * up leaves Y incomplete and is not reported here (bsp_spmm with bsp_check
 * reports it).
 */
bsp_status_t bsp_spmm_noalloc(const uint64_t *bitmaps, const uint32_t *offsets,
                              const void *values, bsp_dtype_t dtype, int64_t M,
                              int64_t K, const void *X, int64_t N, void *Y,
                              bsp_stream_t stream);

/* ------------------------------------------------------------------------
 * IE-BME: the low-bit union-bitmap format ("UnionSparse", sections
 * "IE-BME", "Area Partitioning", "Shared Union Mask", "IE-BME Storage
 * Layout") and its decode-path product with LSPD decoding (section
 * "Low-Bit Shared-Memory Parallel Decoding").
 *
 * Local tiles (LTs) of 64 x 64 over M and K zero-padded to multiples of 64,
 * row-major; each LT cut into 2 x 2 areas of 32 x 32 (area a = 2 ra + ca).
 * Position (i, j) of the 32 x 32 logical grid groups the four values
 * W[64 ti + 32 ra + i][64 tj + 32 ca + j]; its union-mask bit is 1 iff one
 * of them is nonzero.  Arrays:
 *   masks    u64 [NLT * 16]  each LT's mask row-major, leftmost position in
 *                            the least significant bit (row i = bits
 *                            32 i .. 32 i + 31)
 *   offsets  u32 [NLT + 1]   value counts: offsets[t + 1] - offsets[t] = 4 P_t,
 *                            P_t = active positions of LT t
 *   values   the four area streams of each LT: value index
 *            offsets[t] + a P_t + rank (rank = active positions before (i, j)
 *            in row-major order), zeros kept inside active groups; int8, or
 *            int4 two per byte (value e in byte e / 2, low nibble first, two's
 *            complement).
 * Storage = 4 (NLT + 1) + 128 NLT + ceil(bits * total values / 8) bytes.
 * ------------------------------------------------------------------------ */
typedef struct bsp_union *bsp_union_t;

typedef struct {
    int64_t M, K;
    int32_t bits;          /* 4 or 8                                          */
    int32_t lt;            /* local tile side: 64                             */
    int32_t areas_r, areas_c; /* 2, 2                                         */
    int32_t device;
    int64_t NLT;           /* local tiles of the padded grid                  */
    uint64_t nnz;          /* nonzero weights                                 */
    uint64_t total_values; /* stored values (offsets[NLT])                    */
    uint64_t value_bytes;  /* bytes of the packed values                      */
    const uint64_t *masks;    /* device, [NLT * 16]                           */
    const uint32_t *offsets;  /* device, [NLT + 1]                            */
    const uint8_t *values;    /* device, [value_bytes] (+32 B slack)          */
    int32_t reordered;        /* 1: rows reordered per LT (bsp_union_encode_reordered) */
} bsp_union_info_t;

/*
 * Encode an integer weight into IE-BME on the device.
 *   W      device int8 [M][K], values in the signed `bits`-bit range
 *          (bits 4: -8..7, BSP_ERR_INVALID_ARG otherwise), 16-B aligned.
 *   M, K   M >= 1, K a multiple of 16; bits = 4: K < 2^21, so that the
 *          W4A4 product's int32 accumulation of 16 w x stays exact
 *          (BSP_ERR_SHAPE otherwise).
 *   stream ordered on it; synchronises it (sizes the values array), so W may
 *          be freed on return.
 *   out    a new handle owning its device arrays and an int32 split-K
 *          workspace [16][M].
 */
bsp_status_t bsp_union_encode(const int8_t *W, int bits, int64_t M, int64_t K,
                              bsp_stream_t stream, bsp_union_t *out);

/*
 * The same with bitmap-aware row reordering ("UnionSparse", "Bitmap-aware
 * row reordering"): each LT's 64 rows are regrouped into the 32 pairs of
 * its logical rows so as to activate fewer union-mask entries, the LT is
 * encoded in that row order, and the permutation is kept with it
 * (u8 [NLT][64]: place k of the reordered LT holds row perm[k] of the LT).
 * Products write Y in the original row order.  The pairing is found on the
 * host (offline): the better of the identity pairing and a greedy pairing,
 * each improved by pair swaps (the page's exact subset DP needs 2^64 states
 * at 64 rows; bsp_reorder_rows runs it on small tiles).  Synchronises stream.
 */
bsp_status_t bsp_union_encode_reordered(const int8_t *W, int bits, int64_t M, int64_t K,
                                        bsp_stream_t stream, bsp_union_t *out);

/* Copy of the per-LT row permutations of a reordered handle into perms
 * (u8 [NLT * 64], host or device); BSP_ERR_INVALID_ARG if not reordered. */
bsp_status_t bsp_union_export_perms(bsp_union_t h, uint8_t *perms, bsp_stream_t stream);

/*
 * Row reordering of one tile, on the host ("UnionSparse", "Grouped Cost
 * Formulation", "Grouped Subset Dynamic Programming").
 *   tile   host int8 [H][KL]; rows are grouped into groups of RA, the KL
 *          columns into KL / CA grouped columns (column j, w + j, ... of the
 *          C_A column areas, w = KL / CA <= 64).
 *   exact  1: the page's subset DP, the minimum grouped cost (H <= 20);
 *          0: the pairing heuristic of bsp_union_encode_reordered (RA = 2).
 *   perm   [H] the canonical permutation (rows ascending in a group, groups
 *          in lexicographic order, taken partition-wise); cost: its grouped
 *          cost (the union-mask entries it activates).
 * BSP_ERR_SHAPE for sizes outside those limits.
 */
bsp_status_t bsp_reorder_rows(const int8_t *tile, int H, int KL, int RA, int CA, int exact,
                              int32_t *perm, int64_t *cost);

/* Free a union handle (synchronises the device first). */
bsp_status_t bsp_union_destroy(bsp_union_t h);

/*
 * Y = W * X, exact int32 accumulation ("UnionSparse" W8A8 / W4A4: the int4
 * activations are int8 values in -8..7).  X device int8 [N][K], Y device
 * int32 [N][M], both 16-B aligned; N >= 1 (runs in blocks of 16 columns).
 * For a 4-bit handle X must hold values in -8..7: the product accumulates
 * 16 w x in int32 and divides once at the end, which is exact only for
 * int4 activations; X is not checked, and other values give undefined
 * results.
 * The decode-path kernel on CUDA cores (dp4a); calls on one handle must be
 * serialised on one stream.  A device-side wait that gives up leaves Y
 * incomplete and is reported by bsp_union_check.
 */
bsp_status_t bsp_union_spmm(bsp_union_t h, const int8_t *X, int64_t N, int32_t *Y,
                            bsp_stream_t stream);

/* Bytes of the three arrays (the closed form above). */
bsp_status_t bsp_union_storage_bytes(bsp_union_t h, uint64_t *bytes);

/* Shape, counts and device pointers of the arrays. */
bsp_status_t bsp_union_info(bsp_union_t h, bsp_union_info_t *out);

/* Copies of the arrays (any of the pointers may be NULL), ordered on stream. */
bsp_status_t bsp_union_export(bsp_union_t h, uint64_t *masks, uint32_t *offsets,
                              uint8_t *values, bsp_stream_t stream);

/* W back from the arrays into device int8 [M][K] (round trip). */
bsp_status_t bsp_union_decode(bsp_union_t h, int8_t *W_out, bsp_stream_t stream);

/* Synchronise stream and report (then clear) a device-side wait that gave up. */
bsp_status_t bsp_union_check(bsp_union_t h, bsp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSP_H */
