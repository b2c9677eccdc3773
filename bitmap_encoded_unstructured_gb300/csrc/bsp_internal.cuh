// Internal declarations shared by the library's translation units.
// Nothing here is part of the public C ABI (include/bsp.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/bsp.h"

#define BSP_MAGIC 0xB5B17A9Eu

struct bsp_handle {
    uint32_t magic;
    int device;
    bsp_dtype_t dtype;
    int64_t M, K;         // logical shape of W (K a multiple of 8, of 16 for int8)
    int64_t Mp, Kp;       // M, K rounded up to multiples of 64: the zero-padded grid of the format
    int64_t NGT, NBT;     // GroupTiles (64x64), BitmapTiles (8x8) of the padded grid
    uint64_t NNZ;
    uint32_t max_gt_nnz;  // largest nonzero count of one GT (sizes the decode stages)
    uint64_t* bitmaps;    // [NBT]
    uint32_t* offsets;    // [NGT + 1]
    void* values;         // [NNZ] elements + >= 16 B zeroed tail slack
    size_t values_alloc;  // bytes allocated for values
    // split-K workspace of the decode path: [BSP_DECODE_MAX_N][M] fp32 or
    // int32, all zero between calls (the last arriving CTA of a row strip
    // reads and clears its slice); one arrival counter per 64-row strip.
    void* ws;
    uint32_t* counters;
    // deterministic split-K (bsp_set_deterministic): fp16 partial sums per
    // split, [det_slots][BSP_DECODE_MAX_N][M] fp32, allocated when first
    // switched on; det_slots bounds the split count in that mode
    int deterministic;
    float* ws_det;
    int det_slots;
    // device error word: a kernel whose bounded wait gave up stores
    // BSP_ERR_TIMEOUT here; bsp_check reads and clears it
    int* err;
    int num_sms;
    // Tiled-CBC column index (bsp_build_column_index), or null: GTiles of
    // 256 x 64, TileOffset u32 [NGT + 1], ColInfo u32 [NGT * 64], bitmaps
    // u64 [NGT * 64 * 4], values [NNZ] (+16 B slack); cbc_tr x cbc_tc GTiles
    uint32_t* cbc_offsets;
    uint32_t* cbc_colinfo;
    uint64_t* cbc_bitmaps;
    void* cbc_values;
    int64_t cbc_tr, cbc_tc;
    // staging for bsp_spmm_host, grown on demand
    void* stage_x;
    size_t stage_x_bytes;
    void* stage_y;
    size_t stage_y_bytes;
};

static inline int bsp_elem_bytes(bsp_dtype_t d) { return d == BSP_INT8 ? 1 : 2; }

// Output modes of the decode-path kernel.
enum bsp_out_mode { BSP_OUT_F16 = 0, BSP_OUT_I32 = 1, BSP_OUT_F32_SCALED = 2 };

// ---- encoder / decoder (encode.cu) ----
bsp_status_t bsp_run_encode(bsp_handle* h, const void* W, cudaStream_t s);
bsp_status_t bsp_run_decode(const bsp_handle* h, void* W_out, cudaStream_t s);
// offsets[0..n] = exclusive prefix sums of counts[0..n-1] (one block, on s);
// *overflow (device) is set when a sum does not fit uint32.
bsp_status_t bsp_exclusive_scan_u32(const uint32_t* counts, int64_t n, uint32_t* offsets, int* overflow,
                                    cudaStream_t s);
// Check that offsets and bitmaps agree (imported arrays) and set
// h->max_gt_nnz; synchronises s.
bsp_status_t bsp_run_validate(bsp_handle* h, cudaStream_t s);

// ---- IE-BME row reordering (union_reorder.cu), host ----
// act[r]: grouped activity of row r of a tile of H rows (bit j = grouped
// column j); writes the canonical permutation perm[H] of the optimal (exact:
// subset DP, H <= 20) or heuristic (R_A = 2 pairing) grouping into groups of
// RA rows and returns its cost.
int64_t bsp_reorder_rows_act(const uint64_t* act, int H, int RA, int exact, int32_t* perm);

// ---- CUDA-core decode-path product (spmm_decode.cu) ----
// Everything the decode kernel reads and writes besides X and Y: the
// encoded arrays, the shape, and the split-K scratch (workspace
// [BSP_DECODE_MAX_N][M] fp32/int32 that is all zero between calls, one
// arrival counter per 64-row strip, zeroed; an error word).
struct bsp_decode_problem {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const void* values;
    bsp_dtype_t dtype;
    int64_t M, K;         // logical shape: Y rows, X row length
    int64_t Mp, Kp;       // padded grid: Mp / 64 row strips, Kp / 64 GT columns
    uint32_t max_gt_nnz;  // bound on the nonzeros of one GT (4096: unknown)
    int device, num_sms;
    void* ws;
    uint32_t* counters;
    int* err;
    // deterministic split-K: [det_slots][N][M] fp32 slots, or null (atomic
    // accumulation into ws)
    float* ws_det = nullptr;
    int det_slots = 0;
    uint64_t values_bytes = 0;  // bytes allocated for values (0: unknown)
};

bsp_decode_problem bsp_problem_of(const bsp_handle* h);

// X: [N][K] (fp16 or int8), N in 1..BSP_DECODE_MAX_N.  Output by mode:
// F16 -> Y half [N][M]; I32 -> Y int32 [N][M]; F32_SCALED -> Y float [N][M]
// with row_scale[M].  skip_zero_octets: spMspV mode (N must be 1), where
// activations with |x| <= tau are pruned (tau = 0: exact zeros).
bsp_status_t bsp_run_spmm_decode(const bsp_decode_problem& p, const void* X, int N,
                                 void* Y, bsp_out_mode mode,
                                 const float* row_scale, bool skip_zero_octets,
                                 cudaStream_t s, float tau = 0.0f);

// Split-K factor chosen for a problem (exposed for tests and tuning).
int bsp_decode_splits(const bsp_decode_problem& p, int N);
// Largest split count the decode kernels (and the narrow kernel) choose for a problem at any N
// (ignoring BSP_SPLITK): the slot count of the deterministic workspace.
int bsp_decode_split_cap(const bsp_decode_problem& p);

// ---- tcgen05 prefill-path product (spmm_prefill.cu), fp16 only ----
// X: [N][K] fp16, Y: [N][M] fp16, any N >= 1 (used for N > BSP_DECODE_MAX_N).
bsp_status_t bsp_run_spmm_prefill(const bsp_decode_problem& p, const void* X, int64_t N, void* Y,
                                  cudaStream_t s);

// ---- tcgen05 narrow kernel (spmm_narrow.cu), fp16 or int8, 1 <= N <= 16 ----
// Persistent, balanced over the SM slots; tiles split between CTAs meet in
// the decode problem's workspace (zero between calls, fp32 [M][16] here;
// int32 for int8, whose tiles of more than 16 GT columns meet there too)
// or, fp16 in deterministic mode, in its slots ([slots][M][16]), and a
// second kernel converts them.  int8: X int8 [N][K], Y int32 [N][M], exact.
bsp_status_t bsp_run_spmm_narrow(const bsp_decode_problem& p, const void* X, int64_t N, void* Y,
                                 cudaStream_t s);
// Slots the deterministic mode needs for the automatic CTA count: the
// largest number of CTAs that share one tile.
int bsp_narrow_det_slots(const bsp_decode_problem& p);

// ---- Tiled-CBC column index and its spMspV (tiled_cbc.cu) ----
// Build the index from the handle's arrays (allocates; synchronises s).
bsp_status_t bsp_run_build_cbc(bsp_handle* h, cudaStream_t s);
// y = W x' over the index, columns with |x| <= tau skipped (tau = 0: exact
// zeros); fp16 -> fp16 y, int8 -> int32 y.
bsp_status_t bsp_run_spmspv_cbc(const bsp_handle* h, const void* x, void* y, float tau, cudaStream_t s);

// ---- process-wide tuning (bsp_tuning.cu) ----
// Tuning knobs of the dispatch, read once per process from the environment
// (BSP_SPLITK, BSP_NARROW_CTAS, BSP_UNION_SPLITK, BSP_NARROW_MIN_N,
// BSP_PF_KSPLIT, BSP_PF_SC) on first use and changed afterwards only by
// bsp_set_tuning.  0 means "automatic" for the split counts and the C ring
// depth; BSP_TUNE_PREFILL_KSPLIT is -1 (automatic), 0 or 1.
int64_t bsp_tune(bsp_tune_t knob);
// Smallest N (<= BSP_DECODE_MAX_N) that runs the tcgen05 narrow kernel for
// weights of this dtype (BSP_TUNE_NARROW_MIN_N, BSP_TUNE_NARROW_MIN_N_I8).
int64_t bsp_narrow_min_n(bsp_dtype_t dtype);
// Spin cap of the kernels' bounded waits, and whether producers skip their
// first copies (a wait that runs out, for the timeout tests).  Both are
// fixed (bspx::kSpinCap, no skipping) unless the library was built with
// BSP_TESTING (libbsp_test.so), where bsp_testing.h can change them.
uint32_t bsp_spin_cap();
int bsp_test_stall();

#include <mutex>
// Per-device one-time setup of a kernel's launch attributes (opt-in
// shared memory), safe when several host threads make their first call at
// the same time.  run() returns the setter's error, and tries again on the
// next call if it failed.
struct bsp_attr_once {
    std::mutex mu;
    bool done[64] = {};
    template <class F>
    bool run(int device, F set)
    {
        if (device < 0 || device >= 64) return false;
        std::lock_guard<std::mutex> g(mu);
        if (!done[device]) done[device] = set() == cudaSuccess;
        return done[device];
    }
};
