// Narrow product Y = W * X for 1 <= N <= 16 on the 5th-generation tensor
// cores, the decoded weight tile held in tensor memory: fp16 weights and X,
// or int8 weights and X multiplied as their exact fp16 copies (int32 Y).
//
// Method: "load as sparse, compute as dense" ("Unified Static-Dynamic
// Pruning for Efficient LLM Inference", section 4.3; "SpInfer: How bitmaps
// make sparse LLMs actually fast", sections "Shared Memory Bitmap Decoding
// (SMBD)" and "The async pipeline").  The compressed GroupTiles stream into
// shared memory; decoder warps expand them into a dense fp16 tile and one
// MMA of N = 16 per K = 16 multiplies it by the X tile.  At N <= 16 the
// MMAs are almost free: the decode (one predicated shared-memory load per
// position) sets the pace, so everything here serves the decoders.
//
// The decoded tile goes to tensor memory (tcgen05.st), not to shared
// memory: tcgen05.mma reads its A operand from there, so the A tile costs
// no shared-memory bandwidth at all (neither the decoders' stores nor the
// MMA's operand reads), leaving the shared-memory pipes to the value loads.
// tcgen05.st lets warp w write only TMEM lanes 32 (w % 4) .. + 31, and A's
// lane is the row, so a decoder warp owns 32 consecutive rows: lane l row
// 32 (w % 4) + l of the 128-row tile, all eight octets (row-bytes) of the
// step's GT column, 8 x 8 positions per lane per step.
//
// Work: a 128-row tile of W (two GT row strips) times the 16 columns of Y
// takes KT steps, one GT column (K = 64) each.  The kernel is persistent and
// balanced (stream-K): CTA c of P takes the steps [c T / P, (c + 1) T / P)
// of the T = tiles x KT steps in tile-major order, so every CTA has the same
// work and the pipeline stays full across tile boundaries.  A CTA
// accumulates each tile it touches (a segment) in one of two TMEM
// accumulators, alternating, so the epilogue of one segment overlaps the
// MMAs of the next.  A tile covered by one segment is written to Y directly;
// the segments of a tile split between CTAs add their fp32 partial sums into
// the workspace (vector reductions, fire and forget), or store them to
// per-segment slots in deterministic mode, and a small second kernel,
// launched as a programmatic dependent of the first, converts those tiles
// to fp16 (and clears the workspace).  The fp16 product kernel is itself
// launched as a programmatic dependent of whatever precedes it on the
// stream: its prologue (tensor memory, barriers, the first ring of the
// encoded weight's copies, which no kernel writes after encoding) overlaps
// the tail of the previous kernel.  Every warp waits for that kernel before
// it reads X, writes Y or the workspace, or starts a bounded wait that
// depends on it, so no poll cap counts the time the previous kernel takes.
//
// int8: values are 16 per 16-B chunk; each stored value is decoded into
// its fp16 copy (exact), the B producer converts each int8 X tile (TMA into
// a staging buffer) into the fp16 X stage, and the accumulator restarts
// every RUN_I8 steps of a segment so that every fp32 partial sum stays an
// exact integer; each run is added as int32 (the tile's rows straight to Y
// when the tile is one run of one CTA, else into the int32 workspace).  The
// int8 kernels are launched in plain stream order.  Warps:
//   0       C producer: bitmaps + value spans of the step's two GTs (bulk
//           copies) into the C ring (the rest of shared memory, stages
//           sized for the densest GT)
//   1       TMEM allocation; MMA issuer (tcgen05.mma.cta_group::1.kind::f16,
//           A from tensor memory, B = the X tile in shared memory, M = 128,
//           N = 16, K = 16, four per step)
//   2       B producer: the 16 x 64 X tile of each step by TMA (rows past N
//           read as zeros); int8: converted to fp16 by this warp
//   3 ..    decoders, NG groups of four warps (one per TMEM lane quadrant);
//           group g takes the CTA's steps g, g + NG, ... and owns A stage g
//           in tensor memory.  Per step a warp scans the popcounts of its 32
//           BitmapTiles (its half of a GT), writes their row starts to a
//           private table, then decodes its 256 row-bytes.  The group that
//           decodes the last step of a segment is also its epilogue
//           (tcgen05.ld of the accumulator, then Y or the workspace).
// Every wait is bounded; a wait that gives up stores BSP_ERR_TIMEOUT in the
// error word, and the CTA still drains its copies, waits for its MMAs and
// frees its tensor memory before it exits.
#include "bsp_internal.cuh"
#include "bsp_ptx.cuh"
#include "bsp_bits.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <type_traits>

// split model: fixed cost of a CTA in GT-column steps
#ifndef BSP_NARROW_CTA_COST
#define BSP_NARROW_CTA_COST 6
#endif
// resident CTAs per SM (1 or 2): shared memory and registers are split
// between them
#ifndef BSP_NARROW_MINB
#define BSP_NARROW_MINB 2
#endif
// decoder groups of four warps (steps in flight, A stages in tensor memory)
#ifndef BSP_NARROW_GROUPS
#define BSP_NARROW_GROUPS 3
#endif

namespace {

constexpr int BM = 128, BN = 16, BK = 64;  // tile rows, MMA columns, GT columns per step
constexpr int NG = BSP_NARROW_GROUPS;
static_assert(NG >= 1 && NG <= 6, "decoder groups");
constexpr int DEC_WARPS = 4 * NG;
constexpr int CPROD = 0, MMAW = 1, BPROD = 2, DEC0 = 3;
constexpr int WARPS = DEC0 + DEC_WARPS;
constexpr int THREADS = WARPS * 32;
[[maybe_unused]] constexpr uint32_t kSleepNs = 1000;  // suspend hint of the waiting polls (BSP_NARROW_WAIT=0)
// longest sleep between the polls of a waiting producer, MMA issuer, decoder
#ifndef BSP_NARROW_SLEEP_PROD
#define BSP_NARROW_SLEEP_PROD 256
#endif
#ifndef BSP_NARROW_SLEEP_MMA
#define BSP_NARROW_SLEEP_MMA 64
#endif
#ifndef BSP_NARROW_SLEEP_DEC
#define BSP_NARROW_SLEEP_DEC 256
#endif

constexpr int SB = 8;                      // X tile stages
constexpr int SC_MAX = 16;                 // barrier slots of the C ring
constexpr int MINB = BSP_NARROW_MINB;
static_assert(MINB == 1 || MINB == 2, "one or two CTAs per SM");
// shared memory of a CTA: all of it, or half of the SM's 228 KB less the
// 1 KB the driver reserves per resident CTA
constexpr int SMEM_MAX = MINB == 1 ? 227 * 1024 : 228 * 1024 / 2 - 1024;
constexpr int B_STAGE = BN * BK * 2;       // 2 KB
constexpr int RS_WARP = 32 * 8 * 2;        // a decoder warp's row-start table: [BT][row] u16
constexpr int XS_STAGE = BN * BK;          // an int8 X tile as it arrives (1 KB)
constexpr int OFF_B = 0;                   // 1024-B aligned (the X tiles' 128-B swizzle)
constexpr int OFF_RS = OFF_B + SB * B_STAGE;
constexpr int OFF_XS = OFF_RS + DEC_WARPS * RS_WARP;
// barriers: c_full[SC_MAX] c_empty[SC_MAX] b_full[SB] b_empty[SB] a_full[NG] a_empty[NG]
// acc_full[2] acc_empty[2] drain xs_full[2]
constexpr int NBAR = 2 * SC_MAX + 2 * SB + 2 * NG + 7;
// The rest of the layout: after two int8 X staging tiles for int8 weights.
template <bool I8>
struct Layout {
    static constexpr int OFF_BAR = OFF_XS + (I8 ? 2 * XS_STAGE : 0);
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;  // TMEM address (4 B)
    static constexpr int OFF_C = (OFF_TMEM + 16 + 127) & ~127;
    static constexpr int C_BYTES = SMEM_MAX - 1024 - OFF_C;  // 1024: slack to align the base to 1024 B
};
// int8 weights: the tensor cores multiply fp16 copies of the int8 values
// (exact), accumulating in fp32; a run of at most RUN_I8 steps sums at most
// 64 RUN_I8 products of magnitude <= 127 * 128, below 2^24, so every fp32
// partial sum is an exact integer.  Each run leaves the accumulator as int32.
constexpr uint32_t RUN_I8 = 16;
static_assert(64u * RUN_I8 * 127u * 128u < (1u << 24), "exact fp32 runs");
// tensor memory: two accumulators (16 fp32 columns each, 32 apart), then NG
// decoded A tiles of 128 lanes x 64 fp16 = 32 columns each
constexpr uint32_t D_COLS = 32;
constexpr uint32_t A_OFF = 2 * D_COLS;
constexpr uint32_t A_COLS = BK / 2;
constexpr uint32_t tmem_cols_for(uint32_t need)
{
    uint32_t c = 32;
    while (c < need) c <<= 1;
    return c;
}
constexpr uint32_t TMEM_COLS = tmem_cols_for(A_OFF + NG * A_COLS);
static_assert(TMEM_COLS * MINB <= 512, "tensor memory of the resident CTAs");

// One C stage: two GT slots (512 B of bitmaps, then the 16-B chunks that
// hold the GT's value span, `vpc` values per chunk) and a 16-B header (the
// value shifts).  The slot is sized for the densest GT of the matrix, so the
// number of stages that fit follows the density.
constexpr uint32_t c_slot_bytes(uint32_t max_gt_nnz, uint32_t vpc)
{
    return (512u + 16u * ((max_gt_nnz + vpc - 1u) / vpc + 1u) + 127u) & ~127u;
}
constexpr uint32_t c_stage_bytes(uint32_t slot) { return (2u * slot + 16u + 127u) & ~127u; }
static_assert(Layout<true>::C_BYTES >= NG * (int)c_stage_bytes(c_slot_bytes(4096, 8)) && NG <= SC_MAX,
              "a dense C stage per decoder group");
static_assert((B_STAGE % 1024) == 0 && (OFF_RS % 16) == 0, "alignment of the X tiles and tables");

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// M = 128, N = 16.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct NarrowArgs {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const uint8_t* values;
    void* Y;                   // fp16 or (int8 weights) int32, [N][M]
    int64_t M, N, K;           // logical: Y rows, columns, X row length
    int64_t Mp, KT;            // padded grid: rows (a multiple of 64), GT columns
    int64_t T;                 // steps of the whole product: tiles x KT
    int64_t P;                 // CTAs (1 <= P <= T)
    uint32_t c_slot, c_stage;  // C ring geometry (bytes): GT slot, stage
    int sc;                    // C stages in use, NG..SC_MAX
    // partial sums of the tiles split between CTAs: fp32 [M][16] (int32 for
    // int8 weights), zero between calls (reductions; the finishing kernel
    // clears it), or in deterministic mode (fp16) the slots [slots][M][16],
    // one per segment
    float* ws;
    float* ws_det;
    int* err;
    uint32_t spin_cap;
};

// The balanced partition: CTA c owns steps [c T / P, (c + 1) T / P), so the
// owner of step x is the largest c whose range starts at or before x.
__host__ __device__ __forceinline__ int64_t part_begin(int64_t c, int64_t T, int64_t P) { return c * T / P; }
__host__ __device__ __forceinline__ int64_t step_owner(int64_t x, int64_t T, int64_t P)
{
    return ((x + 1) * P - 1) / T;
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled canonical layout: rows of 128 B, 8-row atoms of 1 KB (stride
// 1024 B between atoms), atoms 1024-B aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);       // start address
    d |= (uint64_t)1u << 16;                        // leading offset (unused for swizzled K-major)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // stride offset: 1024 B between 8-row atoms
    d |= (uint64_t)1u << 46;                        // descriptor version of sm_100
    d |= (uint64_t)2u << 61;                        // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            bspx::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bspx::smem_u32(bar))
        : "memory");
}

// D (tensor memory) += A (tensor memory, 128 lanes x 8 columns = 16 fp16
// per row) * B (shared-memory descriptor), or D = A * B when accum is 0.
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t accum)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(kIdesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bspx::smem_u32(bar))
                 : "memory");
}

// Bounded wait for phase `parity` of `bar` (at most `cap` polls).  Between
// polls a waiting thread sleeps, starting at 32 ns and doubling up to
// `max_ns`, so warps that wait (for data, for the MMAs, for a free stage)
// leave the issue slots to the decoders.
#ifndef BSP_NARROW_WAIT
#define BSP_NARROW_WAIT 1
#endif
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, uint32_t cap, uint32_t max_ns)
{
#if BSP_NARROW_WAIT == 0
    return bspx::mbar_wait_sleep(bar, parity, cap, kSleepNs);
#else
    uint32_t ns = 32;
    for (uint32_t i = 0; i < cap; ++i) {
        if (bspx::mbar_try_wait(bar, parity)) return true;
        __nanosleep(ns);
        if (ns < max_ns) ns <<= 1;
    }
    return false;
#endif
}

// Wait until the grids this one depends on (programmatic dependent launch)
// have completed and their memory is visible; returns at once otherwise.
__device__ __forceinline__ void wait_prior_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// ws[0..3] += v[0..3], one vector reduction without a return value
__device__ __forceinline__ void red_add_v4(float* ws, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(ws), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// 16 consecutive TMEM columns of this thread's lane (32x32b shape, x16).
// Whole warps only: the .aligned form runs on a reconverged warp.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 4 consecutive TMEM columns of this thread's lane from registers (32x32b
// shape, x4): one decoded row-byte.  Whole warps only (the callers run
// converged: the decode has no divergent branch).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}

// The eight positions of one BT row-byte as four words of two fp16 each
// (position 2k in the low half of word k): a set bit takes the next packed
// value (shared memory, in order), a clear bit gives 0.  The loads are plain
// predicated loads the compiler schedules; they stay after the ring-barrier
// wait, whose inline assembly clobbers memory.
__device__ __forceinline__ void decode_rowbyte(const uint16_t* vp, uint32_t byte, uint32_t* w)
{
    uint32_t h[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        h[c] = 0u;
        if (byte & (1u << c)) {
            h[c] = *vp;
            ++vp;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __byte_perm(h[2 * k], h[2 * k + 1], 0x5410);
}

// The same for int8 values: each stored value becomes its fp16 copy (exact:
// |v| <= 128).
__device__ __forceinline__ void decode_rowbyte(const int8_t* vp, uint32_t byte, uint32_t* w)
{
    uint32_t h[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        h[c] = 0u;
        if (byte & (1u << c)) {
            h[c] = __half_as_ushort(__short2half_rn((short)*vp));
            ++vp;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __byte_perm(h[2 * k], h[2 * k + 1], 0x5410);
}

__device__ __forceinline__ void red_add_s32(int* p, int v)
{
    asm volatile("red.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16 int8 values (one 16-B load) as fp16 in two 16-B chunks
__device__ __forceinline__ void i8x16_to_f16(const uint4 v, uint4& lo, uint4& hi)
{
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t x = wv[q];
        const uint32_t b0 = __half_as_ushort(__short2half_rn((short)(int8_t)(x & 0xFFu)));
        const uint32_t b1 = __half_as_ushort(__short2half_rn((short)(int8_t)((x >> 8) & 0xFFu)));
        const uint32_t b2 = __half_as_ushort(__short2half_rn((short)(int8_t)((x >> 16) & 0xFFu)));
        const uint32_t b3 = __half_as_ushort(__short2half_rn((short)(int8_t)(x >> 24)));
        o[2 * q] = b0 | (b1 << 16);
        o[2 * q + 1] = b2 | (b3 << 16);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Grid: P CTAs, persistent: CTA c takes the steps [c T / P, (c + 1) T / P)
// (step x is GT column x % KT of tile x / KT).  I8: int8 weights and X
// (the B producer converts each X tile to fp16), int32 Y, exact runs of at
// most RUN_I8 steps.
template <bool I8>
__global__ void __launch_bounds__(THREADS, MINB)
spmm_narrow_kernel(const __grid_constant__ CUtensorMap tmX, const NarrowArgs a)
{
    using L = Layout<I8>;
    constexpr uint32_t VPC = I8 ? 16u : 8u;        // values per 16-B chunk
    constexpr uint32_t RUN = I8 ? RUN_I8 : 1u;     // steps per exact run (int8 only; fp16 runs are segments)
    const uint32_t SC = (uint32_t)a.sc;
    const uint32_t SLOT = a.c_slot, C_HDR = 2 * SLOT;
    const uint32_t vchunks = (SLOT - 512) / 16;  // value chunks a slot holds
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-B alignment of the shared-window offset (the 128-B swizzle atoms)
    uint8_t* smem = smem_raw + ((1024u - (bspx::smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr uint32_t FULL = 0xFFFFFFFFu;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint64_t* c_full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    uint64_t* c_empty = c_full + SC_MAX;
    uint64_t* b_full = c_empty + SC_MAX;
    uint64_t* b_empty = b_full + SB;
    uint64_t* a_full = b_empty + SB;
    uint64_t* a_empty = a_full + NG;
    uint64_t* acc_full = a_empty + NG;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint64_t* xs_full = drain + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
    auto b_stage = [&](uint32_t s) { return smem + OFF_B + s * B_STAGE; };
    auto c_stage = [&](uint32_t s) { return smem + L::OFF_C + s * a.c_stage; };

    const int64_t M = a.M, N = a.N, T = a.T, P = a.P;
    const uint32_t KTA = (uint32_t)a.KT;  // GT columns of the grid (row pitch, steps per tile)
    const int64_t cta = blockIdx.x;
    const int64_t g0 = part_begin(cta, T, P);
    const uint32_t S = (uint32_t)(part_begin(cta + 1, T, P) - g0);  // steps of this CTA (>= 1: P <= T)
    const int64_t t0 = g0 / KTA;                                    // first tile
    const uint32_t kk0 = (uint32_t)(g0 - t0 * KTA);                 // its first GT column
    const uint32_t cap = a.spin_cap;
    // exact runs (int8): a run restarts the accumulator every RUN steps of a
    // segment.  L0: steps of the CTA's first segment; R0, RT: runs of the
    // first segment and of a whole tile
    const uint32_t L0 = min(S, KTA - kk0);
    const uint32_t R0 = I8 ? (L0 + RUN - 1) / RUN : 1u;
    const uint32_t RT = I8 ? (KTA + RUN - 1) / RUN : 1u;

    if (warp == MMAW) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         bspx::smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < SC; ++s) {
            bspx::mbar_init(c_full + s, 1);
            bspx::mbar_init(c_empty + s, 4);  // the four warps of the step's decoder group
        }
        for (int s = 0; s < SB; ++s) {
            bspx::mbar_init(b_full + s, 1);
            bspx::mbar_init(b_empty + s, 1);
        }
        for (int g = 0; g < NG; ++g) {
            bspx::mbar_init(a_full + g, 4);
            bspx::mbar_init(a_empty + g, 1);
        }
        for (int d = 0; d < 2; ++d) {
            bspx::mbar_init(acc_full + d, 1);
            bspx::mbar_init(acc_empty + d, 4);  // the four warps of an epilogue
        }
        bspx::mbar_init(drain, 1);
        bspx::mbar_init(xs_full, 1);
        bspx::mbar_init(xs_full + 1, 1);
        bspx::fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    bool failed = false;

    if (warp == CPROD) {
        // ---------------- C producer: the two GTs of each step, up to SC steps ahead
        int64_t t = t0;
        uint32_t k = kk0;
        uint32_t offa = 0, offb = 0;
        uint32_t wbase = 0;
        uint32_t s = 0, ph = 0;  // stage and its phase parity
        uint32_t i = 0;          // steps issued
        for (; i < S; ++i) {
            // a stage frees only once the MMAs run, which wait for the
            // previous kernel: wait for it here (unbounded, it completes on
            // its own) so that no bounded wait below counts that time
            if (i == SC) wait_prior_grids();
            if (i >= SC && !__all_sync(FULL, wait_bar(c_empty + s, ph ^ 1u, cap, BSP_NARROW_SLEEP_PROD))) {
                failed = true;
                break;
            }
            const int64_t ta = 2 * t * KTA, tb = ta + KTA;  // the tile's two GT rows
            const bool has_b = (2 * t + 1) * 64 < a.Mp;
            if (i == 0 || k == 0 || k - wbase >= 31) {
                // window of offsets: lane j holds offsets[row + wbase + j] (j <= KT: the row's end)
                wbase = k;
                const uint32_t j = wbase + lane;
                offa = (j <= KTA) ? __ldg(a.offsets + ta + j) : 0u;
                offb = (has_b && j <= KTA) ? __ldg(a.offsets + tb + j) : 0u;
            }
            const int w = (int)(k - wbase);
            const uint32_t oa0 = __shfl_sync(FULL, offa, w), oa1 = __shfl_sync(FULL, offa, w + 1);
            const uint32_t ob0 = __shfl_sync(FULL, offb, w), ob1 = __shfl_sync(FULL, offb, w + 1);
            if (lane == 0) {
                uint8_t* st = c_stage(s);
                uint32_t* hdr = reinterpret_cast<uint32_t*>(st + C_HDR);
                const uint32_t cha = oa0 / VPC, chb = ob0 / VPC;
                uint32_t nca = (oa1 + VPC - 1) / VPC - cha, ncb = has_b ? (ob1 + VPC - 1) / VPC - chb : 0u;
                if (nca > vchunks || ncb > vchunks) {  // a GT denser than the handle recorded
                    atomicExch(a.err, (int)BSP_ERR_INTERNAL);
                    nca = min(nca, vchunks);
                    ncb = min(ncb, vchunks);
                }
                hdr[0] = oa0 - cha * VPC;
                hdr[1] = ob0 - chb * VPC;
                uint32_t bytes = 512 + nca * 16;
                if (has_b) bytes += 512 + ncb * 16;
                bspx::mbar_arrive_expect_tx(c_full + s, bytes);
                bspx::bulk_g2s(st, a.bitmaps + (ta + k) * 64, 512, c_full + s);
                if (nca) bspx::bulk_g2s(st + 512, a.values + (int64_t)cha * 16, nca * 16, c_full + s);
                if (has_b) {
                    bspx::bulk_g2s(st + SLOT, a.bitmaps + (tb + k) * 64, 512, c_full + s);
                    if (ncb) bspx::bulk_g2s(st + SLOT + 512, a.values + (int64_t)chb * 16, ncb * 16, c_full + s);
                }
            }
            if (++s == SC) { s = 0; ph ^= 1u; }
            if (++k == KTA) { k = 0; ++t; }
        }
        // let the last copies land before the CTA can exit (bounded)
        for (uint32_t j = (i > SC ? i - SC : 0); j < i; ++j)
            bspx::mbar_wait_bounded(c_full + (j % SC), (j / SC) & 1u, cap);
    } else if (warp == BPROD && I8) {
        // ---------------- B producer, int8 X: the 16 x 64 int8 tile of step i
        // arrives by TMA in staging buffer i % 2 (the next one is in flight
        // meanwhile); lane l converts row l / 2, half l % 2 (32 values) to
        // fp16 into the 128-B-swizzled X stage (16-B chunk c of row r at
        // chunk position c ^ (r % 8)), then the stage is handed to the MMAs
        // (X may be written by the previous kernel on the stream)
        wait_prior_grids();
        uint8_t* xs = smem + OFF_XS;
        auto x_issue = [&](uint32_t i, uint32_t kx) {
            if (lane == 0) {
                bspx::mbar_arrive_expect_tx(xs_full + (i & 1u), (uint32_t)XS_STAGE);
                tma_load_2d(xs + (i & 1u) * XS_STAGE, &tmX, (int)(kx * BK), 0, xs_full + (i & 1u));
            }
        };
        uint32_t s = 0, ph = 0;
        uint32_t k = kk0;
        uint32_t i = 0;
        x_issue(0, kk0);
        const int r = lane >> 1, hh = lane & 1;
        for (; i < S; ++i) {
            if (i + 1 < S) x_issue(i + 1, k + 1 == KTA ? 0u : k + 1);  // its buffer was converted at step i - 1
            bool ok = wait_bar(xs_full + (i & 1u), (i >> 1) & 1u, cap, BSP_NARROW_SLEEP_PROD);
            if (i >= (uint32_t)SB) ok = ok && wait_bar(b_empty + s, ph ^ 1u, cap, BSP_NARROW_SLEEP_PROD);
            if (!__all_sync(FULL, ok)) {
                failed = true;
                break;
            }
            const uint4* src = reinterpret_cast<const uint4*>(xs + (i & 1u) * XS_STAGE + r * BK + hh * 32);
            uint8_t* dst = b_stage(s) + r * 128;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint4 lo, hi;
                i8x16_to_f16(src[h2], lo, hi);
                const int c0 = 4 * hh + 2 * h2;  // fp16 chunk of the row
                *reinterpret_cast<uint4*>(dst + ((c0 ^ (r & 7)) * 16)) = lo;
                *reinterpret_cast<uint4*>(dst + (((c0 + 1) ^ (r & 7)) * 16)) = hi;
            }
            // the writes are seen by the tensor cores (async proxy), and the
            // staging buffer may be refilled by TMA
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) bspx::mbar_arrive(b_full + s);
            if (++s == (uint32_t)SB) { s = 0; ph ^= 1u; }
            if (++k == KTA) k = 0;
        }
        // staging copies still in flight (a wait gave up) land before the
        // CTA can exit (bounded)
        for (uint32_t q = i; q < S && q <= i + 1; ++q)
            bspx::mbar_wait_bounded(xs_full + (q & 1u), (q >> 1) & 1u, cap);
    } else if (warp == BPROD) {
        // ---------------- B producer: one 16 x 64 X tile per step by TMA
        // (X may be written by the previous kernel on the stream)
        wait_prior_grids();
        uint32_t s = 0, ph = 0;
        uint32_t k = kk0;
        uint32_t i = 0;
        for (; i < S; ++i) {
            if (i >= (uint32_t)SB &&
                !__all_sync(FULL, wait_bar(b_empty + s, ph ^ 1u, cap, BSP_NARROW_SLEEP_PROD))) {
                failed = true;
                break;
            }
            if (lane == 0) {
                bspx::mbar_arrive_expect_tx(b_full + s, (uint32_t)B_STAGE);
                tma_load_2d(b_stage(s), &tmX, (int)(k * BK), 0, b_full + s);
            }
            if (++s == (uint32_t)SB) { s = 0; ph ^= 1u; }
            if (++k == KTA) k = 0;
        }
        for (uint32_t j = (i > (uint32_t)SB ? i - SB : 0); j < i; ++j)
            bspx::mbar_wait_bounded(b_full + (j % SB), (j / SB) & 1u, cap);
    } else if (warp == MMAW) {
        // ---------------- MMA issuer: step i reads A stage i % NG and
        // accumulates into buffer (segment & 1); the first MMA of a segment
        // overwrites the buffer, which the epilogue two segments back must
        // have read
        uint32_t sb = 0, pb = 0;
        uint32_t k = kk0, seg = 0;
        wait_prior_grids();  // the X tiles come after it (see the producer)
        for (uint32_t i = 0; i < S && !failed; ++i) {
            const uint32_t g = i % NG;
            const uint32_t pos = i < L0 ? i : k;  // step within the segment
            const bool first = I8 ? pos % RUN == 0 : (i == 0 || k == 0);
            const bool last = i + 1 == S || k + 1 == KTA || (I8 && (pos + 1) % RUN == 0);
            const uint32_t buf = seg & 1u;
            bool ok = wait_bar(a_full + g, (i / NG) & 1u, cap, BSP_NARROW_SLEEP_MMA);
            ok = ok && wait_bar(b_full + sb, pb, cap, BSP_NARROW_SLEEP_MMA);
            if (first && seg >= 2) ok = ok && wait_bar(acc_empty + buf, ((seg - 2) >> 1) & 1u, cap, BSP_NARROW_SLEEP_MMA);
            if (!__all_sync(FULL, ok)) { failed = true; break; }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t ta = tmem_base + A_OFF + g * A_COLS;
                const uint32_t td = tmem_base + buf * D_COLS;
                const uint64_t bd = smem_desc_sw128(bspx::smem_u32(b_stage(sb)));
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)  // K = 16 per MMA: 8 A columns, 32 B along the swizzled X row
                    umma_f16_ts(td, ta + (uint32_t)(8 * j), bd + (uint64_t)(2 * j), (first && j == 0) ? 0u : 1u);
                umma_commit(b_empty + sb);  // fire once the MMAs above are done
                umma_commit(a_empty + g);
                if (last) umma_commit(acc_full + buf);
            }
            __syncwarp();
            if (++sb == (uint32_t)SB) { sb = 0; pb ^= 1u; }
            if (last) ++seg;
            if (++k == KTA) k = 0;
        }
        // every MMA issued above is done before the CTA frees tensor memory
        if (lane == 0) umma_commit(drain);
        __syncwarp();
        bspx::mbar_wait_bounded(drain, 0, cap);
        __syncwarp();
    } else {
        // ---------------- decoders.  Warp: group G (its steps), TMEM lane
        // quadrant q = rows 32 q .. 32 q + 31 of the tile = half h of GT
        // gsel.  Lane l: row 32 h + l of the GT, which lies in BT row
        // (l / 8) & 1 of TCTile row l / 16 of the half; its row-byte of
        // octet o is row l % 8 of the half's BT (4 (l / 16) + o / 2) * 4 +
        // 2 (o % 2) + (l / 8) % 2 (BTs in GT order).
        const int dw = warp - DEC0;
        const uint32_t G = (uint32_t)(dw >> 2);
        const int q = warp & 3;
        const int gsel = q >> 1, h = q & 1;
        const uint32_t tq = (uint32_t)(32 * q) << 16;  // TMEM lane field of the quadrant
        const uint32_t tA = tmem_base + A_OFF + G * A_COLS + tq;
        uint16_t* rs = reinterpret_cast<uint16_t*>(smem + OFF_RS + dw * RS_WARP);
        const int ri = lane & 7;
        const int bt0 = 16 * (lane >> 4) + ((lane >> 3) & 1);  // the lane's BT of octet 0 (half-local)
        // step i = G, G + NG, ...: its tile, GT column, C stage and parity
        const uint32_t Mp32 = (uint32_t)a.Mp;
        uint32_t t = (uint32_t)t0;
        uint32_t k = kk0 + G;
        while (k >= KTA) { k -= KTA; ++t; }
        uint32_t sc = G, pc = 0;
        uint32_t it = 0;
        for (uint32_t i = G; i < S; i += NG, ++it) {
            bool ok = wait_bar(c_full + sc, pc, cap, BSP_NARROW_SLEEP_DEC);
            // the MMAs of this group's previous step read A stage G: done
            if (it == 1) wait_prior_grids();  // the MMAs wait for the previous kernel (see the producer)
            if (it > 0) ok = ok && wait_bar(a_empty + G, (it - 1) & 1u, cap, BSP_NARROW_SLEEP_DEC);
            if (!__all_sync(FULL, ok)) { failed = true; break; }
            tc_fence_after();
            const bool active = gsel == 0 || (2 * t + 1) * 64 < Mp32;  // a missing second strip: zeros
            __syncwarp();
            if (active) {
                const uint8_t* slot = c_stage(sc) + gsel * SLOT;
                // BT value bases: lane l owns BT 32 h + l (GT order = value order)
                const uint64_t* bms = reinterpret_cast<const uint64_t*>(slot);
                const uint64_t bm = bms[32 * h + lane];
                const uint32_t cnt = (uint32_t)__popcll(bm);
                uint32_t incl = cnt;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t o = __shfl_up_sync(FULL, incl, d);
                    if (lane >= d) incl += o;
                }
                uint32_t base = incl - cnt + reinterpret_cast<const uint32_t*>(c_stage(sc) + C_HDR)[gsel];
                if (h) base += __reduce_add_sync(FULL, (uint32_t)__popcll(bms[lane]));  // the first half's values
                *reinterpret_cast<uint4*>(rs + 8 * lane) = bspx::row_starts(bm, base);
                __syncwarp();
                const uint8_t* bytes = slot + 256 * h;  // byte 8 bt + r: row r of the half's BT bt
                using VT = typename std::conditional<I8, int8_t, uint16_t>::type;
                const VT* vals = reinterpret_cast<const VT*>(slot + 512);
#pragma unroll
                for (int o = 0; o < 8; ++o) {
                    const int bt = bt0 + 4 * (o >> 1) + 2 * (o & 1);
                    const uint32_t byte = bytes[8 * bt + ri];
                    uint32_t w[4];
                    decode_rowbyte(vals + rs[8 * bt + ri], byte, w);
                    tmem_st4(tA + (uint32_t)(4 * o), w);  // octet o: columns 4 o .. 4 o + 3
                }
            } else {
                // rows of a missing second strip: zeros, so that the MMA
                // reads defined values (their Y rows are not written)
                const uint32_t z[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int o = 0; o < 8; ++o) tmem_st4(tA + (uint32_t)(4 * o), z);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                bspx::mbar_arrive(a_full + G);
                bspx::mbar_arrive(c_empty + sc);
            }
            const uint32_t pos = t == (uint32_t)t0 ? i : k;  // step within the segment
            if (i + 1 == S || k + 1 == KTA || (I8 && (pos + 1) % RUN == 0)) {
                // ---------------- epilogue of the segment (int8: the run) this
                // step ends: one row of 16 columns per thread.  Its number
                // among the CTA's accumulator uses picks the buffer.
                const uint32_t seg = !I8 ? t - (uint32_t)t0
                                         : (t == (uint32_t)t0 ? pos / RUN : R0 + (t - (uint32_t)t0 - 1) * RT + k / RUN);
                const uint32_t buf = seg & 1u;
                if (!__all_sync(FULL, wait_bar(acc_full + buf, (seg >> 1) & 1u, cap, BSP_NARROW_SLEEP_DEC))) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                wait_prior_grids();  // Y and the workspace: the previous kernel is done with them
                uint32_t r[16];
                tmem_ld16(tmem_base + buf * D_COLS + tq, r);
                const int64_t m = (int64_t)t * BM + 32 * q + lane;
                if (m < M) {
                    const int64_t first = step_owner((int64_t)t * KTA, T, P);
                    const int64_t nseg = step_owner(((int64_t)t + 1) * KTA - 1, T, P) - first + 1;
                    if (I8) {
                        // exact integers: straight to Y when the tile is one
                        // run of one CTA, else added into the int32 workspace
                        int* Yi = static_cast<int*>(a.Y);
                        int* wsi = reinterpret_cast<int*>(a.ws);
                        if (nseg == 1 && RT == 1) {
#pragma unroll
                            for (int j = 0; j < BN; ++j)
                                if (j < N) Yi[j * M + m] = __float2int_rn(__uint_as_float(r[j]));
                        } else {
#pragma unroll
                            for (int j = 0; j < BN; ++j)
                                if (j < N) red_add_s32(wsi + m * 16 + j, __float2int_rn(__uint_as_float(r[j])));
                        }
                    } else if (nseg == 1) {
                        __half* Yh = static_cast<__half*>(a.Y);
#pragma unroll
                        for (int j = 0; j < BN; ++j)
                            if (j < N) Yh[j * M + m] = __float2half_rn(__uint_as_float(r[j]));
                    } else if (a.ws_det) {
                        float4* d = reinterpret_cast<float4*>(a.ws_det + ((cta - first) * M + m) * 16);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    } else {
                        // columns at or past N are exact zeros (X rows past N read as zeros)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (4 * j < N)
                                red_add_v4(a.ws + m * 16 + 4 * j, __uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                           __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) bspx::mbar_arrive(acc_empty + buf);
            }
            sc += NG;
            if (sc >= SC) { sc -= SC; pc ^= 1u; }
            k += NG;
            while (k >= KTA) { k -= KTA; ++t; }
        }
    }

    // the finishing kernel may start launching (it waits for this grid's
    // completion and memory before it reads the workspace)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (failed && lane == 0) {
        wait_prior_grids();
        atomicExch(a.err, (int)BSP_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMAW) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// Finishing kernel: Y of the tiles whose steps are split between CTAs (and,
// int8, of the tiles of several runs), from the workspace (which it clears)
// or, deterministically, from the segments' slots added in segment order.
// One thread per (row, column < N).
template <bool I8>
__global__ void __launch_bounds__(256)
spmm_narrow_finish_kernel(void* __restrict__ Y, float* __restrict__ ws, const float* __restrict__ ws_det,
                          int64_t M, int64_t N, int64_t KT, int64_t T, int64_t P)
{
    // the next product kernel may start its prologue now (it waits for this
    // grid before it touches Y or the workspace)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t total = M * N;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = e / N, n = e - m * N;
        const int64_t t = m / BM;
        const int64_t first = step_owner(t * KT, T, P);
        const int64_t nseg = step_owner((t + 1) * KT - 1, T, P) - first + 1;
        if (nseg == 1 && (!I8 || KT <= (int64_t)RUN_I8)) continue;  // written by the product kernel
        if (I8) {
            int* wsi = reinterpret_cast<int*>(ws);
            static_cast<int*>(Y)[n * M + m] = wsi[m * 16 + n];
            wsi[m * 16 + n] = 0;
            continue;
        }
        float v;
        if (ws_det) {
            v = 0.f;
            for (int64_t sgi = 0; sgi < nseg; ++sgi) v += ws_det[(sgi * M + m) * 16 + n];
        } else {
            v = ws[m * 16 + n];
            ws[m * 16 + n] = 0.f;
        }
        static_cast<__half*>(Y)[n * M + m] = __float2half_rn(v);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

namespace {

// CTAs of the narrow kernel: every resident slot (MINB per SM), at most one
// per step; BSP_TUNE_NARROW_CTAS overrides.
int64_t narrow_ctas_auto(const bsp_decode_problem& p, int64_t T)
{
    const int64_t slots = (int64_t)(p.num_sms > 0 ? p.num_sms : 1) * MINB;
    return std::max<int64_t>(1, std::min(slots, T));
}

// Largest number of CTAs sharing one tile under the balanced partition.
int64_t max_segments(int64_t tiles, int64_t KT, int64_t T, int64_t P)
{
    int64_t mx = 1;
    for (int64_t t = 0; t < tiles; ++t)
        mx = std::max(mx, step_owner((t + 1) * KT - 1, T, P) - step_owner(t * KT, T, P) + 1);
    return mx;
}

bool any_split(int64_t tiles, int64_t KT, int64_t T, int64_t P) { return max_segments(tiles, KT, T, P) > 1; }

}  // namespace

int bsp_narrow_det_slots(const bsp_decode_problem& p)
{
    const int64_t tiles = (p.Mp + BM - 1) / BM, KT = p.Kp / 64, T = tiles * KT;
    return (int)max_segments(tiles, KT, T, narrow_ctas_auto(p, T));
}

namespace {

template <bool I8>
bsp_status_t launch_narrow(const bsp_decode_problem& p, const void* X, int64_t N, void* Y, cudaStream_t s)
{
    using L = Layout<I8>;
    auto encode = get_encode_fn();
    if (!encode) return BSP_ERR_CUDA;
    // X: [N][K], K contiguous; boxes of 64 (K) x 16 rows, rows past N read
    // as zeros.  fp16: 128-B swizzle, straight into the MMA's X stage; int8:
    // unswizzled 1 KB tiles that the B producer converts
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * (I8 ? 1 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&map, I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               I8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BSP_ERR_INVALID_ARG;

    static bsp_attr_once attr;
    if (!attr.run(p.device, [] {
            return cudaFuncSetAttribute(spmm_narrow_kernel<I8>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
        }))
        return BSP_ERR_CUDA;
    const int64_t tiles = (p.Mp + BM - 1) / BM, KT = p.Kp / 64, T = tiles * KT;
    int64_t P = narrow_ctas_auto(p, T);
    if (const int64_t v = bsp_tune(BSP_TUNE_NARROW_CTAS)) P = std::min(v, T);  // tests, tuning
    // deterministic slots: one per CTA sharing a tile; fewer CTAs share less
    if (p.ws_det && !I8)  // int8 partial sums are exact integers: any order gives the same Y
        while (P > 1 && max_segments(tiles, KT, T, P) > p.det_slots) --P;
    if (P < 1 || P > 0x7FFFFFFF) return BSP_ERR_INTERNAL;
    NarrowArgs a = {};
    a.bitmaps = p.bitmaps;
    a.offsets = p.offsets;
    a.values = (const uint8_t*)p.values;
    a.Y = Y;
    a.M = p.M;
    a.N = N;
    a.K = p.K;
    a.Mp = p.Mp;
    a.KT = KT;
    a.T = T;
    a.P = P;
    a.ws = (float*)p.ws;
    a.ws_det = I8 ? nullptr : p.ws_det;
    a.err = p.err;
    a.spin_cap = bsp_spin_cap();
    // C ring: as many stages as fit, each sized for the densest GT
    a.c_slot = c_slot_bytes(std::min<uint32_t>(p.max_gt_nnz, 4096u), I8 ? 16u : 8u);
    a.c_stage = c_stage_bytes(a.c_slot);
    a.sc = std::min<int>(SC_MAX, L::C_BYTES / (int)a.c_stage);
    if (a.sc < NG) return BSP_ERR_INTERNAL;  // each decoder group needs a stage of its own in flight
    const int smem = L::OFF_C + a.sc * (int)a.c_stage + 1024;
    // programmatic dependent launch for fp16 only: the int8 variant stalled
    // under it (rarely: about one call in a thousand in back-to-back calls,
    // a wait for its first X tile running out) and is launched in plain
    // stream order, which ran clean
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = I8 ? 0 : 1;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)P);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, spmm_narrow_kernel<I8>, map, a) != cudaSuccess) return BSP_ERR_CUDA;
    }
    // int8 tiles of more than one run go through the workspace too
    if (!any_split(tiles, KT, T, P) && !(I8 && KT > (int64_t)RUN_I8)) return BSP_OK;
    // the tiles split between CTAs: converted by a programmatic dependent
    // kernel (launched while the product kernel drains; it waits for it)
    cudaLaunchConfig_t cfg = {};
    const int64_t elems = p.M * N;
    cfg.gridDim = dim3((unsigned)std::min<int64_t>((elems + 255) / 256, (int64_t)p.num_sms * 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, spmm_narrow_finish_kernel<I8>, Y, (float*)p.ws, (const float*)a.ws_det, p.M,
                              (int64_t)N, KT, T, P) == cudaSuccess
               ? BSP_OK
               : BSP_ERR_CUDA;
}

}  // namespace

bsp_status_t bsp_run_spmm_narrow(const bsp_decode_problem& p, const void* X, int64_t N, void* Y, cudaStream_t s)
{
    if (p.dtype != BSP_FP16 && p.dtype != BSP_INT8) return BSP_ERR_DTYPE;
    if (N < 1 || N > BN || p.K > (int64_t)0x7FFFFFFF) return BSP_ERR_INVALID_ARG;
    if (p.device < 0 || p.device >= 64) return BSP_ERR_INVALID_ARG;
    return p.dtype == BSP_INT8 ? launch_narrow<true>(p, X, N, Y, s) : launch_narrow<false>(p, X, N, Y, s);
}
