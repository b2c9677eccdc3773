// Decode-path product Y = W * X for N <= 16 on CUDA cores, and the
// zero-skipping sparse-vector product.
//
// Method (SpInfer's shared-memory bitmap decoding, "SpInfer: How bitmaps
// make sparse LLMs actually fast", sections "Shared Memory Bitmap Decoding
// (SMBD)" and "The async pipeline"; split-K over GroupTiles with a
// reduction workspace as in "Unified Static-Dynamic Pruning for Efficient
// LLM Inference", section 4.2.3 and its Algorithm 1 epilogue; a producer
// that prefetches the next tiles while the consumers compute, as in
// "UnionSparse: ...", section on the DW-PC pipeline):
//
//  * grid = (splits, M/64): a CTA owns one 64-row strip of W (one GT row)
//    and a contiguous range of GT columns, split between two teams of two
//    warps; each team takes a contiguous run of at most 31 GTs.
//  * each team runs an S-stage ring in shared memory with a "full" and an
//    "empty" mbarrier per stage.  Lane 0 of the team's warp 0 is the
//    producer: it issues 1-D bulk copies (cp.async.bulk, the copy engine,
//    no registers involved) of a GT's 64 bitmaps (512 B), its packed value
//    span (the 16-B aligned superset of [offsets[t], offsets[t+1])) and the
//    N rows of the X tile, all completing on the stage's full barrier, and
//    refills a stage once both warps have arrived on its empty barrier.
//  * per GT each warp computes the BT value bases: popcount of each BT and
//    a warp exclusive scan (shfl).
//  * decode + multiply (decode_gt): lane l owns GT rows l and l+32; warp 0
//    of a team takes K-octets (BT columns) 0-3, warp 1 takes 4-7.  For each
//    BT on its rows a lane takes the row's byte of the bitmap, finds the
//    first value by a masked popcount (nonzeros of the earlier rows of the
//    BT), then walks the 8 positions as a static loop: a set bit loads the
//    next packed value from shared memory and multiplies it into the row.
//  * the warps' partial sums are added in shared memory; with one split the
//    CTA writes Y, otherwise it adds into the split-K workspace and the last
//    CTA of the strip (arrival counter) converts, writes Y and clears the
//    workspace and counter for the next call.
//
// spMspV ("Unified Static-Dynamic Pruning ...", sections 4.2-4.2.2:
// activation-inactive columns are neither fetched nor decoded, with a
// metadata-first prefetch): with N = 1 a K-octet (one BT column, 8
// activations) whose activations are all zero marks its BTs inactive.  The
// fetch of a GT is two-step: x row + bitmaps first; then only the value
// segments of active octets.  In the TCA-BME order the two BTs of one
// TCTile row-half that share a column octet are adjacent, so lane l's BT
// pair (2l, 2l+1) is exactly the segment (TCTile row l/8, octet l%8): each
// active lane issues the bulk copy of its own segment.
//
// Every wait is bounded (spin cap); a wait that gives up records
// BSP_ERR_TIMEOUT in the error word, drains its own copies (again bounded)
// and returns.
#include "bsp_internal.cuh"
#include "bsp_ptx.cuh"
#include "bsp_bits.cuh"

#include <cstdlib>
#include <type_traits>

namespace {

__device__ __forceinline__ int bt_local(int br, int bc)
{
    return (((br >> 1) * 4 + (bc >> 1)) << 2) + (br & 1) + ((bc & 1) << 1);
}

// Tuning of the narrow configurations (fp16 N <= 2, int8): ring stages per
// team and the CTAs per SM that the register budget targets.
#ifndef BSP_DEC_NARROW_STAGES
#define BSP_DEC_NARROW_STAGES 2
#endif
#ifndef BSP_DEC_NARROW_MINB
#define BSP_DEC_NARROW_MINB 4
#endif

constexpr int kMaxRun = 31;  // GTs per team run (offsets of a run fit one warp register)
constexpr int kTeams = 2;    // teams (runs) per CTA
constexpr int kSelMax = 3;   // spMspV: at most this many active K-octets of 8 -> selective fetch

template <int NT, bool I8>
struct DecCfg {
    static constexpr int TEAMS = kTeams;
    static constexpr int WARPS = 2 * TEAMS;            // two warps per team
    static constexpr int THREADS = WARPS * 32;
    static constexpr bool WIDE_X = !I8 && NT >= 4;     // fp32 X tile + packed fp32x2 FMA
    static constexpr int MINB = (NT >= 8) ? 2 : (WIDE_X ? 4 : BSP_DEC_NARROW_MINB);  // CTAs per SM for the register budget
    static constexpr int S = WIDE_X ? 2 : BSP_DEC_NARROW_STAGES;  // pipeline stages per team
    static constexpr int LAG = S >= 3 ? 1 : 0;         // refill the stage of GT i-LAG
    static constexpr int EB = I8 ? 1 : 2;
    static constexpr int E16 = 16 / EB;                // elements per 16-B chunk
    static constexpr int VAL_CHUNKS = 4096 / E16 + 1;  // dense GT + misalignment
    static constexpr int XS = WIDE_X ? NT + 4 : 4;     // widened X-tile row stride (floats)
    static constexpr int XRAW = NT * 64 * EB;          // raw X tile bytes [NT][64]
    // stage layout
    static constexpr int ST_BM = 0;
    static constexpr int ST_X = ST_BM + 512;
    static constexpr int ST_VAL = ST_X + ((XRAW + 15) & ~15);
    static constexpr int STAGE = ST_VAL + VAL_CHUNKS * 16;
    // per-warp area: widened X columns of the warp's 4 octets (WIDE_X only), BT bases
    static constexpr int W_XS = 0;
    static constexpr int W_BASE = WIDE_X ? ((32 * XS * 4 + 15) & ~15) : 0;
    static constexpr int W_SIZE = W_BASE + 64 * 4;
    // team slice: stages, two warp areas, barriers (full, full_v, empty)
    static constexpr int T_WARP = S * STAGE;
    static constexpr int T_BAR = T_WARP + 2 * W_SIZE;
    static constexpr int TEAM_BYTES = (T_BAR + 3 * S * 8 + 15) & ~15;
    static constexpr int SMEM = TEAMS * TEAM_BYTES;
    static constexpr int RED_BYTES = 64 * NT * 4;      // per-warp partial sums (alias the stages)
    static_assert(2 * RED_BYTES <= S * STAGE, "reduction buffers must fit the stages");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// two consecutive raw X elements from shared memory, widened
__device__ __forceinline__ void x_pair(const uint8_t* xraw, int idx, float& a, float& b)
{
    const __half2 v = reinterpret_cast<const __half2*>(xraw)[idx >> 1];
    a = __low2float(v);
    b = __high2float(v);
}

__device__ __forceinline__ void x_pair(const uint8_t* xraw, int idx, int& a, int& b)
{
    const uint16_t v = reinterpret_cast<const uint16_t*>(xraw)[idx >> 1];
    a = (int)(int8_t)(v & 0xFF);
    b = (int)(int8_t)(v >> 8);
}

// spMspV activity: an activation is pruned iff |x| <= tau (tau = 0: exact
// zeros, +-0 included; NaN is never pruned)
__device__ __forceinline__ bool active(float v, float tau) { return !(fabsf(v) <= tau); }
__device__ __forceinline__ bool active(int v, float tau) { return !(fabsf((float)v) <= tau); }

__device__ __forceinline__ void write_out(void* Y, int, int64_t idx, float v, float)
{
    reinterpret_cast<__half*>(Y)[idx] = __float2half_rn(v);
}

__device__ __forceinline__ void write_out(void* Y, int mode, int64_t idx, int v, float scale)
{
    if (mode == BSP_OUT_F32_SCALED)
        reinterpret_cast<float*>(Y)[idx] = __fmul_rn(__int2float_rn(v), scale);
    else
        reinterpret_cast<int*>(Y)[idx] = v;
}

// packed pair of fp32 FMAs: acc.{lo,hi} += w * x.{lo,hi}
__device__ __forceinline__ uint64_t ffma2(uint64_t acc, uint64_t ww, uint64_t x)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(ww), "l"(x), "l"(acc));
    return d;
}

__device__ __forceinline__ uint64_t dup2(float w)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(w));
    return r;
}

__device__ __forceinline__ float2 unpack2(uint64_t v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ uint16_t half_of(const uint4& q, int c)
{
    const uint32_t w = c < 2 ? q.x : c < 4 ? q.y : c < 6 ? q.z : q.w;
    return (uint16_t)((c & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// One position of a row-byte, predicated on its bit (no branch): if
// byte & bit, load the next packed fp16 value from shared memory (byte
// address `addr`), advance `addr` and accumulate w * x into `acc` with one
// rounding (fma.rn.f32.f16: the fp16 product is exact in fp32).
#ifndef BSP_POS_ASM_VOLATILE
#define BSP_POS_ASM_VOLATILE 1
#endif
#if BSP_POS_ASM_VOLATILE
#define BSP_POS_ASM asm volatile
#else
// not volatile: the inputs of a step (address, bitmap byte) come from shared-memory loads made after the
// stage's barrier wait, so the compiler cannot move a step above it, and may interleave independent steps
#define BSP_POS_ASM asm
#endif
__device__ __forceinline__ void pos_f16(float& acc, uint32_t& addr, uint32_t byte, uint32_t bit,
                                        uint16_t x)
{
    BSP_POS_ASM(
        "{\n\t.reg .pred p;\n\t.reg .b32 t;\n\t.reg .b16 w;\n\t"
        "and.b32 t, %2, %3;\n\t"
        "setp.ne.b32 p, t, 0;\n\t"
        "@p ld.shared.u16 w, [%1];\n\t"
        "@p add.u32 %1, %1, 2;\n\t"
        "@p fma.rn.f32.f16 %0, w, %4, %0;\n\t}"
        : "+f"(acc), "+r"(addr)
        : "r"(byte), "r"(bit), "h"(x));
}

__device__ __forceinline__ void pos_f16x2(float& acc0, float& acc1, uint32_t& addr, uint32_t byte,
                                          uint32_t bit, uint16_t x0, uint16_t x1)
{
    BSP_POS_ASM(
        "{\n\t.reg .pred p;\n\t.reg .b32 t;\n\t.reg .b16 w;\n\t"
        "and.b32 t, %3, %4;\n\t"
        "setp.ne.b32 p, t, 0;\n\t"
        "@p ld.shared.u16 w, [%2];\n\t"
        "@p add.u32 %2, %2, 2;\n\t"
        "@p fma.rn.f32.f16 %0, w, %5, %0;\n\t"
        "@p fma.rn.f32.f16 %1, w, %6, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1), "+r"(addr)
        : "r"(byte), "r"(bit), "h"(x0), "h"(x1));
}

// One column c of a row-byte in the spMspV loop: if byte & bit (bit =
// 1 << c), load the value at rank popcount(byte & below) (below = bit - 1)
// after the row-byte's first value (byte address `base`) and accumulate
// w * x with one rounding; no branch.
__device__ __forceinline__ void col_f16(float& acc, uint32_t base, uint32_t byte, uint32_t bit, uint32_t below,
                                        uint16_t x)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 t, r, a;\n\t.reg .b16 w;\n\t"
        "and.b32 t, %2, %3;\n\t"
        "setp.ne.b32 p, t, 0;\n\t"
        "and.b32 r, %2, %4;\n\t"
        "popc.b32 r, r;\n\t"
        "shl.b32 r, r, 1;\n\t"
        "add.u32 a, %1, r;\n\t"
        "@p ld.shared.u16 w, [a];\n\t"
        "@p fma.rn.f32.f16 %0, w, %5, %0;\n\t}"
        : "+f"(acc)
        : "r"(base), "r"(byte), "r"(bit), "r"(below), "h"(x));
}

// Accumulator storage of one lane: rows l and l+32, NT columns of Y.
template <int NT, bool I8, bool WIDE>
struct Accum;
template <int NT>
struct Accum<NT, false, false> { float v[2][2 * NT]; };  // even / odd position chains
template <int NT>
struct Accum<NT, false, true> { uint64_t v[2][NT / 2]; };  // packed fp32 pairs
template <int NT>
struct Accum<NT, true, false> { int v[2][NT]; };

// Decode the warp's four K-octets of one GroupTile and multiply them into
// the lane's two rows.
//
// Lane l owns GT rows l and l+32 (BT rows l/8 and l/8+4, BT row-byte l%8).
// Octets bc0..bc0+3 are taken in turn; inside one, the positions c = 0..7
// of the lane's row-byte are a static loop: a set bit loads the next packed
// value (the masked popcount gives the row-byte's first slot, then a
// running index), a clear bit contributes nothing.  All 32 lanes run the
// same instruction stream, and X sits in registers.
#ifndef BSP_DEC_OCT_UNROLL
#define BSP_DEC_OCT_UNROLL 2
#endif

// RS: base_s is a table of row starts, u16 [64 BT][8 rows] (absolute value
// indices in the stage), instead of the 64 BT bases.
template <int NT, bool I8, bool SKIP, int UNR = 0, bool RS = false, typename A>
__device__ __forceinline__ void decode_gt(const uint64_t* bm_st, const uint32_t* base_s,
                                          const uint8_t* vals, const uint8_t* xraw, const float* x_s,
                                          int N, uint32_t act8, int lane, int bc0, A& acc,
                                          uint64_t cols = ~0ull)
{
    using C = DecCfg<NT, I8>;
    // octet loop unroll (UNR if given): the spMspV loop runs over active octets only
    constexpr int OCT_UNROLL = UNR ? UNR : (SKIP ? 1 : (C::WIDE_X ? 4 : BSP_DEC_OCT_UNROLL));
    const int rr = lane & 7;
    const int gb0 = bt_local(lane >> 3, 0), gb1 = bt_local((lane >> 3) + 4, 0);
    const uint32_t rsh = 8u * (uint32_t)(rr & 3);
    const bool hi = rr >= 4;
    const uint32_t lowm = (1u << rsh) - 1u;
    // spMspV: a real loop over the warp's active octets only (a warp-uniform
    // branch, so skipped octets cost no instructions); otherwise all four,
    // unrolled
    uint32_t todo = SKIP ? ((act8 >> bc0) & 0xFu) : 0xFu;
#pragma unroll(OCT_UNROLL)
    for (int it = 0; it < 4; ++it) {
        if (SKIP && todo == 0u) break;
        const int k = SKIP ? __ffs(todo) - 1 : it;
        if (SKIP) todo &= todo - 1u;
        const int bc = bc0 + k;
        uint32_t byte[2], idx[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gl = (h ? gb1 : gb0) + bt_local(0, bc);
            if constexpr (RS) {
                byte[h] = reinterpret_cast<const uint8_t*>(bm_st)[8 * gl + rr];
                idx[h] = reinterpret_cast<const uint16_t*>(base_s)[8 * gl + rr];
            } else {
                const uint2 bm = *reinterpret_cast<const uint2*>(bm_st + gl);
                const uint32_t w32 = hi ? bm.y : bm.x;
                byte[h] = (w32 >> rsh) & 0xFFu;
                // nonzeros of the earlier rows of the BT: masked popcount
                idx[h] = base_s[gl] + (uint32_t)__popc(w32 & lowm) + (hi ? (uint32_t)__popc(bm.x) : 0u);
            }
        }
        if constexpr (I8) {
            // dense int8 row-byte packed into two words, then dp4a per column of Y
            const int8_t* v8 = reinterpret_cast<const int8_t*>(vals);
            uint32_t xlo[NT], xhi[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint2 q = n < N ? *reinterpret_cast<const uint2*>(xraw + n * 64 + 8 * bc) : make_uint2(0, 0);
                xlo[n] = q.x;
                xhi[n] = q.y;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t wlo = 0, whi = 0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t bit = (byte[h] >> c) & 1u;
                    uint32_t b = 0;
                    if (bit) b = (uint32_t)(uint8_t)v8[idx[h]];
                    idx[h] += bit;
                    if (c < 4) wlo |= b << (8 * c);
                    else whi |= b << (8 * (c - 4));
                }
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    acc.v[h][n] = __dp4a((int)wlo, (int)xlo[n], acc.v[h][n]);
                    acc.v[h][n] = __dp4a((int)whi, (int)xhi[n], acc.v[h][n]);
                }
            }
        } else if constexpr (SKIP) {
            // fp16 spMspV (N = 1): only the columns whose activation is not
            // pruned (bit c of the octet's mask, the same for every lane: a
            // warp-uniform loop).  The value of position c is found by the
            // masked popcount of the row-byte below c, without walking the
            // other positions.
            const uint16_t* xs16 = reinterpret_cast<const uint16_t*>(xraw);
            uint32_t m = (uint32_t)(cols >> (8 * bc)) & 0xFFu;
            uint32_t vb[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) vb[h] = bspx::smem_u32(vals) + 2u * idx[h];
            while (m) {
                const int c = __ffs(m) - 1;
                m &= m - 1u;
                const uint16_t xc = xs16[8 * bc + c];
                const uint32_t bit = 1u << c;
#pragma unroll
                for (int h = 0; h < 2; ++h) col_f16(acc.v[h][0], vb[h], byte[h], bit, bit - 1u, xc);
            }
        } else if constexpr (!C::WIDE_X) {
            // N <= 2: fp16 X octet in registers, mixed-precision FMA; two
            // accumulator chains per row (even / odd positions)
            const uint16_t* vh = reinterpret_cast<const uint16_t*>(vals);
            uint16_t xh[NT][8];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint4 q = n < N ? *reinterpret_cast<const uint4*>(xraw + (n * 64 + 8 * bc) * 2)
                                      : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < 8; ++c) xh[n][c] = half_of(q, c);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t addr = bspx::smem_u32(vh + idx[h]);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if constexpr (NT == 1)
                        pos_f16(acc.v[h][c & 1], addr, byte[h], 1u << c, xh[0][c]);
                    else
                        pos_f16x2(acc.v[h][NT * (c & 1)], acc.v[h][NT * (c & 1) + 1], addr, byte[h], 1u << c,
                                  xh[0][c], xh[1][c]);
                }
            }
        } else {
            // N >= 4: fp32 X rows (broadcast loads), packed fp32x2 FMA
            const uint16_t* vh = reinterpret_cast<const uint16_t*>(vals);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint64_t xv[NT / 2];
                const float* xr = x_s + (k * 8 + c) * C::XS;
#pragma unroll
                for (int j = 0; j < NT / 2; j += 2) {
                    const ulonglong2 q = *reinterpret_cast<const ulonglong2*>(xr + 2 * j);
                    xv[j] = q.x;
                    xv[j + 1] = q.y;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float w = 0.f;
                    if ((byte[h] >> c) & 1u) {
                        w = __half2float(__ushort_as_half(vh[idx[h]]));
                        ++idx[h];
                    }
                    const uint64_t ww = dup2(w);
#pragma unroll
                    for (int j = 0; j < NT / 2; ++j) acc.v[h][j] = ffma2(acc.v[h][j], ww, xv[j]);
                }
            }
        }
    }
}

// The last GT column of a K that is not a multiple of 64 holds fewer than
// 64 activations: x_tail_zero clears the rest of the stage's X row (generic
// stores by the producer lane, made before its arrive on the stage barrier
// so that they are released with it; the proxy fence orders them before
// later bulk copies into the same bytes), x_row_copy copies the part inside
// K (a multiple of 16 bytes: K % (16 / eb) == 0).
__device__ __forceinline__ uint32_t x_row_bytes(int64_t K, int64_t gj, int eb)
{
    const int64_t kv = K - gj * 64;
    return (uint32_t)((kv >= 64 ? 64 : kv) * eb);
}

__device__ __forceinline__ void x_tail_zero(uint8_t* dst, int64_t K, int64_t gj, int eb)
{
    const uint32_t bytes = x_row_bytes(K, gj, eb);
    if (bytes < (uint32_t)(64 * eb)) {
        for (uint32_t b = bytes; b < (uint32_t)(64 * eb); b += 16)
            *reinterpret_cast<uint4*>(dst + b) = make_uint4(0, 0, 0, 0);
        bspx::fence_proxy_async_smem();
    }
}

__device__ __forceinline__ void x_row_copy(uint8_t* dst, const uint8_t* row, int64_t K, int64_t gj, int eb,
                                           uint64_t* bar)
{
    bspx::bulk_g2s(dst, row + gj * 64 * eb, x_row_bytes(K, gj, eb), bar);
}

__device__ __forceinline__ float ws_take(float* p) { return atomicExch(p, 0.0f); }
__device__ __forceinline__ int ws_take(int* p) { return atomicExch(p, 0); }

struct Args {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const uint8_t* values;
    const uint8_t* X;
    int N;
    int64_t M, K;     // logical: Y rows, X row length
    int64_t KT;       // GT columns of the padded grid
    int splits, per_split;
    void* ws;
    float* ws_det;      // fp16 deterministic split-K: [splits][N][M] partial sums, else null
    uint32_t* counters;
    int* err;
    void* Y;
    int mode;
    const float* row_scale;
    uint32_t spin_cap;  // polls before a wait gives up
    int stall_first;    // test only: skip the copies of each team's first GT
    float tau;          // spMspV pruning threshold: |x| <= tau counts as zero
};

template <int NT, bool I8, bool SKIP>
__global__ void __launch_bounds__(DecCfg<NT, I8>::THREADS, DecCfg<NT, I8>::MINB)
spmm_decode_kernel(const Args a)
{
    using C = DecCfg<NT, I8>;
    using Acc = std::conditional_t<I8, int, float>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_last;
    constexpr uint32_t FULL = 0xFFFFFFFFu;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int team = warp >> 1, wt = warp & 1;
    uint8_t* tb = smem + team * C::TEAM_BYTES;
    uint8_t* wa = tb + C::T_WARP + wt * C::W_SIZE;
    float* x_s = reinterpret_cast<float*>(wa + C::W_XS);
    uint32_t* base_s = reinterpret_cast<uint32_t*>(wa + C::W_BASE);
    uint64_t* full = reinterpret_cast<uint64_t*>(tb + C::T_BAR);   // [S] metadata (+ values)
    uint64_t* full_v = full + C::S;                                  // [S] values (spMspV)
    uint64_t* empty = full + 2 * C::S;                               // [S] both warps done

    const int64_t K = a.K, M = a.M;
    const int64_t KT = a.KT;
    const int64_t gi = blockIdx.y;
    const int64_t k_begin = (int64_t)blockIdx.x * a.per_split;
    const int64_t k_cnt = min((int64_t)a.per_split, KT - k_begin);
    const int run = (int)((k_cnt + C::TEAMS - 1) / C::TEAMS);
    const int64_t g0 = k_begin + (int64_t)team * run;              // first GT column of the run
    const int cnt = (int)max((int64_t)0, min((int64_t)run, k_begin + k_cnt - g0));
    const int64_t t0 = gi * KT + g0;
    const int N = a.N;
    const bool producer_warp = (wt == 0);
    const int bc0 = 4 * wt;                                         // the warp's K-octets

    // offsets of the run: lane i holds offsets[t0 + i]  (cnt <= 31)
    const uint32_t offv = (cnt > 0 && lane <= cnt) ? __ldg(a.offsets + t0 + lane) : 0u;

    if (producer_warp && lane == 0) {
        for (int s = 0; s < C::S; ++s) {
            bspx::mbar_init(full + s, 1);
            bspx::mbar_init(full_v + s, 1);
            bspx::mbar_init(empty + s, 2);
        }
        bspx::fence_mbar_init();
    }
    __syncthreads();

    auto stage_ptr = [&](int s) { return tb + s * C::STAGE; };

    // Producer: metadata (bitmaps + X rows) of GT i into stage s; with
    // `with_values` also its whole value span, on the same barrier.
    auto issue_meta = [&](int i, int s, bool with_values, uint32_t o0, uint32_t o1) {
        uint8_t* st = stage_ptr(s);
        const int64_t t = t0 + i, gj = g0 + i;
        uint32_t bytes = 512 + (uint32_t)N * x_row_bytes(K, gj, C::EB);
        uint32_t ch0 = 0, nch = 0;
        if (with_values) {
            ch0 = o0 / C::E16;
            nch = (o1 + C::E16 - 1) / C::E16 - ch0;
            bytes += nch * 16;
        }
        for (int n = 0; n < N; ++n) x_tail_zero(st + C::ST_X + n * 64 * C::EB, K, gj, C::EB);
        bspx::mbar_arrive_expect_tx(full + s, bytes);
        bspx::bulk_g2s(st + C::ST_BM, a.bitmaps + t * 64, 512, full + s);
        for (int n = 0; n < N; ++n)
            x_row_copy(st + C::ST_X + n * 64 * C::EB, a.X + (int64_t)n * K * C::EB, K, gj, C::EB, full + s);
        if (with_values && nch)
            bspx::bulk_g2s(st + C::ST_VAL, a.values + (int64_t)ch0 * 16, nch * 16, full + s);
    };

    // spMspV only (producer warp, all lanes): once the metadata of GT i is
    // in, issue the value segments of its active K-octets on full_v[s].
    auto issue_values_skip = [&](int i, int s) {
        uint8_t* st = stage_ptr(s);
        const uint32_t o0 = __shfl_sync(FULL, offv, i);
        const uint32_t ch0 = o0 / C::E16, shift = o0 - ch0 * C::E16;
        const ulonglong2 bb = reinterpret_cast<const ulonglong2*>(st + C::ST_BM)[lane];
        const uint32_t seg = __popcll(bb.x) + __popcll(bb.y);
        uint32_t incl = seg;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(FULL, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t ex = incl - seg;
        const uint8_t* xr = st + C::ST_X;
        bool act = false;
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
            Acc v0, v1;
            x_pair(xr, (lane & 7) * 8 + c, v0, v1);
            act |= active(v0, a.tau) || active(v1, a.tau);
        }
        uint32_t q0 = 0, q1 = 0;
        if (act && seg) {
            q0 = (ex + shift) / C::E16;
            q1 = (ex + seg + shift + C::E16 - 1) / C::E16;
        }
        uint32_t bytes = (q1 - q0) * 16;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) bytes += __shfl_xor_sync(FULL, bytes, d);
        if (lane == 0) bspx::mbar_arrive_expect_tx(full_v + s, bytes);
        __syncwarp();
        if (q1 > q0)
            bspx::bulk_g2s(st + C::ST_VAL + q0 * 16, a.values + ((int64_t)ch0 + q0) * 16, (q1 - q0) * 16,
                           full_v + s);
    };

    Accum<NT, I8, C::WIDE_X> acc;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < (C::WIDE_X ? NT / 2 : (I8 ? NT : 2 * NT)); ++n) acc.v[h][n] = 0;

    bool failed = false;
    int issued = 0;          // GTs whose metadata copies were issued (producer warp)
    uint32_t vpend = 0;      // spMspV, producer: stages with value copies in flight on full_v
    uint32_t vpar = 0;       // spMspV: parity expected at the next wait on full_v[s], bit s
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(FULL, bspx::mbar_wait_bounded(bar, parity, a.spin_cap));
    };

    // spMspV: a GT with at most kSelMax active K-octets of 8 is fetched
    // selectively in two steps (metadata first, then only the active value
    // segments); a busier GT is fetched whole in one step: skipped segments
    // are ~128 B, close to the DRAM fetch granularity, so selecting them saves
    // little bandwidth and costs a round trip.  Inactive octets are never
    // decoded either way.  The first S GTs of a run are always fetched whole,
    // so the ring starts at once; meanwhile the producer reads the K-octet
    // activity of the later GTs from x (lane i keeps the 8-bit mask of GT i).
    // Consumers apply the same rule from the x tile in shared memory.
    uint32_t my_act = 0xFFu;
    // producer warp only (all lanes): is GT i fetched selectively?
    auto selective = [&](int i) {
        if constexpr (!SKIP) return false;
        return i >= C::S && __popc(__shfl_sync(FULL, my_act, i)) <= kSelMax;
    };

    // prologue: fill the ring
    if (producer_warp) {
        for (int i = 0; i < C::S && i < cnt; ++i) {
            const uint32_t p0 = __shfl_sync(FULL, offv, i);
            const uint32_t p1 = __shfl_sync(FULL, offv, i + 1);
            if (lane == 0 && !(a.stall_first && i == 0)) issue_meta(i, i, true, p0, p1);
        }
        issued = cnt < C::S ? cnt : C::S;
        if constexpr (SKIP) {
            // lane i reads the 64 activations of GT i (one octet per 16-B or
            // 8-B load) and keeps their K-octet activity mask
            if (lane >= C::S && lane < cnt) {
                const uint8_t* xp = a.X + (g0 + lane) * 64 * C::EB;
                const int64_t kv = K - (g0 + lane) * 64;  // activations of this GT column inside K
                uint32_t act = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    bool nz = false;
                    if (8 * j >= kv) break;
                    if constexpr (C::EB == 2) {
                        const uint4 q = __ldg(reinterpret_cast<const uint4*>(xp) + j);
                        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __half2 h2 = *reinterpret_cast<const __half2*>(&w[e]);
                            nz |= active(__low2float(h2), a.tau) || active(__high2float(h2), a.tau);
                        }
                    } else {
                        const uint2 q = __ldg(reinterpret_cast<const uint2*>(xp) + j);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            nz |= active((int)(int8_t)(((e < 4 ? q.x : q.y) >> (8 * (e & 3))) & 0xFFu), a.tau);
                    }
                    act |= (nz ? 1u : 0u) << j;
                }
                my_act = act;
            }
        }
    }

    int i_fail = 0;
    for (int i = 0; i < cnt && !failed; ++i) {
        i_fail = i;
        const int s = i % C::S;
        const uint32_t ph = (uint32_t)((i / C::S) & 1);
        uint8_t* st = stage_ptr(s);
        const uint32_t o0 = __shfl_sync(FULL, offv, i);

        if constexpr (SKIP) {
            // producer: once the metadata of a selective GT i+1 is in, fetch its active values
            if (producer_warp && i + 1 < cnt && selective(i + 1)) {
                const int s1 = (i + 1) % C::S;
                if (!wait(full + s1, (uint32_t)(((i + 1) / C::S) & 1))) { failed = true; break; }
                issue_values_skip(i + 1, s1);
                vpend |= 1u << s1;
            }
        }
        if (!wait(full + s, ph)) { failed = true; break; }

        // BT value bases (all 64 BTs; each warp keeps its own copy)
        const uint64_t* bm_st = reinterpret_cast<const uint64_t*>(st + C::ST_BM);
        const ulonglong2 bb = reinterpret_cast<const ulonglong2*>(bm_st)[lane];
        const uint32_t c0 = __popcll(bb.x), c1 = __popcll(bb.y);
        uint32_t incl = c0 + c1;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(FULL, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t shift = o0 - (o0 / C::E16) * C::E16;
        const uint32_t ex = incl - (c0 + c1) + shift;  // span misalignment folded in
        base_s[2 * lane] = ex;
        base_s[2 * lane + 1] = ex + c0;

        const uint8_t* xraw = st + C::ST_X;
        if constexpr (C::WIDE_X) {
            // the warp's 32 X columns widened to fp32 [32][XS]; lane owns column 32*wt + lane
            float xa[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n)
                xa[n] = n < N ? __half2float(reinterpret_cast<const __half*>(xraw)[n * 64 + 32 * wt + lane]) : 0.f;
#pragma unroll
            for (int j = 0; j < NT; j += 4)
                *reinterpret_cast<float4*>(x_s + lane * C::XS + j) = make_float4(xa[j], xa[j + 1], xa[j + 2], xa[j + 3]);
        }
        uint32_t act8 = 0xFFu;
        if constexpr (SKIP) {
            // K-octet j is active iff one of x[8j .. 8j+7] is not pruned
            Acc va, vb;
            x_pair(xraw, 2 * lane, va, vb);
            const uint32_t bal = __ballot_sync(FULL, active(va, a.tau) || active(vb, a.tau));
            act8 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) act8 |= (((bal >> (4 * j)) & 0xFu) ? 1u : 0u) << j;
            if (i >= C::S && __popc(act8) <= kSelMax) {  // selective GT: its values came on full_v[s]
                if (!wait(full_v + s, (vpar >> s) & 1u)) { failed = true; break; }
                vpar ^= 1u << s;
                vpend &= ~(1u << s);
            }
            if (a.tau > 0.f) {
                // prune: this warp's 32 columns of the x tile, |x| <= tau -> 0
                // (the other warp may read them meanwhile for its activity
                // mask, which is the same either way)
                const int col = 32 * wt + lane;
                if constexpr (I8) {
                    int8_t* xc = reinterpret_cast<int8_t*>(st + C::ST_X) + col;
                    if (!active((int)*xc, a.tau)) *xc = 0;
                } else {
                    __half* xc = reinterpret_cast<__half*>(st + C::ST_X) + col;
                    if (!active(__half2float(*xc), a.tau)) *xc = __ushort_as_half(0);
                }
            }
        }
        __syncwarp();

        decode_gt<NT, I8, SKIP>(bm_st, base_s, st + C::ST_VAL, xraw, x_s, N, act8, lane, bc0, acc);
        __syncwarp();
        if (lane == 0) bspx::mbar_arrive(empty + s);

        // producer: refill the stage of GT j = i - LAG with GT j + S once both
        // warps are done with GT j
        if (producer_warp) {
            const int j = i - C::LAG;
            if (j >= 0 && j + C::S < cnt) {
                const int sj = j % C::S;
                if (!wait(empty + sj, (uint32_t)((j / C::S) & 1))) { failed = true; break; }
                const uint32_t p0 = __shfl_sync(FULL, offv, j + C::S);
                const uint32_t p1 = __shfl_sync(FULL, offv, j + C::S + 1);
                const bool sel = selective(j + C::S);
                if (lane == 0) issue_meta(j + C::S, sj, !sel, p0, p1);
                issued = j + C::S + 1;
            }
        }
    }

    if (failed) {
        // a wait gave up: record the timeout, then let this team's copies
        // that are still in flight land (each wait bounded) before leaving
        if (lane == 0) atomicExch(a.err, (int)BSP_ERR_TIMEOUT);
        if (producer_warp) {
            for (int j = i_fail; j < issued; ++j)
                bspx::mbar_wait_bounded(full + (j % C::S), (uint32_t)((j / C::S) & 1), a.spin_cap);
            if constexpr (SKIP)
                for (int t = 0; t < C::S; ++t)
                    if ((vpend >> t) & 1u) bspx::mbar_wait_bounded(full_v + t, (vpar >> t) & 1u, a.spin_cap);
        }
    }

    // ---- CTA reduction: each warp writes its 64 partial rows, then sum
    __syncthreads();
    Acc* red = reinterpret_cast<Acc*>(tb + wt * C::RED_BYTES);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = lane + 32 * h;
        if constexpr (C::WIDE_X) {
#pragma unroll
            for (int j = 0; j < NT / 2; ++j) {
                const float2 f = unpack2(acc.v[h][j]);
                red[row * NT + 2 * j] = f.x;
                red[row * NT + 2 * j + 1] = f.y;
            }
        } else if constexpr (I8) {
#pragma unroll
            for (int n = 0; n < NT; ++n) red[row * NT + n] = acc.v[h][n];
        } else {
#pragma unroll
            for (int n = 0; n < NT; ++n) red[row * NT + n] = acc.v[h][n] + acc.v[h][n + NT];
        }
    }
    __syncthreads();

    Acc* ws = reinterpret_cast<Acc*>(a.ws);
    // deterministic split-K (fp16): each split stores its partial sums to a
    // slot of its own and the last CTA adds the slots in split order
    float* det = nullptr;
    if constexpr (!I8)
        if (a.ws_det) det = a.ws_det + (int64_t)blockIdx.x * N * M;
    for (int i = threadIdx.x; i < 64 * NT; i += C::THREADS) {
        const int r = i / NT, n = i % NT;
        Acc sum = Acc(0);
#pragma unroll
        for (int t = 0; t < C::TEAMS; ++t)
#pragma unroll
            for (int w = 0; w < 2; ++w)
                sum += reinterpret_cast<const Acc*>(smem + t * C::TEAM_BYTES + w * C::RED_BYTES)[i];
        const int64_t m = gi * 64 + r;
        if (n < N && m < M) {  // rows past M are padding
            if (a.splits == 1)
                write_out(a.Y, a.mode, (int64_t)n * M + m, sum, a.row_scale ? a.row_scale[m] : 1.0f);
            else if (det)
                det[(int64_t)n * M + m] = (float)sum;
            else
                atomicAdd(ws + (int64_t)n * M + m, sum);
        }
    }
    if (a.splits == 1) return;

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.counters + gi, 1u) == (uint32_t)(a.splits - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = threadIdx.x; i < 64 * N; i += C::THREADS) {
        const int n = i >> 6, r = i & 63;
        const int64_t m = gi * 64 + r;
        if (m >= M) continue;
        Acc v;
        if constexpr (!I8) {
            if (det) {
                v = 0.f;
                for (int sp = 0; sp < a.splits; ++sp) v += __ldcg(a.ws_det + ((int64_t)sp * N + n) * M + m);
            } else {
                v = ws_take(ws + (int64_t)n * M + m);
            }
        } else {
            v = ws_take(ws + (int64_t)n * M + m);
        }
        write_out(a.Y, a.mode, (int64_t)n * M + m, v, a.row_scale ? a.row_scale[m] : 1.0f);
    }
    if (threadIdx.x == 0) a.counters[gi] = 0u;
}

// ---------------------------------------------------------------------------
// GT-per-warp kernel, fp16 N <= 2.
//
// One producer warp and CW consumer warps share one ring of S stages.
// Consumer c decodes whole GroupTiles (i = c, c + CW, ...): lane l owns GT
// rows l and l+32 over all eight K-octets, so the per-GT work that does not
// scale with the positions (the wait, the BT popcount scan, the release)
// is paid once per GT instead of once per GT and warp.  A stage holds the
// bitmaps, a 16-byte header (the misalignment of the value span), the N
// X rows of the GT column and the value span, sized for the largest GT of
// the matrix (its nonzero count is recorded at encode / import time), so a
// sparse matrix gets small stages and more of them fit on an SM.
#ifndef BSP_GTW_CONSUMERS
#define BSP_GTW_CONSUMERS 2
#endif
#ifndef BSP_GTW_STAGES
#define BSP_GTW_STAGES 4
#endif
#ifndef BSP_GTW_MINB
#define BSP_GTW_MINB 8
#endif
#ifndef BSP_GTW_OCT_UNROLL
#define BSP_GTW_OCT_UNROLL 1
#endif
// consumers: a row-start table per GT (1) or BT bases + masked popcounts per
// row-byte (0).  The table pays where few positions are decoded (spMspV);
// for the plain product its cost exceeds the saving (measured).
#ifndef BSP_GTW_RS_SPMM
#define BSP_GTW_RS_SPMM 0
#endif
#ifndef BSP_GTW_RS_SKIP
#define BSP_GTW_RS_SKIP 1
#endif

namespace gtw {
constexpr int CW = BSP_GTW_CONSUMERS;  // consumer warps
constexpr int S = BSP_GTW_STAGES;      // ring stages
// GT i goes to consumer i % CW and stage i % S.  With S a multiple of CW
// every stage has one consumer, which has seen the previous GT of its
// stage land before it waits for the next one: a parity wait can then
// never be two phases behind (and mistake an old phase for the new one).
static_assert(S % CW == 0 && S >= 2 * CW, "stages: a multiple of the consumers, two per consumer at least");
constexpr int THREADS = 32 * (1 + CW);
constexpr int HDR = 16;                // stage header after the bitmaps
constexpr uint32_t kSleepNs = 500;     // suspend hint of the waiting polls

// bytes of one stage and offset of its value span, for N X rows and a GT
// of at most max_nnz fp16 values
inline void stage_geometry(int nt, uint32_t max_nnz, uint32_t& stage_bytes, uint32_t& val_off)
{
    val_off = 512 + HDR + (uint32_t)nt * 128;
    const uint32_t chunks = (max_nnz * 2 + 15) / 16 + 1;  // + 1: misalignment of the span
    stage_bytes = (val_off + chunks * 16 + 127) & ~127u;
}
constexpr int AREA = 1024;  // per consumer: row starts u16 [64][8], or BT bases u32 [64]
inline size_t smem_bytes(uint32_t stage_bytes) { return (size_t)S * stage_bytes + CW * AREA + 3 * S * 8; }
// spMspV: a GT beyond the first S (which start the ring at once) with at
// most BSP_GTW_SELMAX active K-octets is fetched selectively (metadata
// first, then only the value segments of its active octets).  The second
// round trip costs more than it saves unless most of the values can be
// left behind: with 85%-zero activations (3 in 4 octets active) fetching
// whole GTs is faster, so the default asks for 6 of 8 octets inactive.
#ifndef BSP_GTW_SELMAX
#define BSP_GTW_SELMAX 2
#endif
__device__ __forceinline__ bool gtw_selective(int i, uint32_t act8)
{
    return i >= S && __popc(act8) <= BSP_GTW_SELMAX;
}
}  // namespace gtw

struct GtwArgs {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const uint8_t* values;
    const uint8_t* X;
    int N;
    int64_t M, K;     // logical: Y rows, X row length
    int64_t KT;       // GT columns of the padded grid
    int splits, per_split;
    float* ws;
    float* ws_det;    // deterministic split-K: [splits][N][M] partial sums, else null
    uint32_t* counters;
    int* err;
    __half* Y;
    uint32_t spin_cap;
    uint32_t stage_bytes, val_off;
    int stall_first;  // test only: skip the copies of the first GT
    float tau;        // spMspV pruning threshold: |x| <= tau counts as zero
};

template <int NT, bool SKIP>
__global__ void __launch_bounds__(gtw::THREADS, BSP_GTW_MINB)
spmm_decode_gtw_kernel(const GtwArgs a)
{
    using namespace gtw;
    constexpr bool RS = SKIP ? (BSP_GTW_RS_SKIP != 0) : (BSP_GTW_RS_SPMM != 0);
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_last;
    constexpr uint32_t FULL = 0xFFFFFFFFu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t SB = a.stage_bytes;
    uint32_t* bases = reinterpret_cast<uint32_t*>(smem + S * SB);             // [CW][AREA / 4]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB + CW * AREA);  // [S]
    uint64_t* empty = full + S;                                                // [S]
    uint64_t* full_v = full + 2 * S;                                           // [S] spMspV values

    const int64_t K = a.K, M = a.M, KT = a.KT;
    const int64_t gi = blockIdx.y;
    const int64_t k_begin = (int64_t)blockIdx.x * a.per_split;
    const int cnt = (int)max((int64_t)0, min((int64_t)a.per_split, KT - k_begin));
    const int64_t t0 = gi * KT + k_begin;
    const int N = a.N;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            bspx::mbar_init(full + s, 1);
            bspx::mbar_init(empty + s, 1);
            bspx::mbar_init(full_v + s, 1);
        }
        bspx::fence_mbar_init();
    }
    __syncthreads();

    bool failed = false;
    Accum<NT, false, false> acc;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < 2 * NT; ++n) acc.v[h][n] = 0.f;

    if (warp == 0 && !SKIP) {
        // ---- producer: GT i into stage i % S once its previous GT is released
        uint32_t offv = 0;
        int wbase = 0;
        uint32_t s = 0, ph = 0;
        int i = 0;  // GTs issued
        for (; i < cnt; ++i) {
            if (i >= S && !__all_sync(FULL, bspx::mbar_wait_sleep(empty + s, ph ^ 1u, a.spin_cap, kSleepNs))) {
                failed = true;
                break;
            }
            if (i == 0 || i - wbase >= 31) {  // window: lane j holds offsets[t0 + wbase + j]
                wbase = i;
                const int j = wbase + lane;
                offv = (j <= cnt) ? __ldg(a.offsets + t0 + j) : 0u;
            }
            const uint32_t o0 = __shfl_sync(FULL, offv, i - wbase), o1 = __shfl_sync(FULL, offv, i - wbase + 1);
            if (lane == 0 && !(a.stall_first && i == 0)) {
                uint8_t* st = smem + s * SB;
                const uint32_t ch0 = o0 / 8, nch = (o1 + 7) / 8 - ch0;
                *reinterpret_cast<uint32_t*>(st + 512) = o0 - ch0 * 8;
                for (int n = 0; n < N; ++n) x_tail_zero(st + 512 + HDR + n * 128, K, k_begin + i, 2);
                bspx::mbar_arrive_expect_tx(full + s, 512u + (uint32_t)N * x_row_bytes(K, k_begin + i, 2) + nch * 16u);
                bspx::bulk_g2s(st, a.bitmaps + (t0 + i) * 64, 512, full + s);
                for (int n = 0; n < N; ++n)
                    x_row_copy(st + 512 + HDR + n * 128, a.X + (int64_t)n * K * 2, K, k_begin + i, 2, full + s);
                if (nch) bspx::bulk_g2s(st + a.val_off, a.values + (int64_t)ch0 * 16, nch * 16, full + s);
            }
            if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
        // let the copies still in flight land before the stages are reused (bounded)
        for (int k = (i > S ? i - S : 0); k < i; ++k)
            bspx::mbar_wait_bounded(full + (k % S), (uint32_t)((k / S) & 1), a.spin_cap);
    } else if (warp == 0) {
        // ---- spMspV producer ("metadata first"): a GT with an inactive K-octet
        // (beyond the first S, which start the ring) is fetched in two steps:
        // bitmaps + x, then, once those are in, only the value segments of
        // its active octets.  The producer never blocks on one GT: each pass
        // issues the values of the oldest selective GT whose metadata has
        // landed and the metadata of the next GT whose stage is free, and
        // naps when neither is ready.
        uint32_t offv = 0, actv = 0;
        int wbase = -64, awbase = -64;  // offsets / activity windows: lane j holds GT base + j
        uint32_t selmask = 0;           // bit k % 32: GT k is selective
        uint32_t vpend = 0, vpar = 0;   // stages with value copies in flight, their parities
        int next = 0, vnext = 0;        // next GT to issue, oldest GT whose values may be pending
        uint32_t idle = 0;
        // value segments of selective GT p (its metadata has landed).  In
        // GT order the BT pair (2l, 2l+1) is the segment (TCTile row l/8,
        // octet l%8); runs of adjacent active segments go as one copy,
        // issued by the run's first lane.
        auto issue_values = [&](int p) {
            const int sp = p % S;
            uint8_t* st = smem + sp * SB;
            const uint32_t* hdr = reinterpret_cast<const uint32_t*>(st + 512);
            const uint32_t shift = hdr[0], ch0 = hdr[1], a8 = hdr[2];
            const ulonglong2 bb = reinterpret_cast<const ulonglong2*>(st)[lane];
            const uint32_t seg = __popcll(bb.x) + __popcll(bb.y);
            uint32_t incl = seg;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(FULL, incl, d);
                if (lane >= d) incl += o;
            }
            const uint32_t ex = incl - seg;
            const bool act = (a8 >> (lane & 7)) & 1u;
            const uint32_t q0 = (ex + shift) / 8, q1 = (ex + seg + shift + 7) / 8;
            const uint32_t A = __ballot_sync(FULL, act);
            const bool first = act && !(lane > 0 && ((A >> (lane - 1)) & 1u));
            const uint32_t above = lane == 31 ? 0u : (~A & (~0u << (lane + 1)));  // inactive lanes above
            const int e = above ? __ffs(above) - 2 : 31;                          // last lane of the run
            const uint32_t q1e = __shfl_sync(FULL, q1, e);
            uint32_t bytes = (first && q1e > q0) ? (q1e - q0) * 16 : 0u;
            const uint32_t mine = bytes;
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) bytes += __shfl_xor_sync(FULL, bytes, d);
            if (lane == 0) bspx::mbar_arrive_expect_tx(full_v + sp, bytes);
            __syncwarp();
            if (mine)
                bspx::bulk_g2s(st + a.val_off + q0 * 16, a.values + ((int64_t)ch0 + q0) * 16, mine, full_v + sp);
            vpend |= 1u << sp;
        };
        while (next < cnt || vnext < next) {
            bool prog = false;
            while (vnext < next && !((selmask >> (vnext & 31)) & 1u)) ++vnext;
            if (vnext < next) {
                const uint32_t landed =
                    lane == 0 ? (uint32_t)bspx::mbar_try_wait(full + vnext % S, (uint32_t)((vnext / S) & 1)) : 0u;
                if (__shfl_sync(FULL, landed, 0)) {
                    issue_values(vnext);
                    ++vnext;
                    prog = true;
                }
            }
            if (next < cnt) {
                const int sn = next % S;
                uint32_t free = next < S ? 1u : 0u;
                if (!free && lane == 0)
                    free = (uint32_t)bspx::mbar_try_wait(empty + sn, (uint32_t)(((next / S) & 1) ^ 1));
                if (__shfl_sync(FULL, free, 0)) {
                    if (vpend & (1u << sn)) {  // the stage's previous selective GT was consumed
                        vpend &= ~(1u << sn);
                        vpar ^= 1u << sn;
                    }
                    if (next - wbase >= 31) {
                        wbase = next;
                        const int j = wbase + lane;
                        offv = (j <= cnt) ? __ldg(a.offsets + t0 + j) : 0u;
                    }
                    const uint32_t o0 = __shfl_sync(FULL, offv, next - wbase);
                    const uint32_t o1 = __shfl_sync(FULL, offv, next - wbase + 1);
                    uint32_t a8 = 0xFFu;
                    if (next >= S) {
                        if (next - awbase >= 32) {
                            // lane j: K-octet activity of GT awbase + j, from x (one octet per 16-B load)
                            awbase = next;
                            const int j = awbase + lane;
                            uint32_t act = 0xFFu;
                            if (j < cnt) {
                                act = 0;
                                const uint4* xp = reinterpret_cast<const uint4*>(a.X + (k_begin + j) * 64 * 2);
                                const int64_t kv = K - (k_begin + j) * 64;  // activations inside K
#pragma unroll
                                for (int o = 0; o < 8; ++o) {
                                    if (8 * o >= kv) break;
                                    const uint4 q = __ldg(xp + o);
                                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
                                    bool nz = false;
#pragma unroll
                                    for (int e2 = 0; e2 < 4; ++e2) {
                                        const __half2 h2 = *reinterpret_cast<const __half2*>(&w[e2]);
                                        nz |= active(__low2float(h2), a.tau) || active(__high2float(h2), a.tau);
                                    }
                                    act |= (nz ? 1u : 0u) << o;
                                }
                            }
                            actv = act;
                        }
                        a8 = __shfl_sync(FULL, actv, next - awbase);
                    }
                    const bool sel = gtw_selective(next, a8);
                    if (sel) selmask |= 1u << (next & 31);
                    else selmask &= ~(1u << (next & 31));
                    if (lane == 0 && !(a.stall_first && next == 0)) {
                        uint8_t* st = smem + sn * SB;
                        const uint32_t ch0 = o0 / 8, nch = sel ? 0u : (o1 + 7) / 8 - ch0;
                        uint32_t* hdr = reinterpret_cast<uint32_t*>(st + 512);
                        hdr[0] = o0 - ch0 * 8;
                        hdr[1] = ch0;
                        hdr[2] = a8;
                        x_tail_zero(st + 512 + HDR, K, k_begin + next, 2);
                        bspx::mbar_arrive_expect_tx(full + sn, 512u + x_row_bytes(K, k_begin + next, 2) + nch * 16u);
                        bspx::bulk_g2s(st, a.bitmaps + (t0 + next) * 64, 512, full + sn);
                        x_row_copy(st + 512 + HDR, a.X, K, k_begin + next, 2, full + sn);
                        if (nch) bspx::bulk_g2s(st + a.val_off, a.values + (int64_t)ch0 * 16, nch * 16, full + sn);
                    }
                    ++next;
                    prog = true;
                }
            }
            if (prog) {
                idle = 0;
            } else {
                if (++idle > a.spin_cap) {
                    failed = true;
                    break;
                }
                __nanosleep(64);
            }
        }
        // let the copies still in flight land before the stages are reused (bounded)
        for (int k = (next > S ? next - S : 0); k < next; ++k)
            bspx::mbar_wait_bounded(full + (k % S), (uint32_t)((k / S) & 1), a.spin_cap);
        for (int t = 0; t < S; ++t)
            if ((vpend >> t) & 1u) bspx::mbar_wait_bounded(full_v + t, (vpar >> t) & 1u, a.spin_cap);
    } else {
        // ---- consumers
        const int cw = warp - 1;
        uint32_t* base_s = bases + cw * (AREA / 4);
        uint32_t vpar = 0;  // spMspV: parity of the next full_v wait, bit per stage
        for (int i = cw; i < cnt; i += CW) {
            const int s = i % S;
            if (!__all_sync(FULL, bspx::mbar_wait_sleep(full + s, (uint32_t)((i / S) & 1), a.spin_cap, kSleepNs))) {
                failed = true;
                break;
            }
            const uint8_t* st = smem + s * SB;
            const uint64_t* bm_st = reinterpret_cast<const uint64_t*>(st);
            const uint32_t shift = *reinterpret_cast<const uint32_t*>(st + 512);
            const uint8_t* xraw = st + 512 + HDR;
            uint32_t act8 = 0xFFu;
            uint64_t cols = ~0ull;
            if constexpr (SKIP) {
                // column c is active iff x[c] is not pruned; K-octet j iff
                // one of its columns is
                const __half* xh = reinterpret_cast<const __half*>(xraw);
                const uint32_t m_lo = __ballot_sync(FULL, active(__half2float(xh[lane]), a.tau));
                const uint32_t m_hi = __ballot_sync(FULL, active(__half2float(xh[lane + 32]), a.tau));
                cols = (uint64_t)m_lo | ((uint64_t)m_hi << 32);
                act8 = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) act8 |= (((cols >> (8 * j)) & 0xFFull) ? 1u : 0u) << j;
                if (gtw_selective(i, act8)) {  // selective GT: its values come on full_v[s]
                    if (!__all_sync(FULL, bspx::mbar_wait_sleep(full_v + s, (vpar >> s) & 1u, a.spin_cap, kSleepNs))) {
                        failed = true;
                        break;
                    }
                    vpar ^= 1u << s;
                }
            }
            // BT value bases: popcounts and a warp exclusive scan
            const ulonglong2 bb = reinterpret_cast<const ulonglong2*>(bm_st)[lane];
            const uint32_t c0 = __popcll(bb.x), c1 = __popcll(bb.y);
            uint32_t incl = c0 + c1;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(FULL, incl, d);
                if (lane >= d) incl += o;
            }
            const uint32_t ex = incl - (c0 + c1) + shift;
            if constexpr (RS) {
                // first value of every BT row of the GT: BTs 2 lane, 2 lane + 1
                uint4* rs = reinterpret_cast<uint4*>(base_s) + 2 * lane;
                rs[0] = bspx::row_starts(bb.x, ex);
                rs[1] = bspx::row_starts(bb.y, ex + c0);
            } else {
                base_s[2 * lane] = ex;
                base_s[2 * lane + 1] = ex + c0;
            }
            __syncwarp();
            decode_gt<NT, false, SKIP, BSP_GTW_OCT_UNROLL, RS>(bm_st, base_s, st + a.val_off, xraw, nullptr, N, act8,
                                                               lane, 0, acc, cols);
            decode_gt<NT, false, SKIP, BSP_GTW_OCT_UNROLL, RS>(bm_st, base_s, st + a.val_off, xraw, nullptr, N, act8,
                                                               lane, 4, acc, cols);
            __syncwarp();
            if (lane == 0) bspx::mbar_arrive(empty + s);
        }
    }
    if (failed && lane == 0) atomicExch(a.err, (int)BSP_ERR_TIMEOUT);

    // ---- CTA reduction over the consumers (the buffer aliases the ring)
    __syncthreads();
    float* red = reinterpret_cast<float*>(smem);  // [CW][64][NT]
    if (warp > 0) {
        const int cw = warp - 1;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int n = 0; n < NT; ++n)
                red[(cw * 64 + lane + 32 * h) * NT + n] = acc.v[h][n] + acc.v[h][n + NT];
    }
    __syncthreads();
    float* det = a.ws_det ? a.ws_det + (int64_t)blockIdx.x * N * M : nullptr;  // deterministic split-K slot
    for (int i = threadIdx.x; i < 64 * NT; i += THREADS) {
        const int r = i / NT, n = i % NT;
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < CW; ++c) sum += red[c * 64 * NT + i];
        const int64_t m = gi * 64 + r;
        if (n < N && m < M) {  // rows past M are padding
            if (a.splits == 1)
                a.Y[(int64_t)n * M + m] = __float2half_rn(sum);
            else if (det)
                det[(int64_t)n * M + m] = sum;
            else
                atomicAdd(a.ws + (int64_t)n * M + m, sum);
        }
    }
    if (a.splits == 1) return;

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.counters + gi, 1u) == (uint32_t)(a.splits - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = threadIdx.x; i < 64 * N; i += THREADS) {
        const int n = i >> 6, r = i & 63;
        const int64_t m = gi * 64 + r;
        if (m >= M) continue;
        float v = 0.f;
        if (det) {
            for (int sp = 0; sp < a.splits; ++sp) v += __ldcg(a.ws_det + ((int64_t)sp * N + n) * M + m);
        } else {
            v = ws_take(a.ws + (int64_t)n * M + m);
        }
        a.Y[(int64_t)n * M + m] = __float2half_rn(v);
    }
    if (threadIdx.x == 0) a.counters[gi] = 0u;
}

// Split of the GT columns for the GT-per-warp kernel: the split whose
// number of CTA waves times (GTs per CTA + a fixed 4) is smallest (ties:
// fewer CTAs),
// with at least 2 CW GTs per CTA when the row strip has that many.
int gtw_splits_auto(int64_t strips, int64_t KT, int64_t slots)
{
    int64_t best = 1, best_cost = INT64_MAX;
    for (int64_t sp = 1; sp <= KT; ++sp) {
        const int64_t per = (KT + sp - 1) / sp;
        if (per < 2 * gtw::CW && sp > 1) break;
        const int64_t real = (KT + per - 1) / per;
        const int64_t ctas = strips * real;
        // a CTA's start (first copies) and end (reduction) cost about 4 GTs
        const int64_t cost = ((ctas + slots - 1) / slots) * (per + 4);
        if (cost < best_cost) {
            best_cost = cost;
            best = real;
        }
    }
    return (int)best;
}

// BSP_TUNE_SPLITK overrides the choice (tests and tuning)
int gtw_splits(int64_t strips, int64_t KT, int64_t slots)
{
    const int64_t v = bsp_tune(BSP_TUNE_SPLITK);
    if (v >= 1) return (int)std::min<int64_t>(v, KT);
    return gtw_splits_auto(strips, KT, slots);
}

// CTAs of the GT-per-warp kernel resident at once on the whole GPU
int64_t gtw_slots(const bsp_decode_problem& p, int NT)
{
    uint32_t stage_bytes = 0, val_off = 0;
    gtw::stage_geometry(NT, std::min<uint32_t>(p.max_gt_nnz, 4096u), stage_bytes, val_off);
    const size_t smem = gtw::smem_bytes(stage_bytes);
    int per_sm = (int)std::min<size_t>((size_t)BSP_GTW_MINB, (size_t)(227 * 1024) / (smem + 1024));
    if (per_sm < 1) per_sm = 1;
    return (int64_t)p.num_sms * per_sm;
}

// In deterministic mode the split count is bounded by the handle's slots.
int clamp_det(const bsp_decode_problem& p, int splits)
{
    if (p.ws_det && splits > p.det_slots) return p.det_slots;
    return splits;
}

template <int NT, bool SKIP>
bsp_status_t launch_gtw(const bsp_decode_problem& p, const void* X, int N, void* Y, float tau, cudaStream_t s)
{
    using namespace gtw;
    static bsp_attr_once attr;
    if (p.device < 0 || p.device >= 64) return BSP_ERR_INVALID_ARG;
    uint32_t stage_bytes = 0, val_off = 0;
    stage_geometry(NT, 4096, stage_bytes, val_off);
    const size_t smem_max = smem_bytes(stage_bytes);
    if (!attr.run(p.device, [&] {
            return cudaFuncSetAttribute(spmm_decode_gtw_kernel<NT, SKIP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
        }))
        return BSP_ERR_CUDA;
    stage_geometry(NT, std::min<uint32_t>(p.max_gt_nnz, 4096u), stage_bytes, val_off);
    const size_t smem = smem_bytes(stage_bytes);
    const int64_t strips = p.Mp / 64, KT = p.Kp / 64;
    const int splits0 = clamp_det(p, gtw_splits(strips, KT, gtw_slots(p, NT)));
    const int per_split = (int)((KT + splits0 - 1) / splits0);
    const int splits = (int)((KT + per_split - 1) / per_split);
    GtwArgs a;
    a.bitmaps = p.bitmaps;
    a.offsets = p.offsets;
    a.values = (const uint8_t*)p.values;
    a.X = (const uint8_t*)X;
    a.N = N;
    a.M = p.M;
    a.K = p.K;
    a.KT = p.Kp / 64;
    a.splits = splits;
    a.per_split = per_split;
    a.ws = (float*)p.ws;
    a.ws_det = splits > 1 ? p.ws_det : nullptr;
    a.counters = p.counters;
    a.err = p.err;
    a.Y = (__half*)Y;
    a.spin_cap = bsp_spin_cap();
    a.stage_bytes = stage_bytes;
    a.val_off = val_off;
    a.stall_first = bsp_test_stall();
    a.tau = tau;
    dim3 grid((unsigned)splits, (unsigned)strips);
    spmm_decode_gtw_kernel<NT, SKIP><<<grid, THREADS, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <int NT, bool I8, bool SKIP>
bsp_status_t launch(const bsp_decode_problem& p, const void* X, int N, void* Y, int mode,
                    const float* row_scale, float tau, cudaStream_t s)
{
    using C = DecCfg<NT, I8>;
    // the opt-in shared-memory size is set once per device
    static bsp_attr_once attr;
    if (p.device < 0 || p.device >= 64) return BSP_ERR_INVALID_ARG;
    if (!attr.run(p.device, [&] {
            return cudaFuncSetAttribute(spmm_decode_kernel<NT, I8, SKIP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        }))
        return BSP_ERR_CUDA;
    const int64_t KT = p.Kp / 64;
    int splits = clamp_det(p, bsp_decode_splits(p, N));
    const int per_split = (int)((KT + splits - 1) / splits);
    splits = (int)((KT + per_split - 1) / per_split);  // drop empty splits
    Args a;
    a.bitmaps = p.bitmaps;
    a.offsets = p.offsets;
    a.values = (const uint8_t*)p.values;
    a.X = (const uint8_t*)X;
    a.N = N;
    a.M = p.M;
    a.K = p.K;
    a.KT = p.Kp / 64;
    a.splits = splits;
    a.per_split = per_split;
    a.ws = p.ws;
    a.ws_det = (!I8 && splits > 1) ? p.ws_det : nullptr;
    a.counters = p.counters;
    a.err = p.err;
    a.Y = Y;
    a.mode = mode;
    a.row_scale = row_scale;
    a.spin_cap = bsp_spin_cap();
    a.stall_first = bsp_test_stall();
    a.tau = tau;
    dim3 grid((unsigned)splits, (unsigned)(p.Mp / 64));
    spmm_decode_kernel<NT, I8, SKIP><<<grid, C::THREADS, C::SMEM, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <bool I8, bool SKIP>
bsp_status_t dispatch_nt(const bsp_decode_problem& p, const void* X, int N, void* Y, int mode,
                         const float* row_scale, float tau, cudaStream_t s)
{
    if (N <= 1) return launch<1, I8, SKIP>(p, X, N, Y, mode, row_scale, tau, s);
    if constexpr (!SKIP) {
        if (N <= 2) return launch<2, I8, false>(p, X, N, Y, mode, row_scale, tau, s);
        if (N <= 4) return launch<4, I8, false>(p, X, N, Y, mode, row_scale, tau, s);
        if (N <= 8) return launch<8, I8, false>(p, X, N, Y, mode, row_scale, tau, s);
        return launch<16, I8, false>(p, X, N, Y, mode, row_scale, tau, s);
    }
    return BSP_ERR_INVALID_ARG;
}

}  // namespace

namespace {

int team_splits(const bsp_decode_problem& p, bool env)
{
    const int64_t strips = p.Mp / 64, KT = p.Kp / 64;
    // each team run must fit kMaxRun GTs
    const int64_t min_splits = (KT + (int64_t)kMaxRun * kTeams - 1) / ((int64_t)kMaxRun * kTeams);
    int64_t splits;
    const int64_t forced = env ? bsp_tune(BSP_TUNE_SPLITK) : 0;
    if (forced >= 1) {
        splits = forced;
    } else {
        // about 8 GTs per team run, and at least ~2 CTAs per SM
        splits = (KT + 8 * kTeams - 1) / (8 * kTeams);
        const int64_t want_ctas = 2 * (int64_t)p.num_sms;
        if (strips * splits < want_ctas) splits = (want_ctas + strips - 1) / strips;
    }
    if (splits > KT) splits = KT;
    if (splits < min_splits) splits = min_splits;
    if (splits < 1) splits = 1;
    return (int)splits;
}

}  // namespace

int bsp_decode_splits(const bsp_decode_problem& p, int N)
{
    (void)N;
    return team_splits(p, true);
}

int bsp_decode_split_cap(const bsp_decode_problem& p)
{
    const int64_t strips = p.Mp / 64, KT = p.Kp / 64;
    int cap = team_splits(p, false);
    for (int nt = 1; nt <= 2; ++nt) cap = std::max(cap, gtw_splits_auto(strips, KT, gtw_slots(p, nt)));
    cap = std::max(cap, bsp_narrow_det_slots(p));
    // cap >= the team kernel's floor (runs of at most kMaxRun GTs), so a
    // count clamped to it still satisfies that floor
    return cap;
}

bsp_status_t bsp_run_spmm_decode(const bsp_decode_problem& p, const void* X, int N, void* Y,
                                 bsp_out_mode mode, const float* row_scale,
                                 bool skip_zero_octets, cudaStream_t s, float tau)
{
    if (N < 1 || N > BSP_DECODE_MAX_N) return BSP_ERR_INVALID_ARG;
    if (skip_zero_octets && N != 1) return BSP_ERR_INVALID_ARG;
    if (!(tau >= 0.f)) return BSP_ERR_INVALID_ARG;  // also rejects NaN
    const bool i8 = p.dtype == BSP_INT8;
#ifndef BSP_DEC_GTW
#define BSP_DEC_GTW 1
#endif
    if (BSP_DEC_GTW && !i8 && mode == BSP_OUT_F16 && N <= 2) {
        if (skip_zero_octets) return launch_gtw<1, true>(p, X, N, Y, tau, s);
        return N == 1 ? launch_gtw<1, false>(p, X, N, Y, tau, s) : launch_gtw<2, false>(p, X, N, Y, tau, s);
    }
    if (i8)
        return skip_zero_octets ? dispatch_nt<true, true>(p, X, N, Y, mode, row_scale, tau, s)
                                : dispatch_nt<true, false>(p, X, N, Y, mode, row_scale, tau, s);
    return skip_zero_octets ? dispatch_nt<false, true>(p, X, N, Y, mode, row_scale, tau, s)
                            : dispatch_nt<false, false>(p, X, N, Y, mode, row_scale, tau, s);
}

bsp_decode_problem bsp_problem_of(const bsp_handle* h)
{
    bsp_decode_problem p;
    p.bitmaps = h->bitmaps;
    p.offsets = h->offsets;
    p.values = h->values;
    p.dtype = h->dtype;
    p.M = h->M;
    p.K = h->K;
    p.Mp = h->Mp;
    p.Kp = h->Kp;
    p.max_gt_nnz = h->max_gt_nnz;
    p.device = h->device;
    p.num_sms = h->num_sms;
    p.ws = h->ws;
    p.ws_det = h->deterministic ? h->ws_det : nullptr;
    p.det_slots = h->det_slots;
    p.values_bytes = h->values_alloc;
    p.counters = h->counters;
    p.err = h->err;
    return p;
}
