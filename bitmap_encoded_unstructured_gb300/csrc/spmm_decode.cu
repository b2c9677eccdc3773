// Decode-path product Y = W * X for N <= 16 on CUDA cores, and the
// zero-skipping sparse-vector product.
//
// Method (SpInfer's shared-memory bitmap decoding, "SpInfer: How bitmaps
// make sparse LLMs actually fast", sections "Shared Memory Bitmap Decoding
// (SMBD)" and "The async pipeline"; split-K over GroupTiles with a
// reduction workspace as in "Unified Static-Dynamic Pruning for Efficient
// LLM Inference", section 4.2.3 and its Algorithm 1 epilogue; a producer
// lane that prefetches the next tiles while the warp computes, as in
// "UnionSparse: ...", section on the DW-PC pipeline):
//
//  * grid = (splits, M/64): a CTA owns one 64-row strip of W (one GT row)
//    and a contiguous range of GT columns; each of its warps takes a
//    contiguous run of at most 31 GTs of that range.
//  * each warp runs its own S-stage ring in shared memory.  Lane 0 is the
//    producer: for GT i+S it issues 1-D bulk copies (cp.async.bulk, the
//    copy engine, no registers involved) of the GT's 64 bitmaps (512 B),
//    its packed value span (the 16-B aligned superset of
//    [offsets[t], offsets[t+1])) and the N rows of the X tile, all
//    completing on the stage's mbarrier; meanwhile all 32 lanes decode and
//    multiply GT i.
//  * per GT: popcount of each BT and a warp exclusive scan (shfl) give the
//    BT value bases; the X tile is widened to fp32 / int32 [64][N].
//  * decode + multiply: lane l owns GT rows l and l+32.  For each of the 8
//    BTs on a row it takes the row's byte of the bitmap, finds the first
//    value by a masked popcount (nonzeros of the earlier rows of the BT),
//    then walks the set bits: acc[n] += w * x[col][n].
//  * the warps' partial sums are added in shared memory; with one split the
//    CTA writes Y, otherwise it adds into the handle's workspace and the
//    last CTA of the strip (arrival counter) converts, writes Y and clears
//    the workspace and counter for the next call.
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
// Every wait is bounded (bspx::kSpinCap); a wait that gives up records
// BSP_ERR_TIMEOUT in the handle's error word, drains its own copies (again
// bounded) and returns.
#include "bsp_internal.cuh"
#include "bsp_ptx.cuh"

#include <cstdlib>
#include <type_traits>

namespace {

__device__ __forceinline__ int bt_local(int br, int bc)
{
    return (((br >> 1) * 4 + (bc >> 1)) << 2) + (br & 1) + ((bc & 1) << 1);
}

constexpr int kMaxRun = 31;  // GTs per warp run (offsets of a run fit one warp register)

template <int NT, bool I8>
struct DecCfg {
    static constexpr int WARPS = 4;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int S = 2;                        // pipeline stages per warp
    static constexpr int EB = I8 ? 1 : 2;
    static constexpr int E16 = 16 / EB;                // elements per 16-B chunk
    static constexpr int VAL_CHUNKS = 4096 / E16 + 1;  // dense GT + misalignment
    static constexpr bool WIDE_X = !I8 && NT >= 4;     // fp32 X tile + packed fp32x2 FMA
    static constexpr int XS = WIDE_X ? NT + 4 : 4;     // widened X-tile row stride (floats)
    static constexpr int XRAW = NT * 64 * EB;          // raw X tile bytes [NT][64]
    // stage layout
    static constexpr int ST_BM = 0;
    static constexpr int ST_X = ST_BM + 512;
    static constexpr int ST_VAL = ST_X + ((XRAW + 15) & ~15);
    static constexpr int STAGE = ST_VAL + VAL_CHUNKS * 16;
    // warp slice layout
    static constexpr int W_STAGES = 0;
    static constexpr int W_XS = S * STAGE;
    static constexpr int W_BASE = W_XS + ((64 * XS * 4 + 15) & ~15);
    static constexpr int W_BAR = W_BASE + 64 * 4;
    static constexpr int WARP_BYTES = (W_BAR + 2 * S * 8 + 15) & ~15;
    static constexpr int SMEM = WARPS * WARP_BYTES;
    static constexpr int RED_BYTES = 64 * NT * 4;      // per-warp reduction buffer (aliases stage 0)
    static_assert(RED_BYTES <= STAGE, "reduction buffer must fit a stage");
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

// fp32 += fp16 * fp16, one rounding (the fp16 product is exact in fp32)
__device__ __forceinline__ void fma_f16(float& acc, uint16_t w, uint16_t x)
{
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(w), "h"(x));
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

// Accumulator storage of one lane: rows l and l+32, NT columns of Y.
template <int NT, bool I8, bool WIDE>
struct Accum;
template <int NT>
struct Accum<NT, false, false> { float v[2][NT]; };
template <int NT>
struct Accum<NT, false, true> { uint64_t v[2][NT / 2]; };  // packed fp32 pairs
template <int NT>
struct Accum<NT, true, false> { int v[2][NT]; };

// Decode one GroupTile and multiply it into the lane's two rows.
//
// Lane l owns GT rows l and l+32 (BT rows l/8 and l/8+4, BT row-byte l%8).
// BT columns (K-octets) are taken in turn; inside one, the positions
// c = 0..7 of the lane's row-byte are a static loop: a set bit loads the
// next packed value (the masked popcount gives the row-byte's first slot,
// then a running index), a clear bit contributes zero.  So all 32 lanes
// run the same instruction stream, and X can sit in registers.
template <int NT, bool I8, bool SKIP, typename A>
__device__ __forceinline__ void decode_gt(const uint64_t* bm_st, const uint32_t* base_s,
                                          const uint8_t* vals, const uint8_t* xraw, const float* x_s,
                                          int N, uint32_t act8, int lane, A& acc)
{
    using C = DecCfg<NT, I8>;
    const int rr = lane & 7;
    const uint64_t lowmask = (1ull << (8 * rr)) - 1ull;
#pragma unroll 1
    for (int bc = 0; bc < 8; ++bc) {
        if (SKIP && !((act8 >> bc) & 1u)) continue;
        uint32_t byte[2], idx[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gl = bt_local((lane >> 3) + 4 * h, bc);
            const uint64_t bm = bm_st[gl];
            byte[h] = (uint32_t)(bm >> (8 * rr)) & 0xFFu;
            idx[h] = base_s[gl] + (uint32_t)__popcll(bm & lowmask);
        }
        if constexpr (I8) {
            // dense int8 row-byte packed into two words, then dp4a per column of Y
            const int8_t* v8 = reinterpret_cast<const int8_t*>(vals);
            uint32_t xlo[NT], xhi[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint2 q = *reinterpret_cast<const uint2*>(xraw + n * 64 + 8 * bc);
                xlo[n] = n < N ? q.x : 0u;
                xhi[n] = n < N ? q.y : 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t wlo = 0, whi = 0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if ((byte[h] >> c) & 1u) {
                        const uint32_t b = (uint32_t)(uint8_t)v8[idx[h]];
                        ++idx[h];
                        if (c < 4) wlo |= b << (8 * c);
                        else whi |= b << (8 * (c - 4));
                    }
                }
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    acc.v[h][n] = __dp4a((int)wlo, (int)xlo[n], acc.v[h][n]);
                    acc.v[h][n] = __dp4a((int)whi, (int)xhi[n], acc.v[h][n]);
                }
            }
        } else if constexpr (!C::WIDE_X) {
            // N <= 2: fp16 X octet in registers, mixed-precision FMA
            const uint16_t* vh = reinterpret_cast<const uint16_t*>(vals);
            uint4 xq[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n)
                xq[n] = n < N ? *reinterpret_cast<const uint4*>(xraw + (n * 64 + 8 * bc) * 2) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint16_t w = 0;
                    if ((byte[h] >> c) & 1u) {
                        w = vh[idx[h]];
                        ++idx[h];
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n) fma_f16(acc.v[h][n], w, half_of(xq[n], c));
                }
            }
        } else {
            // N >= 4: fp32 X rows (broadcast loads), packed fp32x2 FMA
            const uint16_t* vh = reinterpret_cast<const uint16_t*>(vals);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint64_t xv[NT / 2];
                const float* xr = x_s + (bc * 8 + c) * C::XS;
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

__device__ __forceinline__ float ws_take(float* p) { return atomicExch(p, 0.0f); }
__device__ __forceinline__ int ws_take(int* p) { return atomicExch(p, 0); }

struct Args {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const uint8_t* values;
    const uint8_t* X;
    int N;
    int64_t M, K;
    int splits, per_split;
    void* ws;
    uint32_t* counters;
    int* err;
    void* Y;
    int mode;
    const float* row_scale;
    uint32_t spin_cap;  // polls before a wait gives up
    int stall_first;    // test only: skip the copies of each warp's first GT
};

template <int NT, bool I8, bool SKIP>
__global__ void __launch_bounds__(DecCfg<NT, I8>::THREADS)
spmm_decode_kernel(const Args a)
{
    using C = DecCfg<NT, I8>;
    using Acc = std::conditional_t<I8, int, float>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_last;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t* wb = smem + warp * C::WARP_BYTES;
    float* x_s = reinterpret_cast<float*>(wb + C::W_XS);
    uint32_t* base_s = reinterpret_cast<uint32_t*>(wb + C::W_BASE);
    uint64_t* bar_a = reinterpret_cast<uint64_t*>(wb + C::W_BAR);      // [S]: bitmaps+x (+values)
    uint64_t* bar_v = bar_a + C::S;                                      // [S]: values (spMspV)

    const int64_t K = a.K, M = a.M;
    const int64_t KT = K >> 6;
    const int64_t gi = blockIdx.y;
    const int64_t k_begin = (int64_t)blockIdx.x * a.per_split;
    const int64_t k_cnt = min((int64_t)a.per_split, KT - k_begin);
    const int run = (int)((k_cnt + C::WARPS - 1) / C::WARPS);
    const int64_t g0 = k_begin + (int64_t)warp * run;                    // first GT column of the run
    const int cnt = (int)max((int64_t)0, min((int64_t)run, k_begin + k_cnt - g0));
    const int64_t t0 = gi * KT + g0;
    const int N = a.N;

    // offsets of the run: lane i holds offsets[t0 + i]  (cnt <= 31)
    const uint32_t offv = (cnt > 0 && lane <= cnt) ? __ldg(a.offsets + t0 + lane) : 0u;

    if (lane == 0) {
        for (int s = 0; s < C::S; ++s) {
            bspx::mbar_init(bar_a + s, 1);
            bspx::mbar_init(bar_v + s, 1);
        }
        bspx::fence_mbar_init();
    }
    __syncwarp();

    auto stage_ptr = [&](int s) { return wb + C::W_STAGES + s * C::STAGE; };

    // Producer: metadata (bitmaps + X rows) of GT i into stage s; with
    // `with_values` also its whole value span, on the same barrier.
    auto issue_meta = [&](int i, int s, bool with_values, uint32_t o0, uint32_t o1) {
        uint8_t* st = stage_ptr(s);
        const int64_t t = t0 + i, gj = g0 + i;
        uint32_t bytes = 512 + (uint32_t)(N * 64 * C::EB);
        uint32_t ch0 = 0, nch = 0;
        if (with_values) {
            ch0 = o0 / C::E16;
            nch = (o1 + C::E16 - 1) / C::E16 - ch0;
            bytes += nch * 16;
        }
        bspx::mbar_arrive_expect_tx(bar_a + s, bytes);
        bspx::bulk_g2s(st + C::ST_BM, a.bitmaps + t * 64, 512, bar_a + s);
        for (int n = 0; n < N; ++n)
            bspx::bulk_g2s(st + C::ST_X + n * 64 * C::EB, a.X + ((int64_t)n * K + gj * 64) * C::EB,
                           64 * C::EB, bar_a + s);
        if (with_values && nch)
            bspx::bulk_g2s(st + C::ST_VAL, a.values + (int64_t)ch0 * 16, nch * 16, bar_a + s);
    };

    Accum<NT, I8, C::WIDE_X> acc;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < (C::WIDE_X ? NT / 2 : NT); ++n) acc.v[h][n] = 0;

    bool failed = false;

    // Spmspv only: once the metadata of GT i is in, issue its active value
    // segments on bar_v[s].  All lanes call this (it reads the bitmaps).
    auto issue_values_skip = [&](int i, int s) {
        uint8_t* st = stage_ptr(s);
        const uint32_t o0 = __shfl_sync(0xFFFFFFFFu, offv, i);
        const uint32_t ch0 = o0 / C::E16, shift = o0 - ch0 * C::E16;
        const uint64_t b0 = reinterpret_cast<const uint64_t*>(st + C::ST_BM)[2 * lane];
        const uint64_t b1 = reinterpret_cast<const uint64_t*>(st + C::ST_BM)[2 * lane + 1];
        const uint32_t seg = __popcll(b0) + __popcll(b1);
        uint32_t incl = seg;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t ex = incl - seg;
        // activity of octet (lane & 7): x[8j .. 8j+7] of this GT
        const uint8_t* xr = st + C::ST_X;
        bool act = false;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            Acc v0, v1;
            if (c % 2 == 0) {
                x_pair(xr, (lane & 7) * 8 + c, v0, v1);
                act |= (v0 != Acc(0)) || (v1 != Acc(0));
            }
        }
        uint32_t q0 = 0, q1 = 0;
        if (act && seg) {
            q0 = (ex + shift) / C::E16;
            q1 = (ex + seg + shift + C::E16 - 1) / C::E16;
        }
        uint32_t bytes = (q1 - q0) * 16;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) bytes += __shfl_xor_sync(0xFFFFFFFFu, bytes, d);
        if (lane == 0) bspx::mbar_arrive_expect_tx(bar_v + s, bytes);
        __syncwarp();
        if (q1 > q0)
            bspx::bulk_g2s(st + C::ST_VAL + q0 * 16, a.values + ((int64_t)ch0 + q0) * 16, (q1 - q0) * 16,
                           bar_v + s);
    };

    // prologue: fill the ring
    for (int i = 0; i < C::S && i < cnt; ++i) {
        const uint32_t p0 = __shfl_sync(0xFFFFFFFFu, offv, i);
        const uint32_t p1 = __shfl_sync(0xFFFFFFFFu, offv, i + 1);
        if (lane == 0 && !(a.stall_first && i == 0)) issue_meta(i, i, !SKIP, p0, p1);
    }
    int issued = cnt < C::S ? cnt : C::S;   // GTs whose metadata copies were issued
    int valued = 0;                          // spMspV: GTs whose value copies were issued

    if constexpr (SKIP) {
        if (cnt > 0) {
            if (!__all_sync(0xFFFFFFFFu, bspx::mbar_wait_bounded(bar_a + 0, 0, a.spin_cap))) failed = true;
            if (!failed) { issue_values_skip(0, 0); valued = 1; }
        }
    }
    int i_fail = 0;

    for (int i = 0; i < cnt && !failed; ++i) {
        i_fail = i;
        const int s = i % C::S;
        const uint32_t ph = (uint32_t)((i / C::S) & 1);
        uint8_t* st = stage_ptr(s);
        const uint32_t o0 = __shfl_sync(0xFFFFFFFFu, offv, i);

        if constexpr (SKIP) {
            // metadata of GT i+1 is (or will be) in; fetch its active values now
            if (i + 1 < cnt) {
                const int s1 = (i + 1) % C::S;
                const uint32_t ph1 = (uint32_t)(((i + 1) / C::S) & 1);
                if (!__all_sync(0xFFFFFFFFu, bspx::mbar_wait_bounded(bar_a + s1, ph1, a.spin_cap))) { failed = true; break; }
                issue_values_skip(i + 1, s1);
                valued = i + 2;
            }
            if (!__all_sync(0xFFFFFFFFu, bspx::mbar_wait_bounded(bar_v + s, ph, a.spin_cap))) { failed = true; break; }
        } else {
            if (!__all_sync(0xFFFFFFFFu, bspx::mbar_wait_bounded(bar_a + s, ph, a.spin_cap))) { failed = true; break; }
        }

        // BT value bases: popcounts and a warp exclusive scan
        const uint64_t* bm_st = reinterpret_cast<const uint64_t*>(st + C::ST_BM);
        const uint64_t b0 = bm_st[2 * lane], b1 = bm_st[2 * lane + 1];
        const uint32_t c0 = __popcll(b0), c1 = __popcll(b1);
        uint32_t incl = c0 + c1;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t ex = incl - (c0 + c1);
        const uint32_t shift = o0 - (o0 / C::E16) * C::E16;
        // bases are stored with the span misalignment folded in
        base_s[2 * lane] = ex + shift;
        base_s[2 * lane + 1] = ex + c0 + shift;

        const uint8_t* xraw = st + C::ST_X;
        if constexpr (C::WIDE_X) {
            // X tile widened to fp32 [64][XS]; lane owns columns 2*lane, 2*lane+1
            float xa[NT], xb[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n < N) {
                    x_pair(xraw, n * 64 + 2 * lane, xa[n], xb[n]);
                } else {
                    xa[n] = 0.f;
                    xb[n] = 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < NT; j += 4) {
                *reinterpret_cast<float4*>(x_s + (2 * lane) * C::XS + j) = make_float4(xa[j], xa[j + 1], xa[j + 2], xa[j + 3]);
                *reinterpret_cast<float4*>(x_s + (2 * lane + 1) * C::XS + j) = make_float4(xb[j], xb[j + 1], xb[j + 2], xb[j + 3]);
            }
        }
        uint32_t act8 = 0xFFu;
        if constexpr (SKIP) {
            // K-octet j is active iff one of x[8j .. 8j+7] is nonzero
            Acc va, vb;
            x_pair(xraw, 2 * lane, va, vb);
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, (va != Acc(0)) || (vb != Acc(0)));
            act8 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) act8 |= (((bal >> (4 * j)) & 0xFu) ? 1u : 0u) << j;
        }
        __syncwarp();

        decode_gt<NT, I8, SKIP>(bm_st, base_s, st + C::ST_VAL, xraw, x_s, N, act8, lane, acc);
        __syncwarp();

        // refill this stage with GT i+S
        if (i + C::S < cnt) {
            const uint32_t p0 = __shfl_sync(0xFFFFFFFFu, offv, i + C::S);
            const uint32_t p1 = __shfl_sync(0xFFFFFFFFu, offv, i + C::S + 1);
            if (lane == 0) issue_meta(i + C::S, s, !SKIP, p0, p1);
            issued = i + C::S + 1;
        }
    }

    if (failed) {
        // a wait gave up: record the timeout, then let this warp's copies
        // that are still in flight land (each wait bounded) before leaving
        if (lane == 0) atomicExch(a.err, (int)BSP_ERR_TIMEOUT);
        for (int j = i_fail; j < issued; ++j)
            bspx::mbar_wait_bounded(bar_a + (j % C::S), (uint32_t)((j / C::S) & 1), a.spin_cap);
        if constexpr (SKIP)
            for (int j = i_fail; j < valued; ++j)
                bspx::mbar_wait_bounded(bar_v + (j % C::S), (uint32_t)((j / C::S) & 1), a.spin_cap);
    }

    // ---- CTA reduction over warps, then output or split-K accumulation
    __syncthreads();
    Acc* red = reinterpret_cast<Acc*>(wb + C::W_STAGES);  // stage 0 is free now
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if constexpr (C::WIDE_X) {
#pragma unroll
            for (int j = 0; j < NT / 2; ++j) {
                const float2 f = unpack2(acc.v[h][j]);
                red[(lane + 32 * h) * NT + 2 * j] = f.x;
                red[(lane + 32 * h) * NT + 2 * j + 1] = f.y;
            }
        } else {
#pragma unroll
            for (int n = 0; n < NT; ++n) red[(lane + 32 * h) * NT + n] = acc.v[h][n];
        }
    }
    __syncthreads();

    Acc* ws = reinterpret_cast<Acc*>(a.ws);
    for (int i = threadIdx.x; i < 64 * NT; i += C::THREADS) {
        const int r = i / NT, n = i % NT;
        Acc sum = Acc(0);
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w)
            sum += reinterpret_cast<const Acc*>(smem + w * C::WARP_BYTES + C::W_STAGES)[i];
        if (n < N) {
            const int64_t m = gi * 64 + r;
            if (a.splits == 1)
                write_out(a.Y, a.mode, (int64_t)n * M + m, sum, a.row_scale ? a.row_scale[m] : 1.0f);
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
        const Acc v = ws_take(ws + (int64_t)n * M + m);
        write_out(a.Y, a.mode, (int64_t)n * M + m, v, a.row_scale ? a.row_scale[m] : 1.0f);
    }
    if (threadIdx.x == 0) a.counters[gi] = 0u;
}

template <int NT, bool I8, bool SKIP>
bsp_status_t launch(const bsp_handle* h, const void* X, int N, void* Y, int mode,
                    const float* row_scale, cudaStream_t s)
{
    using C = DecCfg<NT, I8>;
    // the opt-in shared-memory size is set once per device
    static bool attr_done[64] = {};
    if (h->device < 0 || h->device >= 64) return BSP_ERR_INVALID_ARG;
    if (!attr_done[h->device]) {
        if (cudaFuncSetAttribute(spmm_decode_kernel<NT, I8, SKIP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return BSP_ERR_CUDA;
        attr_done[h->device] = true;
    }
    const int64_t KT = h->K / 64;
    int splits = bsp_decode_splits(h, N);
    const int per_split = (int)((KT + splits - 1) / splits);
    splits = (int)((KT + per_split - 1) / per_split);  // drop empty splits
    Args a;
    a.bitmaps = h->bitmaps;
    a.offsets = h->offsets;
    a.values = (const uint8_t*)h->values;
    a.X = (const uint8_t*)X;
    a.N = N;
    a.M = h->M;
    a.K = h->K;
    a.splits = splits;
    a.per_split = per_split;
    a.ws = h->ws;
    a.counters = h->counters;
    a.err = h->err;
    a.Y = Y;
    a.mode = mode;
    a.row_scale = row_scale;
    a.spin_cap = bspx::kSpinCap;
    if (const char* e = std::getenv("BSP_SPIN_CAP")) a.spin_cap = (uint32_t)std::strtoul(e, nullptr, 10);
    a.stall_first = std::getenv("BSP_TEST_STALL") != nullptr;
    dim3 grid((unsigned)splits, (unsigned)(h->M / 64));
    spmm_decode_kernel<NT, I8, SKIP><<<grid, C::THREADS, C::SMEM, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <bool I8, bool SKIP>
bsp_status_t dispatch_nt(const bsp_handle* h, const void* X, int N, void* Y, int mode,
                         const float* row_scale, cudaStream_t s)
{
    if (N <= 1) return launch<1, I8, SKIP>(h, X, N, Y, mode, row_scale, s);
    if constexpr (!SKIP) {
        if (N <= 2) return launch<2, I8, false>(h, X, N, Y, mode, row_scale, s);
        if (N <= 4) return launch<4, I8, false>(h, X, N, Y, mode, row_scale, s);
        if (N <= 8) return launch<8, I8, false>(h, X, N, Y, mode, row_scale, s);
        return launch<16, I8, false>(h, X, N, Y, mode, row_scale, s);
    }
    return BSP_ERR_INVALID_ARG;
}

}  // namespace

int bsp_decode_splits(const bsp_handle* h, int N)
{
    (void)N;
    const int64_t strips = h->M / 64, KT = h->K / 64;
    const int warps = 4;
    // each warp run must fit kMaxRun GTs
    const int64_t min_splits = (KT + (int64_t)kMaxRun * warps - 1) / ((int64_t)kMaxRun * warps);
    int64_t splits;
    if (const char* e = std::getenv("BSP_SPLITK")) {
        splits = std::atol(e);
    } else {
        // about 8 GTs per warp run, and at least ~2 CTAs per SM
        splits = (KT + 8 * warps - 1) / (8 * warps);
        const int64_t want_ctas = 2 * (int64_t)h->num_sms;
        if (strips * splits < want_ctas) splits = (want_ctas + strips - 1) / strips;
    }
    if (splits > KT) splits = KT;
    if (splits < min_splits) splits = min_splits;
    if (splits < 1) splits = 1;
    (void)strips;
    return (int)splits;
}

bsp_status_t bsp_run_spmm_decode(const bsp_handle* h, const void* X, int N, void* Y,
                                 bsp_out_mode mode, const float* row_scale,
                                 bool skip_zero_octets, cudaStream_t s)
{
    if (N < 1 || N > BSP_DECODE_MAX_N) return BSP_ERR_INVALID_ARG;
    if (skip_zero_octets && N != 1) return BSP_ERR_INVALID_ARG;
    const bool i8 = h->dtype == BSP_INT8;
    if (i8)
        return skip_zero_octets ? dispatch_nt<true, true>(h, X, N, Y, mode, row_scale, s)
                                : dispatch_nt<true, false>(h, X, N, Y, mode, row_scale, s);
    return skip_zero_octets ? dispatch_nt<false, true>(h, X, N, Y, mode, row_scale, s)
                            : dispatch_nt<false, false>(h, X, N, Y, mode, row_scale, s);
}
