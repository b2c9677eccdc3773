// Tiled-CBC column index of an encoded weight and the sparse-vector product
// that fetches only the columns whose activation survives.
//
// Format: "Unified Static-Dynamic Pruning for Efficient LLM Inference"
// (SPDP), section 4.1 "Tiled-CBC: Unified Compression Format".  GTiles of
// TM x TK = 256 x 64 elements tile W row-major (M, K zero-padded); inside a
// GTile, column tiles of 256 x 1 each own four uint64 bitmaps (rows 0-63,
// 64-127, 128-191, 192-255; bit r % 64 of word r / 64 <=> element r is
// nonzero), and the GTile's nonzeros are stored column after column, top
// to bottom.  TileOffset (u32 [NGT + 1]) counts the values before each
// GTile; ColInfo (u32 per column) packs the column's first value inside its
// GTile (upper 16 bits) and its nonzero count (lower 16).
//
// Product: section 4.2's dynamic pruning, steps (1)-(3): per GTile the
// activations decide which columns are active; only their bitmaps and
// value spans are read (the ColInfo row gives their offsets), inactive
// columns cost nothing but their ColInfo word, and a GTile whose 64
// activations are all pruned is not touched at all.
//
// Kernel layout (GB300): one warp per (256-row GTile strip, run of
// BSP_CBC_PER GTile columns); lane l owns the 8 consecutive rows of byte
// l % 8 of the column's bitmap word l / 8.  Per active column a lane takes
// its byte of the column's bitmaps (one 32-B read shared by the warp), its
// rank by a masked popcount, and its (at most eight) values with predicated
// loads that the warp coalesces (the column's values are contiguous).
// Split-K partial sums meet through vector reductions in the handle's
// workspace and a programmatic dependent finishing kernel (as in the
// narrow kernel), or in per-split slots in deterministic mode.
#include "bsp_internal.cuh"

#include <algorithm>
#include <cuda_fp16.h>

namespace {

constexpr int TM = 256, TK = 64, WORDS = TM / 64;

inline unsigned grid_for(int64_t n, int block) { return (unsigned)((n + block - 1) / block); }

// ---------------------------------------------------------------- build

// Pass 1: one thread per (GTile, column): the column's four bitmap words
// and its nonzero count, read down the column of the dense W [M][K]
// (neighbouring threads take neighbouring columns: coalesced rows).
template <int EB>
__global__ void cbc_column_kernel(const uint8_t* __restrict__ W, int64_t M, int64_t K, int64_t tc, int64_t ncols,
                                  uint64_t* __restrict__ bitmaps, uint32_t* __restrict__ colnnz)
{
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= ncols) return;
    const int64_t t = idx / TK, c = idx % TK;
    const int64_t gi = t / tc, gj = t % tc;
    const int64_t col = gj * TK + c;
    uint64_t w[WORDS] = {0, 0, 0, 0};
    uint32_t n = 0;
    if (col < K) {
        for (int r = 0; r < TM; ++r) {
            const int64_t row = gi * TM + r;
            if (row >= M) break;
            const uint8_t* p = W + (row * K + col) * EB;
            const bool nz = EB == 2 ? (*reinterpret_cast<const uint16_t*>(p) != 0) : (*p != 0);
            if (nz) {
                w[r >> 6] |= 1ull << (r & 63);
                ++n;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < WORDS; ++j) bitmaps[idx * WORDS + j] = w[j];
    colnnz[idx] = n;
}

// Pass 2: one warp per GTile: ColInfo = (first value of the column inside
// the GTile) << 16 | its count, by a warp scan of the 64 counts; the
// GTile's total for the TileOffset scan.
__global__ void cbc_colinfo_kernel(const uint32_t* __restrict__ colnnz, int64_t ngt, uint32_t* __restrict__ colinfo,
                                   uint32_t* __restrict__ tile_nnz)
{
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= ngt) return;
    const uint32_t a = colnnz[t * TK + 2 * lane], b = colnnz[t * TK + 2 * lane + 1];
    uint32_t incl = a + b;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t ex = incl - a - b;
    colinfo[t * TK + 2 * lane] = (ex << 16) | a;
    colinfo[t * TK + 2 * lane + 1] = ((ex + a) << 16) | b;
    if (lane == 31) tile_nnz[t] = incl;
}

// Pass 3: one thread per (GTile, column): its nonzeros, top to bottom, to
// their slots.
template <int EB>
__global__ void cbc_values_kernel(const uint8_t* __restrict__ W, int64_t M, int64_t K, int64_t tc, int64_t ncols,
                                  const uint32_t* __restrict__ offsets, const uint32_t* __restrict__ colinfo,
                                  uint8_t* __restrict__ values)
{
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= ncols) return;
    const int64_t t = idx / TK, c = idx % TK;
    const int64_t gi = t / tc, gj = t % tc;
    const int64_t col = gj * TK + c;
    if (col >= K) return;
    uint64_t slot = (uint64_t)offsets[t] + (colinfo[idx] >> 16);
    for (int r = 0; r < TM; ++r) {
        const int64_t row = gi * TM + r;
        if (row >= M) break;
        const uint8_t* p = W + (row * K + col) * EB;
        if (EB == 2) {
            const uint16_t v = *reinterpret_cast<const uint16_t*>(p);
            if (v) reinterpret_cast<uint16_t*>(values)[slot++] = v;
        } else if (*p) {
            values[slot++] = *p;
        }
    }
}

// ---------------------------------------------------------------- product

struct CbcArgs {
    const uint32_t* offsets;
    const uint32_t* colinfo;
    const uint64_t* bitmaps;
    const uint8_t* values;
    const uint8_t* x;    // [K] fp16 or int8
    void* y;             // [M] fp16 or int32
    int64_t M, K;
    int64_t tr, tc;      // GTile rows and columns of the padded grid
    int splits, per;     // split-K: GTile columns [part * per, min(tc, (part + 1) * per))
    float tau;           // |x| <= tau is pruned (0: exact zeros); NaN is never pruned
    float* ws;           // fp32 [M] (int32 for int8), zero between calls
    float* ws_det;       // deterministic: [splits][M] fp32, or null
};

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <bool I8>
struct Acc8;
template <>
struct Acc8<false> {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
};
template <>
struct Acc8<true> {
    int32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
};

// Two active columns' share of a lane: its 8 rows are the bits of byte[q];
// the value of the first set one is values[first[q]], the others follow.
// All the loads of both columns are issued before the multiply-adds.
template <bool I8>
__device__ __forceinline__ void column8(const uint8_t* __restrict__ values, const uint32_t (&first)[2],
                                        const uint32_t (&byte)[2], const uint32_t (&xb)[2], Acc8<I8>& acc)
{
    if constexpr (I8) {
        int32_t v[2][8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int8_t* vp = reinterpret_cast<const int8_t*>(values) + first[q];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[q][i] = 0;
                if (byte[q] & (1u << i)) {
                    v[q][i] = __ldg(vp);
                    ++vp;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int32_t x = (int32_t)(int8_t)(xb[q] & 0xFF);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc.v[i] += v[q][i] * x;
        }
    } else {
        unsigned short v[2][8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const unsigned short* vp = reinterpret_cast<const unsigned short*>(values) + first[q];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[q][i] = 0;
                if (byte[q] & (1u << i)) {
                    v[q][i] = __ldg(vp);
                    ++vp;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float x = __half2float(__ushort_as_half((unsigned short)(xb[q] & 0xFFFF)));
#pragma unroll
            for (int i = 0; i < 8; ++i) acc.v[i] = fmaf(__half2float(__ushort_as_half(v[q][i])), x, acc.v[i]);
        }
    }
}

// Activations of GTile column block gj: lane l holds columns 2l, 2l + 1
// (raw bits; zero past K).
template <bool I8>
__device__ __forceinline__ uint32_t load_x_pair(const uint8_t* x, int64_t K, int64_t gj, int lane)
{
    const int64_t c0 = gj * TK + 2 * lane;
    if (c0 >= K) return 0u;  // K is even: c0 < K means c0 + 1 < K
    if constexpr (I8) return *reinterpret_cast<const uint16_t*>(x + c0);
    return *reinterpret_cast<const uint32_t*>(x + 2 * c0);
}

template <bool I8>
__device__ __forceinline__ bool active_x(uint32_t xb, float tau)
{
    if constexpr (I8) return (float)abs((int)(int8_t)(xb & 0xFF)) > tau;
    const float f = __half2float(__ushort_as_half((unsigned short)(xb & 0xFFFF)));
    return !(fabsf(f) <= tau);  // NaN stays active
}

// One entry of a warp's table of the active columns of a GTile: the
// column's four bitmap words, the values before each word's rows, the
// index of its first value and its activation.
struct ColEntry {
    uint64_t w[WORDS];
    uint32_t pre[WORDS];  // values of the column in the rows above word j
    uint32_t base;        // index of the column's first value in the values array
    uint32_t xbits;
    uint32_t pad[2];
};
static_assert(sizeof(ColEntry) == 64, "one table entry per 64 B");
constexpr int WARPS_PER_CTA = 4;

template <bool I8>
__global__ void __launch_bounds__(WARPS_PER_CTA * 32) spmspv_cbc_kernel(const CbcArgs a)
{
    constexpr uint32_t FULL = 0xFFFFFFFFu;
    __shared__ ColEntry table[WARPS_PER_CTA][TK];
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    ColEntry* tab = table[wi];
    const int64_t u = (int64_t)blockIdx.x * WARPS_PER_CTA + wi;
    const int64_t gi = u % a.tr, part = u / a.tr;
    if (part >= a.splits) return;
    const int64_t g0 = part * a.per, g1 = min(a.tc, g0 + a.per);
    const int64_t r_base = gi * TM + 8 * lane;  // the lane's 8 rows: byte lane % 8 of word lane / 8
    const int wj = lane >> 3;
    const uint32_t sh = 8u * (uint32_t)(lane & 7);
    const uint64_t below = (1ull << sh) - 1ull;
    Acc8<I8> acc;
    uint32_t xnext = g0 < g1 ? load_x_pair<I8>(a.x, a.K, g0, lane) : 0u;
    for (int64_t gj = g0; gj < g1; ++gj) {
        const uint32_t xp = xnext;
        if (gj + 1 < g1) xnext = load_x_pair<I8>(a.x, a.K, gj + 1, lane);  // the next block's, ahead
        const uint32_t xb0 = I8 ? (xp & 0xFF) : (xp & 0xFFFF), xb1 = I8 ? ((xp >> 8) & 0xFF) : (xp >> 16);
        const bool act0 = active_x<I8>(xb0, a.tau), act1 = active_x<I8>(xb1, a.tau);
        const uint32_t m0 = __ballot_sync(FULL, act0), m1 = __ballot_sync(FULL, act1);
        if ((m0 | m1) == 0u) continue;  // the whole GTile is pruned: nothing of it is read
        const int64_t t = gi * a.tc + gj;
        // the owners of the active columns (lane l: columns 2l, 2l + 1) read
        // their metadata and fill the table: even columns first, then odd
        const uint32_t toff = __ldg(a.offsets + t);
        const int n0 = __popc(m0), nact = n0 + __popc(m1);
        if (act0 | act1) {
            const uint2 info2 = *reinterpret_cast<const uint2*>(a.colinfo + t * TK + 2 * lane);
            const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
            for (int odd = 0; odd < 2; ++odd) {
                if (!(odd ? act1 : act0)) continue;
                const int c = 2 * lane + odd;
                const ulonglong2* bw = reinterpret_cast<const ulonglong2*>(a.bitmaps + (t * TK + c) * WORDS);
                const ulonglong2 p0 = __ldg(bw), p1 = __ldg(bw + 1);
                ColEntry& e = tab[odd ? n0 + __popc(m1 & lt) : __popc(m0 & lt)];
                e.w[0] = p0.x;
                e.w[1] = p0.y;
                e.w[2] = p1.x;
                e.w[3] = p1.y;
                const uint32_t c0 = (uint32_t)__popcll(p0.x), c1 = c0 + (uint32_t)__popcll(p0.y),
                               c2 = c1 + (uint32_t)__popcll(p1.x);
                e.pre[0] = 0;
                e.pre[1] = c0;
                e.pre[2] = c1;
                e.pre[3] = c2;
                e.base = toff + ((odd ? info2.y : info2.x) >> 16);
                e.xbits = odd ? xb1 : xb0;
            }
        }
        __syncwarp();
        // every lane: its 8 rows of each active column, two columns at a time
        for (int j = 0; j < nact; j += 2) {
            uint32_t byte[2], first[2], xb[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int jj = j + q < nact ? j + q : j;  // a missing second column: none of its bits
                const ColEntry& e = tab[jj];
                const uint64_t w = e.w[wj];
                byte[q] = j + q < nact ? (uint32_t)(w >> sh) & 0xFFu : 0u;
                first[q] = e.base + e.pre[wj] + (uint32_t)__popcll(w & below);
                xb[q] = j + q < nact ? e.xbits : 0u;
            }
            column8<I8>(a.values, first, byte, xb, acc);
        }
        __syncwarp();  // the table is rewritten for the next GTile
    }
    if (r_base >= a.M) return;  // rows of the zero padding (M rounded up to 256)
    const int nr = (int)(a.M - r_base < 8 ? a.M - r_base : 8);
    if (a.splits == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i >= nr) break;
            if constexpr (I8) reinterpret_cast<int32_t*>(a.y)[r_base + i] = acc.v[i];
            else reinterpret_cast<__half*>(a.y)[r_base + i] = __float2half_rn(acc.v[i]);
        }
    } else if constexpr (I8) {
        int32_t* ws = reinterpret_cast<int32_t*>(a.ws);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < nr && acc.v[i]) atomicAdd(ws + r_base + i, acc.v[i]);
    } else if (a.ws_det) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < nr) a.ws_det[part * a.M + r_base + i] = acc.v[i];
    } else if (nr == 8 && (a.M % 4) == 0) {
        red_add_v4(a.ws + r_base, acc.v[0], acc.v[1], acc.v[2], acc.v[3]);
        red_add_v4(a.ws + r_base + 4, acc.v[4], acc.v[5], acc.v[6], acc.v[7]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < nr) atomicAdd(a.ws + r_base + i, acc.v[i]);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Finishing kernel of split products: y from the workspace (cleared) or
// from the per-split slots added in split order.
template <bool I8>
__global__ void __launch_bounds__(256) spmspv_cbc_finish_kernel(void* y, float* ws, const float* ws_det, int64_t M,
                                                                int splits)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < M; r += (int64_t)gridDim.x * blockDim.x) {
        if constexpr (I8) {
            int32_t* w = reinterpret_cast<int32_t*>(ws);
            reinterpret_cast<int32_t*>(y)[r] = w[r];
            w[r] = 0;
        } else {
            float v;
            if (ws_det) {
                v = 0.f;
                for (int p = 0; p < splits; ++p) v += ws_det[(int64_t)p * M + r];
            } else {
                v = ws[r];
                ws[r] = 0.f;
            }
            reinterpret_cast<__half*>(y)[r] = __float2half_rn(v);
        }
    }
}

template <bool I8>
bsp_status_t launch_cbc(const bsp_handle* h, const void* x, void* y, float tau, cudaStream_t s)
{
    CbcArgs a = {};
    a.offsets = h->cbc_offsets;
    a.colinfo = h->cbc_colinfo;
    a.bitmaps = h->cbc_bitmaps;
    a.values = (const uint8_t*)h->cbc_values;
    a.x = (const uint8_t*)x;
    a.y = y;
    a.M = h->M;
    a.K = h->K;
    a.tr = h->cbc_tr;
    a.tc = h->cbc_tc;
    a.tau = tau;
    // runs of BSP_CBC_PER GTile columns per warp (one warp per 256-row strip
    // and run): a warp's round trips (the activations, the active columns'
    // metadata, their values) are few, and many warps hide them.  One
    // column per warp: FC2 (5120 x 20480) with ~85%-zero activations in
    // 21.5 us against 22.8 with two (calls of other layers in between).
    const int64_t halves = a.tr;
#ifndef BSP_CBC_PER
#define BSP_CBC_PER 1
#endif
    int64_t splits = std::max<int64_t>(1, (a.tc + BSP_CBC_PER - 1) / BSP_CBC_PER);
    if (const int64_t v = bsp_tune(BSP_TUNE_SPLITK)) splits = v;  // tests, tuning
    splits = std::min<int64_t>(splits, a.tc);
    if (!I8 && h->deterministic && h->ws_det) splits = std::min<int64_t>(splits, (int64_t)h->det_slots * BSP_DECODE_MAX_N);
    a.per = (int)((a.tc + splits - 1) / splits);
    a.splits = (int)((a.tc + a.per - 1) / a.per);
    a.ws = (float*)h->ws;
    a.ws_det = (!I8 && h->deterministic && a.splits > 1) ? h->ws_det : nullptr;
    const int64_t units = halves * a.splits;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    spmspv_cbc_kernel<I8><<<grid_for(units, WARPS_PER_CTA), WARPS_PER_CTA * 32, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return BSP_ERR_CUDA;
    if (a.splits == 1) return BSP_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(grid_for(h->M, 256), (int64_t)h->num_sms * 4));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, spmspv_cbc_finish_kernel<I8>, y, (float*)h->ws, (const float*)a.ws_det, h->M,
                              a.splits) == cudaSuccess
               ? BSP_OK
               : BSP_ERR_CUDA;
}

}  // namespace

bsp_status_t bsp_run_build_cbc(bsp_handle* h, cudaStream_t s)
{
    const int eb = bsp_elem_bytes(h->dtype);
    const int64_t tr = (h->M + TM - 1) / TM, tc = (h->K + TK - 1) / TK, ngt = tr * tc;
    const int64_t ncols = ngt * TK;
    uint8_t* W = nullptr;
    uint32_t *colnnz = nullptr, *tile_nnz = nullptr;
    int* overflow = nullptr;
    uint32_t* offsets = nullptr;
    uint32_t* colinfo = nullptr;
    uint64_t* bitmaps = nullptr;
    void* values = nullptr;
    bsp_status_t st = BSP_OK;
    auto fail = [&](bsp_status_t e) {
        cudaFree(offsets);
        cudaFree(colinfo);
        cudaFree(bitmaps);
        cudaFree(values);
        return e;
    };
    if (cudaMalloc(&W, (size_t)h->M * h->K * eb) != cudaSuccess || cudaMalloc(&colnnz, ncols * 4) != cudaSuccess ||
        cudaMalloc(&tile_nnz, ngt * 4) != cudaSuccess || cudaMalloc(&overflow, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&offsets, (ngt + 1) * 4) != cudaSuccess || cudaMalloc(&colinfo, ncols * 4) != cudaSuccess ||
        cudaMalloc(&bitmaps, ncols * WORDS * 8) != cudaSuccess)
        st = BSP_ERR_OOM;
    if (st == BSP_OK) st = bsp_run_decode(h, W, s);
    if (st == BSP_OK) {
        if (eb == 2)
            cbc_column_kernel<2><<<grid_for(ncols, 256), 256, 0, s>>>(W, h->M, h->K, tc, ncols, bitmaps, colnnz);
        else
            cbc_column_kernel<1><<<grid_for(ncols, 256), 256, 0, s>>>(W, h->M, h->K, tc, ncols, bitmaps, colnnz);
        cbc_colinfo_kernel<<<grid_for(ngt * 32, 256), 256, 0, s>>>(colnnz, ngt, colinfo, tile_nnz);
        if (cudaMemsetAsync(overflow, 0, sizeof(int), s) != cudaSuccess) st = BSP_ERR_CUDA;
    }
    if (st == BSP_OK) st = bsp_exclusive_scan_u32(tile_nnz, ngt, offsets, overflow, s);
    uint32_t total = 0;
    int ovf = 0;
    if (st == BSP_OK && (cudaMemcpyAsync(&total, offsets + ngt, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                         cudaMemcpyAsync(&ovf, overflow, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                         cudaStreamSynchronize(s) != cudaSuccess))
        st = BSP_ERR_CUDA;
    if (st == BSP_OK && (ovf || total != h->NNZ)) st = BSP_ERR_INTERNAL;  // the same nonzeros as the handle
    const size_t vbytes = ((size_t)total * eb + 16 + 15) & ~(size_t)15;
    if (st == BSP_OK && cudaMalloc(&values, vbytes) != cudaSuccess) st = BSP_ERR_OOM;
    if (st == BSP_OK) {
        if (cudaMemsetAsync(values, 0, vbytes, s) != cudaSuccess) st = BSP_ERR_CUDA;
        if (eb == 2)
            cbc_values_kernel<2><<<grid_for(ncols, 256), 256, 0, s>>>(W, h->M, h->K, tc, ncols, offsets, colinfo,
                                                                      (uint8_t*)values);
        else
            cbc_values_kernel<1><<<grid_for(ncols, 256), 256, 0, s>>>(W, h->M, h->K, tc, ncols, offsets, colinfo,
                                                                      (uint8_t*)values);
        if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) st = BSP_ERR_CUDA;
    }
    cudaFree(W);
    cudaFree(colnnz);
    cudaFree(tile_nnz);
    cudaFree(overflow);
    if (st != BSP_OK) return fail(st);
    cudaFree(h->cbc_offsets);
    cudaFree(h->cbc_colinfo);
    cudaFree(h->cbc_bitmaps);
    cudaFree(h->cbc_values);
    h->cbc_offsets = offsets;
    h->cbc_colinfo = colinfo;
    h->cbc_bitmaps = bitmaps;
    h->cbc_values = values;
    h->cbc_tr = tr;
    h->cbc_tc = tc;
    return BSP_OK;
}

bsp_status_t bsp_run_spmspv_cbc(const bsp_handle* h, const void* x, void* y, float tau, cudaStream_t s)
{
    return h->dtype == BSP_INT8 ? launch_cbc<true>(h, x, y, tau, s) : launch_cbc<false>(h, x, y, tau, s);
}
