// IE-BME: low-bit union-bitmap format and its decode-path product
// ("UnionSparse", sections "IE-BME" and "LSPD").
//
// Format (64 x 64 local tiles over the zero-padded grid, row-major; 2 x 2
// areas of 32 x 32, area a = 2 ra + ca):
//   masks    u64 [NLT][16]   the 32 x 32 union mask of each LT, row-major,
//                            leftmost position in the LSB (row i = 32-bit
//                            word i of the LT)
//   offsets  u32 [NLT + 1]   value counts: o_t = sum of 4 P_t before t
//   values   int8 (or int4, two per byte, low nibble first): LT t's area a
//                            stream at value index o_t + a P_t + rank
// Position (i, j) is active iff one of the four values W[ra 32 + i][ca 32 + j]
// of the LT is nonzero; every area then stores its value at the position's
// rank (zeros included), so one rank indexes all four streams.
//
// Product (N <= 16 per launch, int32 exact), on CUDA cores: the tensor
// cores' integer rate is far below their floating-point rate on this GPU,
// and the four-way byte dot product dp4a takes four positions per
// instruction.  CTA = 4 warps, grid (splits, 64-row strips); each warp takes
// every fourth LT column of its split and runs its own two-stage ring of
// bulk copies (union mask 128 B, the N rows of X for the LT's 64 columns,
// the LT's value span rounded out to 16 B).  LSPD per lane: lane i owns
// logical row i; a warp prefix of the row popcounts gives the row's first
// rank, a masked popcount the first rank of each 4-position segment; for
// each area the four values from that rank on are fetched as one unaligned
// 32-bit word and one prmt expands them over the segment's active
// positions (zeros elsewhere); dp4a against four X values per column of Y.
// Split-K through an int32 workspace (exact and order-independent) and a
// per-strip arrival counter; the last CTA of a strip writes Y.
#include "bsp_internal.cuh"
#include "bsp_ptx.cuh"

#include <cstdlib>
#include <new>
#include <thread>
#include <vector>

#define BSP_UNION_MAGIC 0xB5B1E0BEu

struct bsp_union {
    uint32_t magic;
    int device, num_sms;
    int bits;                 // 4 or 8
    int64_t M, K, Mp, Kp;     // logical and padded shape
    int64_t NLT;              // local tiles of the padded grid
    uint64_t nnz;             // nonzero weights
    uint64_t total;           // stored values (offsets[NLT])
    uint64_t value_bytes;     // bytes of the packed values (closed form)
    uint64_t* masks;          // [NLT * 16]
    uint32_t* offsets;        // [NLT + 1]
    uint8_t* values;          // [value_bytes + 32 zeroed slack]
    uint8_t* perms;           // row reordering: [NLT][64], row k of LT t is row perms[64 t + k]; or null
    int32_t* ws;              // split-K workspace [16][M], zero between calls
    uint32_t* counters;       // [Mp / 64], zero between calls
    int* err;
};

namespace {

constexpr int LT = 64, HALF = 32;
constexpr uint32_t FULL = 0xFFFFFFFFu;

bool valid(const bsp_union* h) { return h != nullptr && h->magic == BSP_UNION_MAGIC; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

inline unsigned blocks_for(int64_t n, int block) { return (unsigned)((n + block - 1) / block); }

__device__ __forceinline__ int w_at(const int8_t* W, int64_t M, int64_t K, int64_t r, int64_t c)
{
    return (r < M && c < K) ? (int)W[r * K + c] : 0;
}

// Row of the LT that takes place k (0..63) of its reordered layout.
__device__ __forceinline__ int lt_row(const uint8_t* perms, int64_t t, int k)
{
    return perms ? (int)perms[t * LT + k] : k;
}

// Grouped activity of every row of every LT (bit j: one of the row's values
// in columns j and 32 + j of the LT is nonzero), for the row reordering.
// One warp per LT, lane l: rows l and 32 + l.
__global__ void ub_rowact_kernel(const int8_t* __restrict__ W, int64_t M, int64_t K, int64_t KT, int64_t NLT,
                                 uint64_t* __restrict__ act)
{
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int l = threadIdx.x & 31;
    if (t >= NLT) return;
    const int64_t r0 = (t / KT) * LT, c0 = (t % KT) * LT;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint64_t a = 0;
        for (int j = 0; j < HALF; ++j)
            if (w_at(W, M, K, r0 + h * HALF + l, c0 + j) != 0 || w_at(W, M, K, r0 + h * HALF + l, c0 + HALF + j) != 0)
                a |= 1ull << j;
        act[t * LT + h * HALF + l] = a;
    }
}

// Pass 1, one warp per LT, lane i = logical row i: the row's union word
// (bit j: one of the four area values at (i, j) is nonzero), 4 P_t per LT,
// the nonzero count, and a flag for values outside the b-bit range.
__global__ void ub_mask_kernel(const int8_t* __restrict__ W, int64_t M, int64_t K, int64_t KT, int64_t NLT,
                               int bits, const uint8_t* __restrict__ perms, uint32_t* __restrict__ masks32,
                               uint32_t* __restrict__ counts, unsigned long long* nnz, int* bad)
{
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int i = threadIdx.x & 31;
    if (t >= NLT) return;
    const int64_t r0 = (t / KT) * LT, c0 = (t % KT) * LT;
    const int lo = -(1 << (bits - 1)), hi = (1 << (bits - 1)) - 1;
    uint32_t row = 0;
    int nz = 0, out = 0;
    for (int j = 0; j < HALF; ++j) {
        bool any = false;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int v = w_at(W, M, K, r0 + lt_row(perms, t, (a >> 1) * HALF + i), c0 + (a & 1) * HALF + j);
            any |= v != 0;
            nz += v != 0;
            out |= (v < lo) | (v > hi);
        }
        row |= (any ? 1u : 0u) << j;
    }
    masks32[t * 32 + i] = row;
    int p = __popc(row);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        p += __shfl_xor_sync(FULL, p, d);
        nz += __shfl_xor_sync(FULL, nz, d);
    }
    out = __any_sync(FULL, out);
    if (i == 0) {
        counts[t] = 4u * (uint32_t)p;
        atomicAdd(nnz, (unsigned long long)nz);
        if (out) atomicExch(bad, 1);
    }
}

// Pass 2, one warp per LT: every area's value at every active position, at
// value index o_t + a P_t + rank (int4: nibbles OR-ed into zeroed words).
__global__ void ub_pack_kernel(const int8_t* __restrict__ W, int64_t M, int64_t K, int64_t KT, int64_t NLT,
                               int bits, const uint8_t* __restrict__ perms, const uint32_t* __restrict__ masks32,
                               const uint32_t* __restrict__ offsets, uint8_t* __restrict__ values)
{
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int i = threadIdx.x & 31;
    if (t >= NLT) return;
    const int64_t r0 = (t / KT) * LT, c0 = (t % KT) * LT;
    const uint32_t row = masks32[t * 32 + i];
    const uint32_t pc = __popc(row);
    uint32_t incl = pc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, incl, d);
        if (i >= d) incl += o;
    }
    const uint32_t P = __shfl_sync(FULL, incl, 31);
    const uint32_t base = incl - pc;
    const uint64_t o = offsets[t];
    for (int j = 0; j < HALF; ++j) {
        if (!((row >> j) & 1u)) continue;
        const uint32_t r = base + __popc(row & ((1u << j) - 1u));
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int v = w_at(W, M, K, r0 + lt_row(perms, t, (a >> 1) * HALF + i), c0 + (a & 1) * HALF + j);
            const uint64_t e = o + (uint64_t)a * P + r;
            if (bits == 8)
                values[e] = (uint8_t)(int8_t)v;
            else
                atomicOr(reinterpret_cast<unsigned int*>(values) + (e >> 3), ((unsigned)v & 0xFu) << (4 * (e & 7)));
        }
    }
}

// W back from the arrays (round trip), one warp per LT, lane i = row i.
__global__ void ub_decode_kernel(const uint32_t* __restrict__ masks32, const uint32_t* __restrict__ offsets,
                                 const uint8_t* __restrict__ values, const uint8_t* __restrict__ perms, int bits,
                                 int64_t M, int64_t K, int64_t KT, int64_t NLT, int8_t* __restrict__ W)
{
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int i = threadIdx.x & 31;
    if (t >= NLT) return;
    const int64_t r0 = (t / KT) * LT, c0 = (t % KT) * LT;
    const uint32_t row = masks32[t * 32 + i];
    const uint32_t pc = __popc(row);
    uint32_t incl = pc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, incl, d);
        if (i >= d) incl += o;
    }
    const uint32_t P = __shfl_sync(FULL, incl, 31);
    const uint32_t base = incl - pc;
    const uint64_t o = offsets[t];
    for (int j = 0; j < HALF; ++j) {
        const bool act = (row >> j) & 1u;
        const uint32_t r = base + __popc(row & ((1u << j) - 1u));
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int64_t rr = r0 + lt_row(perms, t, (a >> 1) * HALF + i), cc = c0 + (a & 1) * HALF + j;
            if (rr >= M || cc >= K) continue;
            int v = 0;
            if (act) {
                const uint64_t e = o + (uint64_t)a * P + r;
                if (bits == 8) {
                    v = (int8_t)values[e];
                } else {
                    const int nib = (values[e >> 1] >> (4 * (e & 1))) & 0xF;
                    v = nib >= 8 ? nib - 16 : nib;
                }
            }
            W[rr * K + cc] = (int8_t)v;
        }
    }
}

}  // namespace

namespace {

// Per-warp ring stage: union mask (128 B), the LT's row permutation (64 B,
// reordered formats), the N rows of X over the LT's 64 columns (64 B each),
// the LT's value span rounded out to 16 B plus 32 B of read-ahead (the
// four-value fetch reads one word past a rank).  PERM: per-warp row
// accumulators [64][NT] that each LT's partial sums are scattered into
// through its permutation.
#ifndef BSP_UNION_STAGES
#define BSP_UNION_STAGES 2
#endif
template <int BITS, int NT, bool PERM>
struct UCfg {
    static constexpr int WARPS = 4, THREADS = 32 * WARPS;
    static constexpr int S = BSP_UNION_STAGES;  // ring stages per warp
    static constexpr int P_OFF = 128;
    static constexpr int X_OFF = 192;
    static constexpr int V_OFF = X_OFF + NT * 64;
    static constexpr int V_BYTES = (BITS == 8 ? 4096 : 2048) + 32;
    static constexpr int STAGE = V_OFF + V_BYTES;            // multiple of 16
    static constexpr int ACC_OFF = WARPS * S * STAGE;
    static constexpr int ACC_BYTES = PERM ? WARPS * 64 * NT * 4 : 0;
    static constexpr int BAR_OFF = ACC_OFF + ACC_BYTES;
    static constexpr int SMEM = BAR_OFF + WARPS * S * 8;
    static_assert(WARPS * 64 * NT * 4 <= ACC_OFF, "reduction buffer aliases the rings");
    static_assert((STAGE % 16) == 0 && (V_OFF % 16) == 0, "bulk-copy alignment");
};

struct UArgs {
    const uint8_t* perms;  // [NLT][64] or null
    const uint32_t* masks32;
    const uint32_t* offsets;
    const uint8_t* values;
    const int8_t* X;
    int N;
    int64_t M, K, KT;
    int splits, per_split;
    int32_t* ws;
    uint32_t* counters;
    int* err;
    int32_t* Y;
    uint32_t spin_cap;
    int stall_first;  // test only: each warp skips the copies of its first LT
};

template <int BITS, int NT, bool PERM>
__global__ void __launch_bounds__(128)
union_spmm_kernel(const UArgs a)
{
    using C = UCfg<BITS, NT, PERM>;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t sel_tbl[16];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);

    if (threadIdx.x < 16) {
        // prmt selector of a 4-position segment pattern n: byte c takes the
        // value at rank popc(n & ((1 << c) - 1)) when bit c is set, else
        // byte 4 (the zero operand)
        const uint32_t n = threadIdx.x;
        uint32_t s = 0, idx = 0;
        for (int c = 0; c < 4; ++c) {
            if ((n >> c) & 1u) s |= (idx++) << (4 * c);
            else s |= 4u << (4 * c);
        }
        sel_tbl[n] = s;
    }
    if (threadIdx.x < C::WARPS * C::S) bspx::mbar_init(bars + threadIdx.x, 1);
    if constexpr (PERM) {
        int32_t* z = reinterpret_cast<int32_t*>(smem + C::ACC_OFF);
        for (int i = threadIdx.x; i < C::WARPS * 64 * NT; i += C::THREADS) z[i] = 0;
    }
    bspx::fence_mbar_init();
    __syncthreads();

    const int N = a.N;
    const int64_t M = a.M, K = a.K, KT = a.KT;
    const int64_t gi = blockIdx.y;
    const int64_t k_begin = (int64_t)blockIdx.x * a.per_split;
    const int64_t k_cnt = min((int64_t)a.per_split, KT - k_begin);
    const int cnt = k_cnt > warp ? (int)((k_cnt - warp + C::WARPS - 1) / C::WARPS) : 0;  // this warp's LTs
    uint8_t* ring = smem + warp * C::S * C::STAGE;
    uint64_t* wbar = bars + warp * C::S;

    auto issue = [&](int u, int s) {  // lane 0: the copies of this warp's LT u into stage s
        const int64_t kt = k_begin + warp + (int64_t)C::WARPS * u;
        const int64_t t = gi * KT + kt;
        const uint32_t o0 = __ldg(a.offsets + t), o1 = __ldg(a.offsets + t + 1);
        const uint64_t b0 = BITS == 8 ? o0 : o0 / 2, b1 = BITS == 8 ? o1 : (o1 + 1) / 2;
        const uint64_t c0 = b0 & ~15ull, c1 = (b1 + 15) & ~15ull;
        const uint32_t vb = (uint32_t)(c1 - c0);
        const int64_t kv = K - kt * LT;
        const uint32_t xb = (uint32_t)(kv >= LT ? LT : kv);  // a multiple of 16 (K is)
        uint8_t* st = ring + s * C::STAGE;
        bspx::mbar_arrive_expect_tx(wbar + s, 128u + (PERM ? 64u : 0u) + (uint32_t)N * xb + vb);
        bspx::bulk_g2s(st, a.masks32 + t * 32, 128, wbar + s);
        if (PERM) bspx::bulk_g2s(st + C::P_OFF, a.perms + t * LT, 64, wbar + s);
        for (int n = 0; n < N; ++n) bspx::bulk_g2s(st + C::X_OFF + n * 64, a.X + n * K + kt * LT, xb, wbar + s);
        if (vb) bspx::bulk_g2s(st + C::V_OFF, a.values + c0, vb, wbar + s);
    };

    int32_t acc[2][NT];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[h][n] = 0;

    bool failed = false;
    // prefetch S - 1 tiles ahead; stalled (test): nothing completes stage 0
    int issued = cnt < C::S - 1 ? cnt : C::S - 1;
    if (lane == 0)
        for (int v = 0; v < issued; ++v)
            if (v > 0 || !a.stall_first) issue(v, v);
    int u = 0;
    for (; u < cnt; ++u) {
        const int s = u % C::S;
        if (u + C::S - 1 < cnt) {  // its stage was released by the __syncwarp that ended LT u - 1
            if (lane == 0) issue(u + C::S - 1, (u + C::S - 1) % C::S);
            issued = u + C::S;
        }
        if (!__all_sync(FULL, bspx::mbar_wait_bounded(wbar + s, (uint32_t)((u / C::S) & 1), a.spin_cap))) {
            failed = true;
            break;
        }
        const uint8_t* st = ring + s * C::STAGE;
        if constexpr (PERM) {  // this LT's partial sums only; scattered below
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int n = 0; n < NT; ++n) acc[h][n] = 0;
        }
        const int64_t t = gi * KT + k_begin + warp + (int64_t)C::WARPS * u;
        const uint32_t o0 = __ldg(a.offsets + t), o1 = __ldg(a.offsets + t + 1);
        const uint32_t P = (o1 - o0) / 4;
        const uint32_t b0 = BITS == 8 ? o0 : o0 / 2;
        const uint32_t shift = b0 & 15u;  // bytes before the LT's first value in the stage
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(st + C::V_OFF);
        const uint32_t* xw = reinterpret_cast<const uint32_t*>(st + C::X_OFF);
        // LSPD: lane = logical row; rank of the row's first active position
        const uint32_t row = reinterpret_cast<const uint32_t*>(st)[lane];
        const uint32_t pc = __popc(row);
        uint32_t incl = pc;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(FULL, incl, d);
            if (lane >= d) incl += o;
        }
        uint32_t r = incl - pc;  // first rank of the current 4-position segment
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t nb = (row >> (4 * q)) & 0xFu;
            const uint32_t sel = sel_tbl[nb];
#pragma unroll
            for (int ar = 0; ar < 4; ++ar) {
                const int ra = ar >> 1, ca = ar & 1;
                const uint32_t e = (uint32_t)ar * P + r;  // value index of the segment's first rank
                uint32_t v4;
                // the funnel shift takes its amount modulo 32: pos << 3 is
                // 8 (pos % 4), np << 2 is 4 (np % 8)
                if constexpr (BITS == 8) {
                    const uint32_t pos = shift + e;
                    v4 = __funnelshift_r(vw[pos >> 2], vw[(pos >> 2) + 1], pos << 3);
                } else {
                    const uint32_t np = 2 * shift + e;  // nibble position
                    const uint32_t v16 = __funnelshift_r(vw[np >> 3], vw[(np >> 3) + 1], np << 2);
                    // four signed nibbles into the high halves of four bytes:
                    // each byte is 16 v, so dp4a accumulates 16 times the
                    // product, divided out (exactly) after the reduction
                    v4 = __byte_perm((v16 << 4) & 0xF0F0u, v16 & 0xF0F0u, 0x5140);
                }
                const int wv = (int)__byte_perm(v4, 0u, sel);
#pragma unroll
                for (int n = 0; n < NT; ++n) acc[ra][n] = __dp4a(wv, (int)xw[n * 16 + ca * 8 + q], acc[ra][n]);
            }
            r += __popc(nb);
        }
        if constexpr (PERM) {
            // place k of the reordered LT is row perm[k]: distinct lanes,
            // distinct rows
            int32_t* accs = reinterpret_cast<int32_t*>(smem + C::ACC_OFF) + warp * 64 * NT;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rowp = st[C::P_OFF + h * 32 + lane];
#pragma unroll
                for (int n = 0; n < NT; ++n) accs[rowp * NT + n] += acc[h][n];
            }
        }
        __syncwarp();
    }
    if (failed) {
        if (lane == 0) {
            atomicExch(a.err, (int)BSP_ERR_TIMEOUT);
            for (int v = u; v < issued; ++v)
                bspx::mbar_wait_bounded(wbar + (v % C::S), (uint32_t)((v / C::S) & 1), a.spin_cap);
        }
        __syncwarp();
    }

    // ---- CTA reduction over the warps (the buffer aliases the rings, or is
    // the row accumulators of a reordered format)
    __syncthreads();
    int32_t* red = reinterpret_cast<int32_t*>(smem + (PERM ? C::ACC_OFF : 0));  // [WARPS][64][NT]
    if constexpr (!PERM) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int n = 0; n < NT; ++n) red[(warp * 64 + h * 32 + lane) * NT + n] = acc[h][n];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * NT; i += C::THREADS) {
        const int rr = i / NT, n = i % NT;
        int32_t sum = 0;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) sum += red[w * 64 * NT + i];
        if constexpr (BITS == 4) sum >>= 4;  // a multiple of 16: exact
        const int64_t m = gi * 64 + rr;
        if (n < N && m < M) {
            if (a.splits == 1) a.Y[(int64_t)n * M + m] = sum;
            else atomicAdd(a.ws + (int64_t)n * M + m, sum);
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
        const int n = i >> 6, rr = i & 63;
        const int64_t m = gi * 64 + rr;
        if (m < M) a.Y[(int64_t)n * M + m] = atomicExch(a.ws + (int64_t)n * M + m, 0);
    }
    if (threadIdx.x == 0) a.counters[gi] = 0u;
}

template <int BITS, int NT, bool PERM>
bsp_status_t launch_union(const bsp_union* h, const int8_t* X, int N, int32_t* Y, cudaStream_t s)
{
    using C = UCfg<BITS, NT, PERM>;
    static bsp_attr_once attr;
    if (h->device < 0 || h->device >= 64) return BSP_ERR_INVALID_ARG;
    if (!attr.run(h->device, [] {
            return cudaFuncSetAttribute(union_spmm_kernel<BITS, NT, PERM>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        }))
        return BSP_ERR_CUDA;
    const int64_t strips = h->Mp / LT, KT = h->Kp / LT;
    // about four CTAs per SM, and at least two LTs per warp
    int64_t splits = (4 * (int64_t)h->num_sms + strips - 1) / strips;
    const int64_t max_splits = (KT + 2 * C::WARPS - 1) / (2 * C::WARPS);
    const int64_t forced = bsp_tune(BSP_TUNE_UNION_SPLITK);
    if (forced >= 1) splits = forced;
    splits = splits < 1 ? 1 : splits;
    if (splits > max_splits && forced < 1) splits = max_splits;
    if (splits > KT) splits = KT;
    if (splits < 1) splits = 1;
    const int per_split = (int)((KT + splits - 1) / splits);
    splits = (KT + per_split - 1) / per_split;
    UArgs a;
    a.perms = h->perms;
    a.masks32 = reinterpret_cast<const uint32_t*>(h->masks);
    a.offsets = h->offsets;
    a.values = h->values;
    a.X = X;
    a.N = N;
    a.M = h->M;
    a.K = h->K;
    a.KT = KT;
    a.splits = (int)splits;
    a.per_split = per_split;
    a.ws = h->ws;
    a.counters = h->counters;
    a.err = h->err;
    a.Y = Y;
    a.spin_cap = bsp_spin_cap();
    a.stall_first = bsp_test_stall();
    union_spmm_kernel<BITS, NT, PERM><<<dim3((unsigned)splits, (unsigned)strips), C::THREADS, C::SMEM, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <int BITS, bool PERM>
bsp_status_t dispatch_union(const bsp_union* h, const int8_t* X, int N, int32_t* Y, cudaStream_t s)
{
    if (N <= 1) return launch_union<BITS, 1, PERM>(h, X, N, Y, s);
    if (N <= 2) return launch_union<BITS, 2, PERM>(h, X, N, Y, s);
    if (N <= 4) return launch_union<BITS, 4, PERM>(h, X, N, Y, s);
    if (N <= 8) return launch_union<BITS, 8, PERM>(h, X, N, Y, s);
    return launch_union<BITS, 16, PERM>(h, X, N, Y, s);
}

void free_union(bsp_union* h)
{
    if (!h) return;
    cudaFree(h->masks);
    cudaFree(h->offsets);
    cudaFree(h->values);
    cudaFree(h->perms);
    cudaFree(h->ws);
    cudaFree(h->counters);
    cudaFree(h->err);
    h->magic = 0;
    delete h;
}

}  // namespace

namespace {

// Per-LT row permutations by the host solver (pairing heuristic for the
// 64-row LTs, R_A = 2), in parallel over LTs.
bsp_status_t solve_perms(bsp_union* h, const int8_t* W, int64_t KT, cudaStream_t s)
{
    uint64_t* act = nullptr;
    if (cudaMalloc(&act, (size_t)h->NLT * LT * 8) != cudaSuccess) return BSP_ERR_OOM;
    ub_rowact_kernel<<<blocks_for(h->NLT * 32, 256), 256, 0, s>>>(W, h->M, h->K, KT, h->NLT, act);
    std::vector<uint64_t> hact((size_t)h->NLT * LT);
    const bool ok = cudaGetLastError() == cudaSuccess &&
                    cudaMemcpyAsync(hact.data(), act, hact.size() * 8, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
                    cudaStreamSynchronize(s) == cudaSuccess;
    cudaFree(act);
    if (!ok) return BSP_ERR_CUDA;
    std::vector<uint8_t> hperm((size_t)h->NLT * LT);
    const int64_t nlt = h->NLT;
    unsigned nt = std::thread::hardware_concurrency();
    nt = nt < 1 ? 1 : (nt > 64 ? 64 : nt);
    if ((int64_t)nt > nlt) nt = (unsigned)nlt;
    std::vector<std::thread> pool;
    for (unsigned w = 0; w < nt; ++w)
        pool.emplace_back([&, w] {
            int32_t perm[LT];
            for (int64_t t = w; t < nlt; t += nt) {
                bsp_reorder_rows_act(hact.data() + t * LT, LT, 2, 0, perm);
                for (int k = 0; k < LT; ++k) hperm[t * LT + k] = (uint8_t)perm[k];
            }
        });
    for (auto& th : pool) th.join();
    if (cudaMalloc(&h->perms, hperm.size()) != cudaSuccess) return BSP_ERR_OOM;
    if (cudaMemcpyAsync(h->perms, hperm.data(), hperm.size(), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BSP_ERR_CUDA;
    return BSP_OK;
}

bsp_status_t union_encode(const int8_t* W, int bits, int64_t M, int64_t K, bool reorder, bsp_stream_t stream,
                          bsp_union_t* out)
{
    if (!out) return BSP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!W || (bits != 4 && bits != 8)) return BSP_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || (K % 16) != 0) return BSP_ERR_SHAPE;
    // W4A4 accumulates 16 times each product: exact while 16 |sum| < 2^31,
    // which |w x| <= 64 and K < 2^21 guarantee
    if (bits == 4 && K >= ((int64_t)1 << 21)) return BSP_ERR_SHAPE;
    if (!aligned16(W)) return BSP_ERR_ALIGN;
    bsp_union* h = new (std::nothrow) bsp_union{};
    if (!h) return BSP_ERR_OOM;
    h->magic = BSP_UNION_MAGIC;
    h->bits = bits;
    h->M = M;
    h->K = K;
    h->Mp = (M + LT - 1) / LT * LT;
    h->Kp = (K + LT - 1) / LT * LT;
    const int64_t KT = h->Kp / LT;
    h->NLT = (h->Mp / LT) * KT;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t* counts = nullptr;
    int* flags = nullptr;  // [0] scan overflow, [1] value out of range
    unsigned long long* nnz = nullptr;
    bsp_status_t st = BSP_OK;
    uint32_t total = 0;
    int hflags[2] = {0, 0};
    unsigned long long hnnz = 0;
    const size_t ws_bytes = (size_t)BSP_DECODE_MAX_N * (size_t)M * 4, cnt_bytes = (size_t)(h->Mp / LT) * 4;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        st = BSP_ERR_CUDA;
        goto done;
    }
    if (cudaMalloc(&h->masks, (size_t)h->NLT * 128) != cudaSuccess ||
        cudaMalloc(&h->offsets, (size_t)(h->NLT + 1) * 4) != cudaSuccess ||
        cudaMalloc(&counts, (size_t)h->NLT * 4) != cudaSuccess || cudaMalloc(&flags, 2 * sizeof(int)) != cudaSuccess ||
        cudaMalloc(&nnz, sizeof(unsigned long long)) != cudaSuccess || cudaMalloc(&h->ws, ws_bytes) != cudaSuccess ||
        cudaMalloc(&h->counters, cnt_bytes) != cudaSuccess || cudaMalloc(&h->err, sizeof(int)) != cudaSuccess) {
        st = BSP_ERR_OOM;
        goto done;
    }
    if (cudaMemsetAsync(flags, 0, 2 * sizeof(int), s) != cudaSuccess ||
        cudaMemsetAsync(nnz, 0, sizeof(unsigned long long), s) != cudaSuccess ||
        cudaMemsetAsync(h->ws, 0, ws_bytes, s) != cudaSuccess || cudaMemsetAsync(h->counters, 0, cnt_bytes, s) != cudaSuccess ||
        cudaMemsetAsync(h->err, 0, sizeof(int), s) != cudaSuccess) {
        st = BSP_ERR_CUDA;
        goto done;
    }
    if (reorder && (st = solve_perms(h, W, KT, s)) != BSP_OK) goto done;
    ub_mask_kernel<<<blocks_for(h->NLT * 32, 256), 256, 0, s>>>(W, M, K, KT, h->NLT, bits, h->perms,
                                                                reinterpret_cast<uint32_t*>(h->masks), counts, nnz,
                                                                flags + 1);
    if (cudaGetLastError() != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }
    st = bsp_exclusive_scan_u32(counts, h->NLT, h->offsets, flags, s);
    if (st != BSP_OK) goto done;
    if (cudaMemcpyAsync(&total, h->offsets + h->NLT, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(hflags, flags, sizeof(hflags), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&hnnz, nnz, sizeof(hnnz), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        st = BSP_ERR_CUDA;
        goto done;
    }
    if (hflags[0]) { st = BSP_ERR_SHAPE; goto done; }
    if (hflags[1]) { st = BSP_ERR_INVALID_ARG; goto done; }
    h->nnz = hnnz;
    h->total = total;
    h->value_bytes = ((uint64_t)total * (uint64_t)bits + 7) / 8;
    // 32 zeroed bytes of slack: the product's copies and four-value fetches
    // read up to 16 B past the last span
    if (cudaMalloc(&h->values, h->value_bytes + 32) != cudaSuccess) { st = BSP_ERR_OOM; goto done; }
    if (cudaMemsetAsync(h->values, 0, h->value_bytes + 32, s) != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }
    ub_pack_kernel<<<blocks_for(h->NLT * 32, 256), 256, 0, s>>>(W, M, K, KT, h->NLT, bits, h->perms,
                                                                reinterpret_cast<const uint32_t*>(h->masks),
                                                                h->offsets, h->values);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) st = BSP_ERR_CUDA;
done:
    cudaFree(counts);
    cudaFree(flags);
    cudaFree(nnz);
    if (st != BSP_OK) {
        free_union(h);
        return st;
    }
    *out = h;
    return BSP_OK;
}

}  // namespace

extern "C" {

bsp_status_t bsp_union_encode(const int8_t* W, int bits, int64_t M, int64_t K, bsp_stream_t stream,
                              bsp_union_t* out)
{
    return union_encode(W, bits, M, K, false, stream, out);
}

bsp_status_t bsp_union_encode_reordered(const int8_t* W, int bits, int64_t M, int64_t K, bsp_stream_t stream,
                                        bsp_union_t* out)
{
    return union_encode(W, bits, M, K, true, stream, out);
}

bsp_status_t bsp_union_export_perms(bsp_union_t h, uint8_t* perms, bsp_stream_t stream)
{
    if (!valid(h) || !perms) return BSP_ERR_INVALID_ARG;
    if (!h->perms) return BSP_ERR_INVALID_ARG;  // not a reordered encoding
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    return cudaMemcpyAsync(perms, h->perms, (size_t)h->NLT * LT, cudaMemcpyDefault, (cudaStream_t)stream) ==
                   cudaSuccess
               ? BSP_OK
               : BSP_ERR_CUDA;
}

bsp_status_t bsp_union_destroy(bsp_union_t h)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    free_union(h);
    return BSP_OK;
}

bsp_status_t bsp_union_spmm(bsp_union_t h, const int8_t* X, int64_t N, int32_t* Y, bsp_stream_t stream)
{
    if (!valid(h) || !X || !Y || N < 1 || N > (int64_t)1 << 30) return BSP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y)) return BSP_ERR_ALIGN;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    for (int64_t n0 = 0; n0 < N; n0 += BSP_DECODE_MAX_N) {  // blocks of 16 columns of Y
        const int nb = (int)((N - n0) < BSP_DECODE_MAX_N ? (N - n0) : BSP_DECODE_MAX_N);
        const int8_t* Xb = X + n0 * h->K;
        int32_t* Yb = Y + n0 * h->M;
        const bsp_status_t st = h->perms ? (h->bits == 8 ? dispatch_union<8, true>(h, Xb, nb, Yb, s)
                                                         : dispatch_union<4, true>(h, Xb, nb, Yb, s))
                                         : (h->bits == 8 ? dispatch_union<8, false>(h, Xb, nb, Yb, s)
                                                         : dispatch_union<4, false>(h, Xb, nb, Yb, s));
        if (st != BSP_OK) return st;
    }
    return BSP_OK;
}

bsp_status_t bsp_union_storage_bytes(bsp_union_t h, uint64_t* bytes)
{
    if (!valid(h) || !bytes) return BSP_ERR_INVALID_ARG;
    *bytes = 4ull * (uint64_t)(h->NLT + 1) + 128ull * (uint64_t)h->NLT + h->value_bytes;
    return BSP_OK;
}

bsp_status_t bsp_union_info(bsp_union_t h, bsp_union_info_t* o)
{
    if (!valid(h) || !o) return BSP_ERR_INVALID_ARG;
    o->M = h->M;
    o->K = h->K;
    o->bits = h->bits;
    o->lt = LT;
    o->areas_r = 2;
    o->areas_c = 2;
    o->device = h->device;
    o->NLT = h->NLT;
    o->nnz = h->nnz;
    o->total_values = h->total;
    o->value_bytes = h->value_bytes;
    o->masks = h->masks;
    o->offsets = h->offsets;
    o->values = h->values;
    o->reordered = h->perms != nullptr;
    return BSP_OK;
}

bsp_status_t bsp_union_export(bsp_union_t h, uint64_t* masks, uint32_t* offsets, uint8_t* values,
                              bsp_stream_t stream)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (masks && cudaMemcpyAsync(masks, h->masks, (size_t)h->NLT * 128, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (offsets && cudaMemcpyAsync(offsets, h->offsets, (size_t)(h->NLT + 1) * 4, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (values && h->value_bytes &&
        cudaMemcpyAsync(values, h->values, (size_t)h->value_bytes, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    return BSP_OK;
}

bsp_status_t bsp_union_decode(bsp_union_t h, int8_t* W_out, bsp_stream_t stream)
{
    if (!valid(h) || !W_out) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    ub_decode_kernel<<<blocks_for(h->NLT * 32, 256), 256, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const uint32_t*>(h->masks), h->offsets, h->values, h->perms, h->bits, h->M, h->K, h->Kp / LT,
        h->NLT, W_out);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

bsp_status_t bsp_union_check(bsp_union_t h, bsp_stream_t stream)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int e = 0;
    if (cudaMemcpyAsync(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (e != 0) {
        cudaMemsetAsync(h->err, 0, sizeof(int), s);
        cudaStreamSynchronize(s);
        return (bsp_status_t)e;
    }
    return BSP_OK;
}

}  // extern "C"
