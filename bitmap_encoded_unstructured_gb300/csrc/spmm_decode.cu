// Decode-path product Y = W * X for N <= 16 on CUDA cores, and the
// zero-skipping sparse-vector product.
//
// Method (SpInfer's shared-memory bitmap decoding, "SpInfer: How bitmaps
// make sparse LLMs actually fast", sections "Shared Memory Bitmap Decoding
// (SMBD)" and "The async pipeline"; split-K over GroupTiles with a
// reduction workspace as in "Unified Static-Dynamic Pruning for Efficient
// LLM Inference", section 4.2.3 and its Algorithm 1 epilogue):
//
//  * grid = (splits, M/64): a CTA owns one 64-row strip of W (one GT row)
//    and a contiguous range of GT columns; its warps take the GTs of that
//    range round-robin, one GT at a time.
//  * per GT a warp stages, in its own shared-memory slice:
//      - the 64 BT bitmaps (lane l loads BTs 2l, 2l+1 with one 16-B load),
//      - the per-BT value bases: popcounts + a warp exclusive scan (shfl),
//      - the GT's packed value span (16-B vector loads of the aligned
//        superset [floor16(off_t), ceil16(off_t+1))),
//      - the X tile of the GT's 64 columns, widened to fp32 / int32.
//  * decode + multiply: lane l owns GT rows l and l+32.  For each of the 8
//    BTs on a row it forms the row's byte of the bitmap, finds the first
//    value by a masked popcount (nonzeros of earlier rows of the BT), then
//    walks the set bits: acc[n] += w * x[col][n] (fp32 FMA / int32 MAD).
//  * the warps' partial sums are added in shared memory; with one split the
//    CTA writes Y, otherwise it adds into the handle's workspace and the
//    last CTA of the strip (arrival counter) converts, writes Y and clears
//    the workspace and counter for the next call.
//
// spMspV ("Unified Static-Dynamic Pruning ...", sections 4.2 and 4.2.1:
// activation-inactive columns are neither fetched nor decoded): with N = 1
// a K-octet (one BT column, 8 activations) whose activations are all zero
// marks its BTs inactive; the 16-B chunks of the value span that hold only
// inactive BTs are not loaded and inactive BTs are not decoded.  In the
// TCA-BME order the two BTs of one TCTile row-half that share a column
// octet are adjacent, so lane l's BT pair (2l, 2l+1) is exactly the
// segment (TCTile row l/8, octet l%8) and the skip is a per-lane flag.
#include "bsp_internal.cuh"

#include <cstdlib>
#include <type_traits>

namespace {

__device__ __forceinline__ int bt_local(int br, int bc)
{
    return (((br >> 1) * 4 + (bc >> 1)) << 2) + (br & 1) + ((bc & 1) << 1);
}

template <int NT, bool I8>
struct DecCfg {
    static constexpr int WARPS = (NT >= 16) ? 7 : 8;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int EB = I8 ? 1 : 2;
    static constexpr int E16 = 16 / EB;                // elements per 16-B chunk
    static constexpr int VAL_CHUNKS = 4096 / E16 + 1;  // dense GT + misalignment
    static constexpr int XS = (NT >= 8) ? NT + 4 : NT; // X-tile row stride (elements)
    static constexpr int VW = NT < 4 ? NT : 4;         // vector width of X-tile rows
    static constexpr int NEED_WORDS = (VAL_CHUNKS + 31) / 32;
    static constexpr int BM_OFF = 0;
    static constexpr int BASE_OFF = BM_OFF + 64 * 8;
    static constexpr int X_OFF = BASE_OFF + 64 * 4;
    static constexpr int VAL_OFF = X_OFF + ((64 * XS * 4 + 15) & ~15);
    static constexpr int NEED_OFF = VAL_OFF + VAL_CHUNKS * 16;
    static constexpr int WARP_BYTES = (NEED_OFF + NEED_WORDS * 4 + 15) & ~15;
    static constexpr int SMEM = WARPS * WARP_BYTES;
    static_assert(64 * NT * 4 <= VAL_OFF - X_OFF, "reduction buffer must fit the X tile");
};

template <typename Acc, int VW>
struct Vec;
template <> struct Vec<float, 1> { using T = float; };
template <> struct Vec<float, 2> { using T = float2; };
template <> struct Vec<float, 4> { using T = float4; };
template <> struct Vec<int, 1> { using T = int; };
template <> struct Vec<int, 2> { using T = int2; };
template <> struct Vec<int, 4> { using T = int4; };

template <bool I8>
__device__ __forceinline__ void load_x_pair(const uint8_t* X, int64_t idx, float& a, float& b)
{
    const __half2 v = __ldg(reinterpret_cast<const __half2*>(X) + (idx >> 1));
    a = __low2float(v);
    b = __high2float(v);
}

template <bool I8>
__device__ __forceinline__ void load_x_pair(const uint8_t* X, int64_t idx, int& a, int& b)
{
    const uint16_t v = __ldg(reinterpret_cast<const uint16_t*>(X) + (idx >> 1));
    a = (int)(int8_t)(v & 0xFF);
    b = (int)(int8_t)(v >> 8);
}

__device__ __forceinline__ float load_val(const uint8_t* vals, uint32_t i, float)
{
    return __half2float(reinterpret_cast<const __half*>(vals)[i]);
}

__device__ __forceinline__ int load_val(const uint8_t* vals, uint32_t i, int)
{
    return (int)reinterpret_cast<const int8_t*>(vals)[i];
}

__device__ __forceinline__ void mac(float& acc, float w, float x) { acc = fmaf(w, x, acc); }
__device__ __forceinline__ void mac(int& acc, int w, int x) { acc += w * x; }

__device__ __forceinline__ void write_out(void* Y, int mode, int64_t idx, float v, float)
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

template <typename V, typename A, int W>
__device__ __forceinline__ V pack_vec(const A* a)
{
    if constexpr (W == 1) return a[0];
    else if constexpr (W == 2) return V{a[0], a[1]};
    else return V{a[0], a[1], a[2], a[3]};
}

template <typename A, typename V>
__device__ __forceinline__ A vec_get(const V& v, int e)
{
    if constexpr (std::is_same_v<V, A>) return v;
    else if constexpr (sizeof(V) == 2 * sizeof(A)) return e == 0 ? v.x : v.y;
    else return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

__device__ __forceinline__ float ws_take(float* p) { return atomicExch(p, 0.0f); }
__device__ __forceinline__ int ws_take(int* p) { return atomicExch(p, 0); }

template <int NT, bool I8, bool SKIP>
__global__ void __launch_bounds__(DecCfg<NT, I8>::THREADS, 2)
spmm_decode_kernel(const uint64_t* __restrict__ bitmaps, const uint32_t* __restrict__ offsets,
                   const uint8_t* __restrict__ values, const uint8_t* __restrict__ X, int N,
                   int64_t M, int64_t K, int splits, int per_split,
                   void* __restrict__ ws_v, uint32_t* __restrict__ counters,
                   void* __restrict__ Y, int mode, const float* __restrict__ row_scale)
{
    using C = DecCfg<NT, I8>;
    using Acc = std::conditional_t<I8, int, float>;
    using XV = typename Vec<Acc, C::VW>::T;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_last;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t* wb = smem + warp * C::WARP_BYTES;
    uint64_t* bm_s = reinterpret_cast<uint64_t*>(wb + C::BM_OFF);
    uint32_t* base_s = reinterpret_cast<uint32_t*>(wb + C::BASE_OFF);
    Acc* x_s = reinterpret_cast<Acc*>(wb + C::X_OFF);
    uint4* val_s = reinterpret_cast<uint4*>(wb + C::VAL_OFF);
    const uint8_t* val_b = wb + C::VAL_OFF;
    uint32_t* need_s = reinterpret_cast<uint32_t*>(wb + C::NEED_OFF);

    const int64_t KT = K >> 6;
    const int64_t gi = blockIdx.y;
    const int64_t k_begin = (int64_t)blockIdx.x * per_split;
    const int64_t k_end = min(KT, k_begin + per_split);
    const uint4* values16 = reinterpret_cast<const uint4*>(values);

    Acc acc[2][NT];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[h][n] = Acc(0);

    for (int64_t gj = k_begin + warp; gj < k_end; gj += C::WARPS) {
        const int64_t t = gi * KT + gj;
        const ulonglong2 bb = __ldg(reinterpret_cast<const ulonglong2*>(bitmaps + t * 64) + lane);
        const uint32_t off0 = __ldg(offsets + t);
        const uint32_t off1 = __ldg(offsets + t + 1);

        // X tile: lane owns columns 2*lane, 2*lane+1 of this GT
        Acc xa[NT], xb[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if (n < N) {
                load_x_pair<I8>(X, (int64_t)n * K + gj * 64 + 2 * lane, xa[n], xb[n]);
            } else {
                xa[n] = Acc(0);
                xb[n] = Acc(0);
            }
        }

        // BT value bases: popcounts and a warp exclusive scan
        const uint32_t c0 = __popcll(bb.x), c1 = __popcll(bb.y);
        uint32_t incl = c0 + c1;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += o;
        }
        const uint32_t ex = incl - (c0 + c1);
        bm_s[2 * lane] = bb.x;
        bm_s[2 * lane + 1] = bb.y;
        base_s[2 * lane] = ex;
        base_s[2 * lane + 1] = ex + c0;

#pragma unroll
        for (int j = 0; j < NT; j += C::VW) {
            *reinterpret_cast<XV*>(x_s + (2 * lane) * C::XS + j) = pack_vec<XV, Acc, C::VW>(xa + j);
            *reinterpret_cast<XV*>(x_s + (2 * lane + 1) * C::XS + j) = pack_vec<XV, Acc, C::VW>(xb + j);
        }

        // value span, as 16-B chunks
        const uint32_t ch0 = off0 / C::E16;
        const uint32_t nch = (off1 + C::E16 - 1) / C::E16 - ch0;
        const uint32_t shift = off0 - ch0 * C::E16;

        uint32_t act8 = 0xFFu;
        if constexpr (SKIP) {
            // octet j <-> lanes 4j..4j+3 (two columns each)
            const bool nz = (xa[0] != Acc(0)) || (xb[0] != Acc(0));
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, nz);
            act8 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) act8 |= (((bal >> (4 * j)) & 0xFu) ? 1u : 0u) << j;
            if (lane < C::NEED_WORDS) need_s[lane] = 0;
            __syncwarp();
            const uint32_t seg = c0 + c1;
            if (((act8 >> (lane & 7)) & 1u) && seg) {
                const uint32_t q0 = (ex + shift) / C::E16;
                const uint32_t q1 = (ex + seg + shift + C::E16 - 1) / C::E16;
                for (uint32_t q = q0; q < q1; ++q) atomicOr(need_s + (q >> 5), 1u << (q & 31));
            }
            __syncwarp();
            for (uint32_t q = lane; q < nch; q += 32)
                if ((need_s[q >> 5] >> (q & 31)) & 1u) val_s[q] = __ldg(values16 + ch0 + q);
        } else {
            for (uint32_t q = lane; q < nch; q += 32) val_s[q] = __ldg(values16 + ch0 + q);
        }
        __syncwarp();

#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = lane + 32 * h;
            const int br = r >> 3, rr = r & 7;
#pragma unroll
            for (int bc = 0; bc < 8; ++bc) {
                if (SKIP && !((act8 >> bc) & 1u)) continue;
                const int gl = bt_local(br, bc);
                const uint64_t bm = bm_s[gl];
                uint32_t byte = (uint32_t)(bm >> (8 * rr)) & 0xFFu;
                uint32_t idx = base_s[gl] + (uint32_t)__popcll(bm & ((1ull << (8 * rr)) - 1ull)) + shift;
                while (byte) {
                    const int c = __ffs(byte) - 1;
                    byte &= byte - 1;
                    const Acc w = load_val(val_b, idx++, Acc(0));
                    const Acc* xr = x_s + (bc * 8 + c) * C::XS;
#pragma unroll
                    for (int j = 0; j < NT; j += C::VW) {
                        const XV xv = *reinterpret_cast<const XV*>(xr + j);
#pragma unroll
                        for (int e = 0; e < C::VW; ++e) mac(acc[h][j + e], w, vec_get<Acc>(xv, e));
                    }
                }
            }
        }
        __syncwarp();
    }

    // ---- CTA reduction over warps, then output or split-K accumulation
    __syncthreads();
    Acc* red = x_s;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < NT; ++n) red[(lane + 32 * h) * NT + n] = acc[h][n];
    __syncthreads();

    Acc* ws = reinterpret_cast<Acc*>(ws_v);
    for (int i = threadIdx.x; i < 64 * NT; i += C::THREADS) {
        const int r = i / NT, n = i % NT;
        Acc sum = Acc(0);
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w)
            sum += reinterpret_cast<const Acc*>(smem + w * C::WARP_BYTES + C::X_OFF)[i];
        if (n < N) {
            const int64_t m = gi * 64 + r;
            if (splits == 1)
                write_out(Y, mode, (int64_t)n * M + m, sum, row_scale ? row_scale[m] : 1.0f);
            else
                atomicAdd(ws + (int64_t)n * M + m, sum);
        }
    }
    if (splits == 1) return;

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(counters + gi, 1u) == (uint32_t)(splits - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = threadIdx.x; i < 64 * N; i += C::THREADS) {
        const int n = i >> 6, r = i & 63;
        const int64_t m = gi * 64 + r;
        const Acc v = ws_take(ws + (int64_t)n * M + m);
        write_out(Y, mode, (int64_t)n * M + m, v, row_scale ? row_scale[m] : 1.0f);
    }
    if (threadIdx.x == 0) counters[gi] = 0u;
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
    dim3 grid((unsigned)splits, (unsigned)(h->M / 64));
    spmm_decode_kernel<NT, I8, SKIP><<<grid, C::THREADS, C::SMEM, s>>>(
        h->bitmaps, h->offsets, (const uint8_t*)h->values, (const uint8_t*)X, N, h->M, h->K,
        splits, per_split, h->ws, h->counters, Y, mode, row_scale);
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
    int64_t splits;
    if (const char* e = std::getenv("BSP_SPLITK")) {
        splits = std::atol(e);
    } else {
        const int64_t want_ctas = 4 * (int64_t)h->num_sms;
        splits = (want_ctas + strips - 1) / strips;
    }
    const int64_t max_splits = KT / 8 > 1 ? KT / 8 : 1;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
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
