// Encoder and decoder of the TCA-BME tile format, on the device.
//
// Format: "SpInfer: How bitmaps make sparse LLMs actually fast", sections
// "How TCA-BME addresses the indexing overhead" (8x8 BitmapTile with one
// uint64, 16x16 TCTile, GroupTile, Stor closed form) and "The Values array
// and why it's confusing at first" (values packed in tile order, a value's
// slot = nonzeros before it).  Tiling readings: GT 64x64 row-major over the
// grid, TCTiles row-major in a GT, BTs of a TCTile in mma A-register order
// (TL, BL, TR, BR), bit p = 8*row + col.
//
// Work unit of every kernel here is one BT row-byte: 8 consecutive elements
// of one row inside one BT (16 B of fp16 or 8 B of int8), so loads along a
// row of W are contiguous across a warp.
#include "bsp_internal.cuh"

namespace {

// BT index inside its GT for BT-row br (0..7) and BT-column bc (0..7).
__device__ __forceinline__ int bt_local(int br, int bc)
{
    return (((br >> 1) * 4 + (bc >> 1)) << 2) + (br & 1) + ((bc & 1) << 1);
}

// Logical shape of W inside its zero-padded grid: M rows, K8 row-bytes per
// row (K / 8), padded width Kp (a multiple of 64).  Row-bytes outside
// [0, M) x [0, K8) are padding: no nonzeros, nothing read or written.
struct EncShape {
    int64_t M, K8, Kp;
};

// Row-byte i of the padded grid -> its index in the logical W, or false.
__device__ __forceinline__ bool logical_rowbyte(int64_t i, const EncShape& sh, int64_t* li)
{
    const int64_t Kp8 = sh.Kp >> 3;
    const int64_t r = i / Kp8, c8 = i - r * Kp8;
    if (r >= sh.M || c8 >= sh.K8) return false;
    *li = r * sh.K8 + c8;
    return true;
}

struct RowByte {
    int64_t g;   // global BT index
    int64_t t;   // GT index
    int rr;      // row inside the BT
};

__device__ __forceinline__ RowByte row_byte(int64_t i, int64_t K)
{
    const int64_t K8 = K >> 3;
    const int64_t r = i / K8;
    const int64_t c8 = i - r * K8;  // BT column block index along the row
    const int64_t t = (r >> 6) * (K >> 6) + (c8 >> 3);
    RowByte rb;
    rb.t = t;
    rb.g = t * 64 + bt_local((int)((r & 63) >> 3), (int)(c8 & 7));
    rb.rr = (int)(r & 7);
    return rb;
}

template <int EB>
struct Row8;  // 8 raw elements of one row-byte

template <>
struct Row8<2> {
    uint4 v;
    __device__ __forceinline__ uint32_t elem(int j) const
    {
        const uint32_t w = (&v.x)[j >> 1];
        return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
    }
    __device__ __forceinline__ void set(int j, uint32_t e)
    {
        uint32_t& w = (&v.x)[j >> 1];
        w = (j & 1) ? ((w & 0xFFFFu) | (e << 16)) : ((w & 0xFFFF0000u) | e);
    }
};

template <>
struct Row8<1> {
    uint2 v;
    __device__ __forceinline__ uint32_t elem(int j) const
    {
        const uint32_t w = (&v.x)[j >> 2];
        return (w >> (8 * (j & 3))) & 0xFFu;
    }
    __device__ __forceinline__ void set(int j, uint32_t e)
    {
        uint32_t& w = (&v.x)[j >> 2];
        const int sh = 8 * (j & 3);
        w = (w & ~(0xFFu << sh)) | (e << sh);
    }
};

template <int EB>
__device__ __forceinline__ Row8<EB> load_row8(const void* W, int64_t i)
{
    Row8<EB> r;
    if constexpr (EB == 2)
        r.v = __ldg(reinterpret_cast<const uint4*>(W) + i);
    else
        r.v = __ldg(reinterpret_cast<const uint2*>(W) + i);
    return r;
}

// Pass 1: one byte of a bitmap per thread (the row-byte's occupancy).
template <int EB>
__global__ void enc_bitmap_kernel(const void* __restrict__ W, int64_t n_rowbytes, EncShape sh,
                                  uint8_t* __restrict__ bitmap_bytes)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_rowbytes) return;
    int64_t li;
    uint32_t byte = 0;
    if (logical_rowbyte(i, sh, &li)) {
        const Row8<EB> e = load_row8<EB>(W, li);
#pragma unroll
        for (int j = 0; j < 8; ++j) byte |= (e.elem(j) != 0u ? 1u : 0u) << j;
    }
    const RowByte rb = row_byte(i, sh.Kp);
    // little-endian: byte rr of the uint64 holds bits 8*rr .. 8*rr+7
    bitmap_bytes[rb.g * 8 + rb.rr] = (uint8_t)byte;
}

// Pass 2: per GT (one warp): BT popcounts, exclusive prefix inside the GT,
// GT nonzero total.
__global__ void enc_count_kernel(const uint64_t* __restrict__ bitmaps, int64_t NGT,
                                 uint32_t* __restrict__ bt_prefix,
                                 uint32_t* __restrict__ gt_nnz, unsigned int* max_nnz)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= NGT) return;
    const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2*>(bitmaps + t * 64) + lane);
    const uint32_t c0 = __popcll(b.x), c1 = __popcll(b.y);
    uint32_t incl = c0 + c1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    const uint32_t ex = incl - (c0 + c1);
    bt_prefix[t * 64 + 2 * lane] = ex;
    bt_prefix[t * 64 + 2 * lane + 1] = ex + c0;
    if (lane == 31) {
        gt_nnz[t] = incl;
        atomicMax(max_nnz, incl);
    }
}

// Pass 3: exclusive scan of the per-GT counts into offsets[NGT+1], one
// block.  Sets *overflow when the total does not fit uint32.
__global__ void enc_scan_kernel(const uint32_t* __restrict__ gt_nnz, int64_t NGT,
                                uint32_t* __restrict__ offsets, int* overflow)
{
    __shared__ unsigned long long warp_sums[32];
    __shared__ unsigned long long carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int64_t base = 0; base < NGT; base += blockDim.x) {
        const int64_t i = base + tid;
        const unsigned long long v = (i < NGT) ? gt_nnz[i] : 0ull;
        unsigned long long incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int nw = blockDim.x >> 5;
            unsigned long long ws = (lane < nw) ? warp_sums[lane] : 0ull;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, ws, d);
                if (lane >= d) ws += o;
            }
            if (lane < nw) warp_sums[lane] = ws;  // inclusive over warps
        }
        __syncthreads();
        const unsigned long long carry = carry_s;
        const unsigned long long before = (warp ? warp_sums[warp - 1] : 0ull) + incl - v;
        const unsigned long long ex = carry + before;
        if (i < NGT) {
            if (ex > 0xFFFFFFFFull) *overflow = 1;
            offsets[i] = (uint32_t)ex;
        }
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sums[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0) {
        if (carry_s > 0xFFFFFFFFull) *overflow = 1;
        offsets[NGT] = (uint32_t)carry_s;
    }
}

__device__ __forceinline__ uint64_t rowbyte_slot(const uint64_t* bitmaps, const uint32_t* offsets,
                                                 const uint32_t* bt_prefix, const RowByte& rb,
                                                 uint32_t* byte_out)
{
    const uint64_t bm = __ldg(bitmaps + rb.g);
    const int sh = 8 * rb.rr;
    *byte_out = (uint32_t)(bm >> sh) & 0xFFu;
    const uint64_t below = bm & ((1ull << sh) - 1ull);
    return (uint64_t)__ldg(offsets + rb.t) + __ldg(bt_prefix + rb.g) + (uint64_t)__popcll(below);
}

// Pass 4: write each row-byte's nonzeros to their packed slots.
template <int EB>
__global__ void enc_pack_kernel(const void* __restrict__ W, int64_t n_rowbytes, EncShape sh,
                                const uint64_t* __restrict__ bitmaps,
                                const uint32_t* __restrict__ offsets,
                                const uint32_t* __restrict__ bt_prefix,
                                uint8_t* __restrict__ values)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_rowbytes) return;
    int64_t li;
    if (!logical_rowbyte(i, sh, &li)) return;  // padding: no nonzeros
    const RowByte rb = row_byte(i, sh.Kp);
    uint32_t byte;
    uint64_t slot = rowbyte_slot(bitmaps, offsets, bt_prefix, rb, &byte);
    const Row8<EB> e = load_row8<EB>(W, li);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if ((byte >> j) & 1u) {
            const uint32_t v = e.elem(j);
            if constexpr (EB == 2)
                reinterpret_cast<uint16_t*>(values)[slot] = (uint16_t)v;
            else
                values[slot] = (uint8_t)v;
            ++slot;
        }
    }
}

// Decoder: dense row-byte from its bitmap byte and packed values.
// The per-BT prefix is recomputed from the bitmaps of the GT (no side array).
template <int EB>
__global__ void dec_kernel(const uint64_t* __restrict__ bitmaps,
                           const uint32_t* __restrict__ offsets,
                           const uint8_t* __restrict__ values, int64_t n_rowbytes,
                           EncShape shape, void* __restrict__ W_out)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_rowbytes) return;
    int64_t li;
    if (!logical_rowbyte(i, shape, &li)) return;  // padding is not part of W
    const RowByte rb = row_byte(i, shape.Kp);
    const int64_t g0 = rb.t * 64;
    uint64_t pre = 0;
    for (int64_t g = g0; g < rb.g; ++g) pre += (uint64_t)__popcll(__ldg(bitmaps + g));
    const uint64_t bm = __ldg(bitmaps + rb.g);
    const int sh = 8 * rb.rr;
    const uint32_t byte = (uint32_t)(bm >> sh) & 0xFFu;
    uint64_t slot = (uint64_t)__ldg(offsets + rb.t) + pre + (uint64_t)__popcll(bm & ((1ull << sh) - 1ull));
    Row8<EB> out;
    out.v = {};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if ((byte >> j) & 1u) {
            uint32_t v;
            if constexpr (EB == 2)
                v = __ldg(reinterpret_cast<const uint16_t*>(values) + slot);
            else
                v = __ldg(values + slot);
            out.set(j, v);
            ++slot;
        }
    }
    if constexpr (EB == 2)
        reinterpret_cast<uint4*>(W_out)[li] = out.v;
    else
        reinterpret_cast<uint2*>(W_out)[li] = out.v;
}

inline unsigned grid_for(int64_t n, int block) { return (unsigned)((n + block - 1) / block); }

// Validation of imported arrays: offsets[0] == 0, for every GT
// offsets[t+1] - offsets[t] == sum of the popcounts of its 64 bitmaps, and
// no bit set in the zero padding of the edge GTs (rows >= M, columns >= K).
// One warp per GT; any violation sets bad[0]; bad[1] gets the largest GT
// nonzero count.
__global__ void validate_kernel(const uint64_t* __restrict__ bitmaps, const uint32_t* __restrict__ offsets,
                                int64_t NGT, int64_t M, int64_t K, int64_t KTp, int* bad)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= NGT) return;
    const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2*>(bitmaps + t * 64) + lane);
    // rows / columns of this GT inside W
    const int64_t vr = M - (t / KTp) * 64, vc = K - (t % KTp) * 64;
    bool pad_ok = true;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int gl = 2 * lane + k;                    // BT inside the GT
        const int tl = gl >> 2, bq = gl & 3;            // TCTile, BT inside it (TL, BL, TR, BR)
        const int br = 2 * (tl >> 2) + (bq & 1), bc = 2 * (tl & 3) + (bq >> 1);
        const int64_t rv = vr - 8 * br, cv = vc - 8 * bc;  // valid rows / columns of the BT (K % 8 == 0)
        uint64_t valid = 0;
        if (cv > 0 && rv > 0) valid = rv >= 8 ? ~0ull : ((1ull << (8 * rv)) - 1ull);
        pad_ok = pad_ok && (((k ? b.y : b.x) & ~valid) == 0ull);
    }
    uint32_t c = __popcll(b.x) + __popcll(b.y);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, d);
    if (!__all_sync(0xFFFFFFFFu, pad_ok) && lane == 0) atomicExch(bad, 1);
    if (lane == 0) {
        const uint32_t o0 = __ldg(offsets + t), o1 = __ldg(offsets + t + 1);
        if (o1 < o0 || o1 - o0 != c || (t == 0 && o0 != 0)) atomicExch(bad, 1);
        atomicMax(bad + 1, (int)c);
    }
}

}  // namespace

bsp_status_t bsp_run_encode(bsp_handle* h, const void* W, cudaStream_t s)
{
    const int eb = bsp_elem_bytes(h->dtype);
    const int64_t n_rowbytes = h->Mp * h->Kp / 8;  // the padded grid
    const EncShape sh{h->M, h->K / 8, h->Kp};
    uint32_t* bt_prefix = nullptr;
    uint32_t* gt_nnz = nullptr;
    int* overflow = nullptr;
    bsp_status_t st = BSP_OK;
    uint32_t total = 0;
    int ovf = 0, maxc = 0;

    if (cudaMalloc(&h->bitmaps, (size_t)h->NBT * 8) != cudaSuccess ||
        cudaMalloc(&h->offsets, (size_t)(h->NGT + 1) * 4) != cudaSuccess ||
        cudaMalloc(&bt_prefix, (size_t)h->NBT * 4) != cudaSuccess ||
        cudaMalloc(&gt_nnz, (size_t)h->NGT * 4) != cudaSuccess ||
        cudaMalloc(&overflow, 2 * sizeof(int)) != cudaSuccess) {  // overflow flag, largest GT count
        st = BSP_ERR_OOM;
        goto done;
    }
    if (cudaMemsetAsync(overflow, 0, 2 * sizeof(int), s) != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }

    if (eb == 2)
        enc_bitmap_kernel<2><<<grid_for(n_rowbytes, 256), 256, 0, s>>>(W, n_rowbytes, sh, (uint8_t*)h->bitmaps);
    else
        enc_bitmap_kernel<1><<<grid_for(n_rowbytes, 256), 256, 0, s>>>(W, n_rowbytes, sh, (uint8_t*)h->bitmaps);
    enc_count_kernel<<<grid_for(h->NGT * 32, 256), 256, 0, s>>>(h->bitmaps, h->NGT, bt_prefix, gt_nnz,
                                                                reinterpret_cast<unsigned int*>(overflow + 1));
    enc_scan_kernel<<<1, 1024, 0, s>>>(gt_nnz, h->NGT, h->offsets, overflow);
    if (cudaGetLastError() != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }
    if (cudaMemcpyAsync(&total, h->offsets + h->NGT, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&ovf, overflow, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&maxc, overflow + 1, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        st = BSP_ERR_CUDA;
        goto done;
    }
    if (ovf) { st = BSP_ERR_SHAPE; goto done; }
    h->NNZ = total;
    h->max_gt_nnz = (uint32_t)maxc;
    // values + at least 16 zeroed bytes of tail slack, so that 16-byte
    // vector loads of the last span never leave the allocation
    h->values_alloc = ((size_t)total * eb + 16 + 15) & ~(size_t)15;
    if (cudaMalloc(&h->values, h->values_alloc) != cudaSuccess) { st = BSP_ERR_OOM; goto done; }
    if (cudaMemsetAsync(h->values, 0, h->values_alloc, s) != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }
    if (eb == 2)
        enc_pack_kernel<2><<<grid_for(n_rowbytes, 256), 256, 0, s>>>(W, n_rowbytes, sh, h->bitmaps, h->offsets,
                                                                     bt_prefix, (uint8_t*)h->values);
    else
        enc_pack_kernel<1><<<grid_for(n_rowbytes, 256), 256, 0, s>>>(W, n_rowbytes, sh, h->bitmaps, h->offsets,
                                                                     bt_prefix, (uint8_t*)h->values);
    if (cudaGetLastError() != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }
    // the temporaries are freed below; make sure the pack has consumed them
    if (cudaStreamSynchronize(s) != cudaSuccess) st = BSP_ERR_CUDA;
done:
    cudaFree(bt_prefix);
    cudaFree(gt_nnz);
    cudaFree(overflow);
    return st;
}

bsp_status_t bsp_exclusive_scan_u32(const uint32_t* counts, int64_t n, uint32_t* offsets, int* overflow,
                                    cudaStream_t s)
{
    enc_scan_kernel<<<1, 1024, 0, s>>>(counts, n, offsets, overflow);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

bsp_status_t bsp_run_decode(const bsp_handle* h, void* W_out, cudaStream_t s)
{
    const int64_t n_rowbytes = h->Mp * h->Kp / 8;
    const EncShape sh{h->M, h->K / 8, h->Kp};
    if (bsp_elem_bytes(h->dtype) == 2)
        dec_kernel<2><<<grid_for(n_rowbytes, 256), 256, 0, s>>>(h->bitmaps, h->offsets, (const uint8_t*)h->values,
                                                                n_rowbytes, sh, W_out);
    else
        dec_kernel<1><<<grid_for(n_rowbytes, 256), 256, 0, s>>>(h->bitmaps, h->offsets, (const uint8_t*)h->values,
                                                                n_rowbytes, sh, W_out);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

bsp_status_t bsp_run_validate(bsp_handle* h, cudaStream_t s)
{
    int* bad = nullptr;
    int hbad = 0, maxc = 0;
    uint32_t last = 0;
    bsp_status_t st = BSP_OK;
    if (cudaMalloc(&bad, 2 * sizeof(int)) != cudaSuccess) return BSP_ERR_OOM;
    if (cudaMemsetAsync(bad, 0, 2 * sizeof(int), s) != cudaSuccess) { st = BSP_ERR_CUDA; goto done; }
    validate_kernel<<<grid_for(h->NGT * 32, 256), 256, 0, s>>>(h->bitmaps, h->offsets, h->NGT, h->M, h->K,
                                                               h->Kp / 64, bad);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(&hbad, bad, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&maxc, bad + 1, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&last, h->offsets + h->NGT, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        st = BSP_ERR_CUDA;
        goto done;
    }
    if (hbad || (uint64_t)last != h->NNZ) st = BSP_ERR_INVALID_ARG;
    h->max_gt_nnz = (uint32_t)maxc;
done:
    cudaFree(bad);
    return st;
}
