// C-ABI entry points of libbsp (declared in include/bsp.h): argument
// checks, handle lifetime and dispatch to the kernels.  No exception or
// abort crosses the boundary; every failure is a bsp_status_t.
#include "bsp_internal.cuh"

#include <cstdlib>
#include <new>

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool valid(const bsp_handle* h) { return h != nullptr && h->magic == BSP_MAGIC; }

// Run on the handle's device, restoring the caller's current device after.
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

void free_handle(bsp_handle* h)
{
    if (!h) return;
    cudaFree(h->bitmaps);
    cudaFree(h->offsets);
    cudaFree(h->values);
    cudaFree(h->ws);
    cudaFree(h->ws_det);
    cudaFree(h->counters);
    cudaFree(h->err);
    cudaFree(h->stage_x);
    cudaFree(h->stage_y);
    cudaFree(h->cbc_offsets);
    cudaFree(h->cbc_colinfo);
    cudaFree(h->cbc_bitmaps);
    cudaFree(h->cbc_values);
    h->magic = 0;
    delete h;
}

bsp_status_t grow(void** p, size_t* have, size_t need)
{
    if (*have >= need) return BSP_OK;
    cudaFree(*p);
    *p = nullptr;
    *have = 0;
    if (cudaMalloc(p, need) != cudaSuccess) { *p = nullptr; return BSP_ERR_OOM; }
    *have = need;
    return BSP_OK;
}

// Split-K workspace (zeroed), strip counters (zeroed) and error word.
bsp_status_t alloc_scratch(bsp_handle* h, cudaStream_t s)
{
    const size_t ws_bytes = (size_t)BSP_DECODE_MAX_N * (size_t)h->M * 4;
    const size_t cnt_bytes = (size_t)(h->Mp / 64) * 4;
    if (cudaMalloc(&h->ws, ws_bytes) != cudaSuccess || cudaMalloc(&h->counters, cnt_bytes) != cudaSuccess ||
        cudaMalloc(&h->err, sizeof(int)) != cudaSuccess)
        return BSP_ERR_OOM;
    if (cudaMemsetAsync(h->ws, 0, ws_bytes, s) != cudaSuccess ||
        cudaMemsetAsync(h->counters, 0, cnt_bytes, s) != cudaSuccess ||
        cudaMemsetAsync(h->err, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return BSP_ERR_CUDA;
    return BSP_OK;
}

// Shapes the library takes: any M >= 1; K a multiple of 8 (fp16) or 16
// (int8), so that every row of W and of X starts on a 16-byte boundary (the
// bulk copies and vector loads need it).  M and K need not be multiples of
// 64: the format covers the zero-padded grid (edge GroupTiles padded with
// zeros, which are not stored).
bool shape_ok(bsp_dtype_t dtype, int64_t M, int64_t K)
{
    if (M <= 0 || K <= 0) return false;
    return (K % (dtype == BSP_INT8 ? 16 : 8)) == 0;
}

bsp_handle* new_handle(bsp_dtype_t dtype, int64_t M, int64_t K)
{
    bsp_handle* h = new (std::nothrow) bsp_handle{};
    if (!h) return nullptr;
    h->magic = BSP_MAGIC;
    h->dtype = dtype;
    h->M = M;
    h->K = K;
    h->Mp = (M + 63) / 64 * 64;
    h->Kp = (K + 63) / 64 * 64;
    h->NGT = (h->Mp / 64) * (h->Kp / 64);
    h->NBT = h->Mp * h->Kp / 64;
    h->max_gt_nnz = 4096;  // set from the arrays by the encoder / the import check
    return h;
}

}  // namespace

extern "C" {

const char* bsp_status_string(bsp_status_t s)
{
    switch (s) {
    case BSP_OK: return "ok";
    case BSP_ERR_INVALID_ARG: return "invalid argument";
    case BSP_ERR_SHAPE: return "bad shape: M, K >= 1, K a multiple of 8 (fp16) or 16 (int8), NNZ < 2^32";
    case BSP_ERR_DTYPE: return "dtype does not match the handle";
    case BSP_ERR_ALIGN: return "pointer not 16-byte aligned";
    case BSP_ERR_OOM: return "allocation failed";
    case BSP_ERR_CUDA: return "CUDA runtime error";
    case BSP_ERR_TIMEOUT: return "device-side wait timed out";
    case BSP_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

bsp_status_t bsp_encode(const void* W, bsp_dtype_t dtype, int64_t M, int64_t K,
                        bsp_stream_t stream, bsp_handle_t* out)
{
    if (!out) return BSP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!W) return BSP_ERR_INVALID_ARG;
    if (dtype != BSP_FP16 && dtype != BSP_INT8) return BSP_ERR_DTYPE;
    if (!shape_ok(dtype, M, K)) return BSP_ERR_SHAPE;
    if (!aligned16(W)) return BSP_ERR_ALIGN;
    bsp_handle* h = new_handle(dtype, M, K);
    if (!h) return BSP_ERR_OOM;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        free_handle(h);
        return BSP_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    bsp_status_t st = bsp_run_encode(h, W, s);
    if (st == BSP_OK) st = alloc_scratch(h, s);
    if (st != BSP_OK) { free_handle(h); return st; }
    *out = h;
    return BSP_OK;
}

bsp_status_t bsp_destroy(bsp_handle_t h)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    free_handle(h);
    return BSP_OK;
}

bsp_status_t bsp_spmm(bsp_handle_t h, const void* X, int64_t N, void* Y, bsp_stream_t stream)
{
    if (!valid(h) || !X || !Y || N < 1 || N > (int64_t)1 << 30) return BSP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y)) return BSP_ERR_ALIGN;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const bsp_out_mode mode = h->dtype == BSP_INT8 ? BSP_OUT_I32 : BSP_OUT_F16;
    if (N <= BSP_DECODE_MAX_N) {
        if (N >= bsp_narrow_min_n(h->dtype)) return bsp_run_spmm_narrow(bsp_problem_of(h), X, N, Y, s);
        return bsp_run_spmm_decode(bsp_problem_of(h), X, (int)N, Y, mode, nullptr, false, s);
    }
    // Larger N, fp16: the tcgen05 prefill kernel.
    if (h->dtype == BSP_FP16) return bsp_run_spmm_prefill(bsp_problem_of(h), X, N, Y, s);
    // Larger N, int8 (no int8 tensor-core path): the decode kernel over column blocks of 16 tokens.
    const int eb = bsp_elem_bytes(h->dtype);
    const int ob = h->dtype == BSP_INT8 ? 4 : 2;
    for (int64_t n0 = 0; n0 < N; n0 += BSP_DECODE_MAX_N) {
        const int nb = (int)((N - n0) < BSP_DECODE_MAX_N ? (N - n0) : BSP_DECODE_MAX_N);
 const bsp_status_t st = bsp_run_spmm_decode(
            bsp_problem_of(h), (const uint8_t*)X + n0 * h->K * eb, nb, (uint8_t*)Y + n0 * h->M * ob, mode, nullptr, false, s);
        if (st != BSP_OK) return st;
    }
    return BSP_OK;
}

bsp_status_t bsp_spmm_scaled(bsp_handle_t h, const int8_t* X, int64_t N, const float* row_scale,
                             float* Y, bsp_stream_t stream)
{
    if (!valid(h) || !X || !Y || !row_scale) return BSP_ERR_INVALID_ARG;
    if (h->dtype != BSP_INT8) return BSP_ERR_DTYPE;
    if (N < 1 || N > BSP_DECODE_MAX_N) return BSP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y)) return BSP_ERR_ALIGN;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    return bsp_run_spmm_decode(bsp_problem_of(h), X, (int)N, Y, BSP_OUT_F32_SCALED, row_scale, false,
                               (cudaStream_t)stream);
}

bsp_status_t bsp_spmspv(bsp_handle_t h, const void* x, void* y, bsp_stream_t stream)
{
    if (!valid(h) || !x || !y) return BSP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return BSP_ERR_ALIGN;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    if (h->cbc_values) return bsp_run_spmspv_cbc(h, x, y, 0.0f, (cudaStream_t)stream);
    const bsp_out_mode mode = h->dtype == BSP_INT8 ? BSP_OUT_I32 : BSP_OUT_F16;
    return bsp_run_spmm_decode(bsp_problem_of(h), x, 1, y, mode, nullptr, true, (cudaStream_t)stream);
}

bsp_status_t bsp_spmspv_threshold(bsp_handle_t h, const void* x, float threshold, void* y, bsp_stream_t stream)
{
    if (!valid(h) || !x || !y || !(threshold >= 0.f)) return BSP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return BSP_ERR_ALIGN;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    if (h->cbc_values) return bsp_run_spmspv_cbc(h, x, y, threshold, (cudaStream_t)stream);
    const bsp_out_mode mode = h->dtype == BSP_INT8 ? BSP_OUT_I32 : BSP_OUT_F16;
    return bsp_run_spmm_decode(bsp_problem_of(h), x, 1, y, mode, nullptr, true, (cudaStream_t)stream, threshold);
}

bsp_status_t bsp_build_column_index(bsp_handle_t h, bsp_stream_t stream)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    return bsp_run_build_cbc(h, (cudaStream_t)stream);
}

bsp_status_t bsp_column_index_bytes(bsp_handle_t h, uint64_t* bytes)
{
    if (!valid(h) || !bytes) return BSP_ERR_INVALID_ARG;
    if (!h->cbc_values) return BSP_ERR_INVALID_ARG;
    const uint64_t ngt = (uint64_t)(h->cbc_tr * h->cbc_tc);
    const uint64_t nbm = ngt * 256 * 64 / 64;
    *bytes = 4ull * (ngt + 1) + 4ull * ngt * 64 + 8ull * nbm + (uint64_t)bsp_elem_bytes(h->dtype) * h->NNZ;
    return BSP_OK;
}

bsp_status_t bsp_column_index_export(bsp_handle_t h, uint32_t* offsets, uint32_t* colinfo, uint64_t* bitmaps,
                                     void* values, bsp_stream_t stream)
{
    if (!valid(h) || !h->cbc_values) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t ngt = (size_t)(h->cbc_tr * h->cbc_tc);
    if (offsets && cudaMemcpyAsync(offsets, h->cbc_offsets, (ngt + 1) * 4, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (colinfo && cudaMemcpyAsync(colinfo, h->cbc_colinfo, ngt * 64 * 4, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (bitmaps && cudaMemcpyAsync(bitmaps, h->cbc_bitmaps, ngt * 64 * 4 * 8, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (values && h->NNZ &&
        cudaMemcpyAsync(values, h->cbc_values, (size_t)h->NNZ * bsp_elem_bytes(h->dtype), cudaMemcpyDefault, s) !=
            cudaSuccess)
        return BSP_ERR_CUDA;
    return BSP_OK;
}

namespace {

// H2D copy of X into the handle's staging buffer, the product, D2H copy of
// Y, all on `stream`; `sync`: then wait for them.
bsp_status_t spmm_host(bsp_handle_t h, const void* X_host, int64_t N, void* Y_host, bsp_stream_t stream, bool sync)
{
    if (!valid(h) || !X_host || !Y_host || N < 1 || N > (int64_t)1 << 30) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t xb = (size_t)N * h->K * bsp_elem_bytes(h->dtype);
    const size_t yb = (size_t)N * h->M * (h->dtype == BSP_INT8 ? 4 : 2);
    bsp_status_t st = grow(&h->stage_x, &h->stage_x_bytes, xb);
    if (st != BSP_OK) return st;
    st = grow(&h->stage_y, &h->stage_y_bytes, yb);
    if (st != BSP_OK) return st;
    if (cudaMemcpyAsync(h->stage_x, X_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    st = bsp_spmm(h, h->stage_x, N, h->stage_y, stream);
    if (st != BSP_OK) return st;
    if (cudaMemcpyAsync(Y_host, h->stage_y, yb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return BSP_ERR_CUDA;
    if (sync && cudaStreamSynchronize(s) != cudaSuccess) return BSP_ERR_CUDA;
    return BSP_OK;
}

}  // namespace

bsp_status_t bsp_spmm_host(bsp_handle_t h, const void* X_host, int64_t N, void* Y_host, bsp_stream_t stream)
{
    return spmm_host(h, X_host, N, Y_host, stream, true);
}

bsp_status_t bsp_spmm_host_async(bsp_handle_t h, const void* X_host, int64_t N, void* Y_host,
                                 bsp_stream_t stream)
{
    return spmm_host(h, X_host, N, Y_host, stream, false);
}

bsp_status_t bsp_storage_bytes(bsp_handle_t h, uint64_t* bytes)
{
    if (!valid(h) || !bytes) return BSP_ERR_INVALID_ARG;
    *bytes = 4ull * (uint64_t)(h->NGT + 1) + 8ull * (uint64_t)h->NBT +
             (uint64_t)bsp_elem_bytes(h->dtype) * h->NNZ;
    return BSP_OK;
}

bsp_status_t bsp_cr(bsp_handle_t h, double* cr)
{
    uint64_t stor = 0;
    const bsp_status_t st = bsp_storage_bytes(h, &stor);
    if (st != BSP_OK) return st;
    if (!cr) return BSP_ERR_INVALID_ARG;
    *cr = (double)bsp_elem_bytes(h->dtype) * (double)h->M * (double)h->K / (double)stor;
    return BSP_OK;
}

bsp_status_t bsp_info(bsp_handle_t h, bsp_info_t* o)
{
    if (!valid(h) || !o) return BSP_ERR_INVALID_ARG;
    o->M = h->M;
    o->K = h->K;
    o->dtype = h->dtype;
    o->gt_m = 64;
    o->gt_k = 64;
    o->device = h->device;
    o->NGT = h->NGT;
    o->NBT = h->NBT;
    o->NNZ = h->NNZ;
    o->bitmaps = h->bitmaps;
    o->offsets = h->offsets;
    o->values = h->values;
    return BSP_OK;
}

bsp_status_t bsp_set_deterministic(bsp_handle_t h, int on)
{
    if (!valid(h) || (on != 0 && on != 1)) return BSP_ERR_INVALID_ARG;
    if (on && !h->ws_det) {
        DeviceGuard g(h->device);
        if (!g.ok) return BSP_ERR_CUDA;
        const int slots = bsp_decode_split_cap(bsp_problem_of(h));
        const size_t bytes = (size_t)slots * BSP_DECODE_MAX_N * (size_t)h->M * 4;
        if (cudaMalloc(&h->ws_det, bytes) != cudaSuccess) {
            h->ws_det = nullptr;
            return BSP_ERR_OOM;
        }
        h->det_slots = slots;
    }
    h->deterministic = on;
    return BSP_OK;
}

bsp_status_t bsp_export(bsp_handle_t h, uint64_t* bitmaps, uint32_t* offsets, void* values,
                        bsp_stream_t stream)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (bitmaps && cudaMemcpyAsync(bitmaps, h->bitmaps, (size_t)h->NBT * 8, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (offsets && cudaMemcpyAsync(offsets, h->offsets, (size_t)(h->NGT + 1) * 4, cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (values && h->NNZ &&
        cudaMemcpyAsync(values, h->values, (size_t)h->NNZ * bsp_elem_bytes(h->dtype), cudaMemcpyDefault, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    return BSP_OK;
}

bsp_status_t bsp_import(const uint64_t* bitmaps, const uint32_t* offsets, const void* values, bsp_dtype_t dtype,
                        int64_t M, int64_t K, uint64_t nnz, bsp_stream_t stream, bsp_handle_t* out)
{
    if (!out) return BSP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!bitmaps || !offsets || (nnz && !values)) return BSP_ERR_INVALID_ARG;
    if (dtype != BSP_FP16 && dtype != BSP_INT8) return BSP_ERR_DTYPE;
    if (!shape_ok(dtype, M, K) || nnz > 0xFFFFFFFFull || nnz > (uint64_t)M * (uint64_t)K) return BSP_ERR_SHAPE;
    bsp_handle* h = new_handle(dtype, M, K);
    if (!h) return BSP_ERR_OOM;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        free_handle(h);
        return BSP_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    const int eb = bsp_elem_bytes(dtype);
    h->NNZ = nnz;
    h->values_alloc = ((size_t)nnz * eb + 16 + 15) & ~(size_t)15;
    if (cudaMalloc(&h->bitmaps, (size_t)h->NBT * 8) != cudaSuccess ||
        cudaMalloc(&h->offsets, (size_t)(h->NGT + 1) * 4) != cudaSuccess ||
        cudaMalloc(&h->values, h->values_alloc) != cudaSuccess) {
        free_handle(h);
        return BSP_ERR_OOM;
    }
    if (cudaMemcpyAsync(h->bitmaps, bitmaps, (size_t)h->NBT * 8, cudaMemcpyDefault, s) != cudaSuccess ||
        cudaMemcpyAsync(h->offsets, offsets, (size_t)(h->NGT + 1) * 4, cudaMemcpyDefault, s) != cudaSuccess ||
        cudaMemsetAsync(h->values, 0, h->values_alloc, s) != cudaSuccess ||
        (nnz && cudaMemcpyAsync(h->values, values, (size_t)nnz * eb, cudaMemcpyDefault, s) != cudaSuccess)) {
        free_handle(h);
        return BSP_ERR_CUDA;
    }
    bsp_status_t st = bsp_run_validate(h, s);
    if (st == BSP_OK) st = alloc_scratch(h, s);
    if (st != BSP_OK) { free_handle(h); return st; }
    *out = h;
    return BSP_OK;
}

bsp_status_t bsp_check(bsp_handle_t h, bsp_stream_t stream)
{
    if (!valid(h)) return BSP_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int e = 0;
    if (cudaMemcpyAsync(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(h->err, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (e) {
        // a call that gave up may have left partial sums and arrival counts
        // behind: restore the zero state the next call relies on
        if (cudaMemsetAsync(h->ws, 0, (size_t)BSP_DECODE_MAX_N * (size_t)h->M * 4, s) != cudaSuccess ||
            cudaMemsetAsync(h->counters, 0, (size_t)(h->Mp / 64) * 4, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return BSP_ERR_CUDA;
    }
    return e ? (bsp_status_t)e : BSP_OK;
}

bsp_status_t bsp_decode(bsp_handle_t h, void* W_out, bsp_stream_t stream)
{
    if (!valid(h) || !W_out) return BSP_ERR_INVALID_ARG;
    if (!aligned16(W_out)) return BSP_ERR_ALIGN;
    DeviceGuard g(h->device);
    if (!g.ok) return BSP_ERR_CUDA;
    return bsp_run_decode(h, W_out, (cudaStream_t)stream);
}

}  // extern "C"
