// bsp_spmm_noalloc: the decode-path product for callers that cannot
// allocate device memory.
//
// The handle-based bsp_spmm keeps its split-K scratch (partial-sum
// workspace, per-strip arrival counters, error word) in memory that
// bsp_encode allocated.  Some callers cannot make that allocation at all:
// code that runs under a host framework which owns every device buffer and
// hands an operator only its inputs and outputs, real-time loops where
// cudaMalloc / cudaFree (and the device synchronisation cudaFree implies)
// is not allowed, or arenas whose memory accounting must not be bypassed.
// This entry point takes the encoded arrays and X / Y from the caller and
// uses a fixed scratch array compiled into the library instead.
//
// The scratch is a file-scope __device__ array of fixed size; every GPU
// that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the address is
// looked up once per device with cudaGetSymbolAddress (on the first call on
// that device, with that device current) and passed to the kernel.
#include "bsp_internal.cuh"

#include <mutex>

namespace {

// workspace [BSP_DECODE_MAX_N][BSP_NOALLOC_MAX_M] fp32 / int32, then one
// counter per 64-row strip, then the error word
constexpr size_t kWsBytes = (size_t)BSP_DECODE_MAX_N * BSP_NOALLOC_MAX_M * 4;
constexpr size_t kCounterBytes = (size_t)(BSP_NOALLOC_MAX_M / 64) * 4;
constexpr size_t kScratchBytes = kWsBytes + kCounterBytes + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
    bool ready = false;
    unsigned char* ptr = nullptr;
    int num_sms = 0;
};

constexpr int kMaxDevices = 64;
DeviceScratch g_dev[kMaxDevices];
std::mutex g_mu;

// Once per device (the device must be current): resolve the scratch
// address, read the SM count and zero the scratch.
bsp_status_t setup(int dev, DeviceScratch** out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceScratch& d = g_dev[dev];
    if (!d.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return BSP_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BSP_ERR_CUDA;
        if (cudaMemset(p, 0, kScratchBytes) != cudaSuccess) return BSP_ERR_CUDA;
        d.ptr = static_cast<unsigned char*>(p);
        d.num_sms = sms;
        d.ready = true;
    }
    *out = &d;
    return BSP_OK;
}

}  // namespace

extern "C" bsp_status_t bsp_spmm_noalloc(const uint64_t* bitmaps, const uint32_t* offsets,
                                         const void* values, bsp_dtype_t dtype, int64_t M, int64_t K,
                                         const void* X, int64_t N, void* Y, bsp_stream_t stream)
{
    if (!bitmaps || !offsets || !values || !X || !Y) return BSP_ERR_INVALID_ARG;
    if (dtype != BSP_FP16 && dtype != BSP_INT8) return BSP_ERR_DTYPE;
    if (M <= 0 || K <= 0 || (M % 64) || (K % 64) || M > BSP_NOALLOC_MAX_M) return BSP_ERR_SHAPE;
    if (N < 1 || N > BSP_DECODE_MAX_N) return BSP_ERR_SHAPE;
    if (((uintptr_t)bitmaps | (uintptr_t)values | (uintptr_t)X | (uintptr_t)Y) & 15u)
        return BSP_ERR_ALIGN;
    if ((uintptr_t)offsets & 3u) return BSP_ERR_ALIGN;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSP_ERR_CUDA;
    DeviceScratch* d = nullptr;
    const bsp_status_t st = setup(dev, &d);
    if (st != BSP_OK) return st;

    cudaStream_t s = (cudaStream_t)stream;
    // The scratch keeps whatever the previous call left: clear the parts
    // this call relies on starting at zero (its workspace slice: 16 M
    // entries, which covers both the CUDA-core kernels' [N][M] layout and
    // the narrow kernel's [M][16]; the strip counters; the error word).
    unsigned char* ws = d->ptr;
    unsigned char* counters = d->ptr + kWsBytes;
    int* err = reinterpret_cast<int*>(d->ptr + kWsBytes + kCounterBytes);
    if (cudaMemsetAsync(ws, 0, (size_t)BSP_DECODE_MAX_N * (size_t)M * 4, s) != cudaSuccess ||
        cudaMemsetAsync(counters, 0, (size_t)(M / 64) * 4, s) != cudaSuccess ||
        cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess)
        return BSP_ERR_CUDA;

    bsp_decode_problem p;
    p.bitmaps = bitmaps;
    p.offsets = offsets;
    p.values = values;
    p.dtype = dtype;
    p.M = M;
    p.K = K;
    p.Mp = M;  // this entry takes multiples of 64 only
    p.Kp = K;
    p.max_gt_nnz = 4096;  // the arrays are not inspected: any GT may be dense
    p.device = dev;
    p.num_sms = d->num_sms;
    // the CUDA-core kernels index the workspace as [n][M] and the narrow
    // kernel as [M][16] (fp32, or int32 for int8): all within the 16 M
    // entries cleared above, the handle's layouts with M as the pitch
    p.ws = ws;
    p.counters = reinterpret_cast<uint32_t*>(counters);
    p.err = err;
    // the dispatch of bsp_spmm
    if (N >= bsp_narrow_min_n(dtype)) return bsp_run_spmm_narrow(p, X, N, Y, s);
    const bsp_out_mode mode = dtype == BSP_INT8 ? BSP_OUT_I32 : BSP_OUT_F16;
    return bsp_run_spmm_decode(p, X, (int)N, Y, mode, nullptr, false, s);
}
