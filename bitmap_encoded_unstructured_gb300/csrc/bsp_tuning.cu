// Process-wide tuning knobs of the dispatch (bsp_set_tuning /
// bsp_get_tuning) and, in the test build only, the switches that make a
// bounded device-side wait run out (include/bsp_testing.h).
//
// The knobs start from the environment, read once per process on first
// use; product calls then read plain atomics, never the environment.
#include "bsp_internal.cuh"
#include "bsp_ptx.cuh"

#include <atomic>
#include <cstdlib>
#include <mutex>

#ifdef BSP_TESTING
#include "../../include/bsp_testing.h"
#endif

// Smallest fp16 N (up to BSP_DECODE_MAX_N) that runs the tcgen05 narrow
// kernel instead of the CUDA-core decode kernels, chosen from measurements
// on the OPT-13B projections: at N = 1 and 2 the GT-per-warp CUDA-core
// kernel is as fast or faster (QKV 29 / 33 us against 33 / 33 us); from
// N = 3 the narrow kernel is (2.6 TB/s against 1.7 for the team kernel).
#ifndef BSP_NARROW_MIN_N_DEFAULT
#define BSP_NARROW_MIN_N_DEFAULT 3
#endif
// The same crossover for int8 weights.  The narrow kernel multiplies exact
// fp16 copies of the int8 values; the CUDA-core alternative is the team
// kernel's dp4a.  Measured on the 11008 x 4096 and 4096 x 11008 layers at 50%
// and 60% (calls rotating over copies larger than L2): team 24.6 / 26.7 /
// 34.9 / 44.7 / 65.7 us at N = 1 / 2 / 3 / 8 / 16, narrow 28.8 at N = 1,
// 30.7 at N = 8, 33.7 at N = 16.
#ifndef BSP_NARROW_MIN_N_I8_DEFAULT
#define BSP_NARROW_MIN_N_I8_DEFAULT 3
#endif

namespace {

constexpr int kKnobs = 7;

struct Range {
    const char* env;
    int64_t lo, hi, dflt;
};

constexpr Range kRange[kKnobs] = {
    {"BSP_SPLITK", 0, 4096, 0},
    {"BSP_NARROW_CTAS", 0, 1 << 20, 0},
    {"BSP_UNION_SPLITK", 0, 4096, 0},
    {"BSP_NARROW_MIN_N", 1, 1024, BSP_NARROW_MIN_N_DEFAULT},
    {"BSP_PF_KSPLIT", -1, 1, -1},
    {"BSP_PF_SC", 0, 4096, 0},
    {"BSP_NARROW_MIN_N_I8", 1, 1024, BSP_NARROW_MIN_N_I8_DEFAULT},
};

std::atomic<int64_t> g_knob[kKnobs];
std::once_flag g_once;

void init_from_env()
{
    for (int i = 0; i < kKnobs; ++i) {
        int64_t v = kRange[i].dflt;
        if (const char* e = std::getenv(kRange[i].env)) {
            char* end = nullptr;
            const long long x = std::strtoll(e, &end, 10);
            if (end != e && x >= kRange[i].lo && x <= kRange[i].hi) v = x;
        }
        g_knob[i].store(v, std::memory_order_relaxed);
    }
}

inline void ensure_init() { std::call_once(g_once, init_from_env); }

#ifdef BSP_TESTING
std::atomic<uint32_t> g_spin_cap{0};
std::atomic<int> g_stall{0};
#endif

}  // namespace

int64_t bsp_tune(bsp_tune_t knob)
{
    ensure_init();
    const int i = (int)knob;
    if (i < 0 || i >= kKnobs) return 0;
    return g_knob[i].load(std::memory_order_relaxed);
}

uint32_t bsp_spin_cap()
{
#ifdef BSP_TESTING
    const uint32_t c = g_spin_cap.load(std::memory_order_relaxed);
    if (c) return c;
#endif
    return bspx::kSpinCap;
}

int bsp_test_stall()
{
#ifdef BSP_TESTING
    return g_stall.load(std::memory_order_relaxed);
#else
    return 0;
#endif
}

extern "C" {

bsp_status_t bsp_set_tuning(bsp_tune_t knob, int64_t value)
{
    ensure_init();
    const int i = (int)knob;
    if (i < 0 || i >= kKnobs) return BSP_ERR_INVALID_ARG;
    if (value < kRange[i].lo || value > kRange[i].hi) return BSP_ERR_INVALID_ARG;
    g_knob[i].store(value, std::memory_order_relaxed);
    return BSP_OK;
}

bsp_status_t bsp_get_tuning(bsp_tune_t knob, int64_t* value)
{
    ensure_init();
    const int i = (int)knob;
    if (i < 0 || i >= kKnobs || !value) return BSP_ERR_INVALID_ARG;
    *value = g_knob[i].load(std::memory_order_relaxed);
    return BSP_OK;
}

#ifdef BSP_TESTING
bsp_status_t bsp_testing_set_stall(int on)
{
    if (on != 0 && on != 1) return BSP_ERR_INVALID_ARG;
    g_stall.store(on, std::memory_order_relaxed);
    return BSP_OK;
}

bsp_status_t bsp_testing_set_spin_cap(uint32_t polls)
{
    g_spin_cap.store(polls, std::memory_order_relaxed);
    return BSP_OK;
}
#endif

}  // extern "C"

int64_t bsp_narrow_min_n(bsp_dtype_t dtype)
{
    return bsp_tune(dtype == BSP_INT8 ? BSP_TUNE_NARROW_MIN_N_I8 : BSP_TUNE_NARROW_MIN_N);
}
