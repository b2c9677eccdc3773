// Narrow product Y = W * X for fp16 and 1 <= N <= 16 on the 5th-generation
// tensor cores: the decode-then-multiply scheme of the prefill kernel
// (spmm_prefill.cu) with one MMA of N = 16 per K = 16.
//
// Method: "load as sparse, compute as dense" ("Unified Static-Dynamic
// Pruning for Efficient LLM Inference", section 4.3; "SpInfer: How bitmaps
// make sparse LLMs actually fast", sections "Shared Memory Bitmap Decoding
// (SMBD)" and "The async pipeline").  At N <= 16 the CUDA-core decode path
// spends one FMA per nonzero and column (and the same again for the zero
// positions, which are predicated, not skipped): at N = 16 that is more
// instruction issue than the HBM budget of a GroupTile allows.  Decoded
// into a dense A tile, the same GroupTile costs four tcgen05.mma
// instructions at any N <= 16; the decode (about one shared-memory load
// per position, no conversion, no FMA) then sets the pace.
//
// CTA tile: 128 rows of W (two GT row strips) x 16 columns of Y; one GT
// column (K = 64) per pipeline step; `splits` CTAs share a tile's GT
// columns (split-K) and meet in the handle's split-K workspace.  Rings:
//   C  compressed data  bitmaps + value spans of the two GTs (bulk copies),
//                       the rest of shared memory in stages sized for the
//                       densest GT (up to SC_MAX), producer -> decoders
//   A  decoded W tile   128 x 64 fp16, K-major, SWIZZLE_128B (16 KB),
//                       2 stages, decoders -> MMA
//   B  X sub-tiles      16 x 64 fp16, K-major, SWIZZLE_128B (TMA, rows
//                       past N read as zeros), 8 stages, producer -> MMA
// Warp roles (21 warps): warp 0 C producer; warp 1 TMEM allocation and the
// MMA issuer (tcgen05.mma.cta_group::1.kind::f16, M = 128, N = 16, K = 16);
// warps 2-3 scanners (row starts of every BT row); warps 4-19 decoders
// (whole row-bytes into the swizzled A tile); warp 20 B producer; warps 4-7
// then the epilogue (tcgen05.ld of their TMEM lane quadrant).
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

// Self-checks (off by default): bounds of every global access and of the
// data-derived shared-memory addresses, recorded in the error word as
// 100 + site, the access skipped.
#ifndef BSP_NW_CHECKS
#define BSP_NW_CHECKS 0
#endif
// split model: fixed cost of a CTA in GT-column steps
#ifndef BSP_NARROW_CTA_COST
#define BSP_NARROW_CTA_COST 6
#endif
// resident CTAs per SM: 1 gives a CTA the whole shared memory (the deepest
// C ring); 2 halves it and caps the registers at 48 per thread, so that a
// second CTA's 21 warps hide the decoders' latency
#ifndef BSP_NARROW_MINB
#define BSP_NARROW_MINB 2
#endif

namespace {

constexpr int BM = 128, BN = 16, BK = 64;  // tile rows, MMA columns, GT columns per step
constexpr int A_BYTES = BM * BK * 2;       // 16384
constexpr int DEC_WARPS = 16;              // eight per GroupTile
constexpr int WPG = DEC_WARPS / 2;         // decoder warps per GroupTile
constexpr int NR = 2;                      // row-bytes per decoder lane and step
static_assert(WPG * 32 * NR == 512, "the decoder warps of a GT cover its 64 x 8 row-bytes");
constexpr int DEC0 = 4;                    // first decoder warp (after producer, MMA, 2 scanners)
constexpr int BPROD = DEC0 + DEC_WARPS;    // B (X tile) producer, the last warp
constexpr int WARPS = BPROD + 1;
constexpr int THREADS = WARPS * 32;
constexpr int RS_BYTES = 64 * 8 * 2;       // row starts of one GT: [BT][row] u16
constexpr uint32_t kSleepNs = 1000;        // suspend hint of the waiting polls

constexpr int SB = 8;                      // X sub-tile stages
constexpr int SA = 2;                      // decoded A tile stages
constexpr int SC_MAX = 12;                 // barrier slots of the C ring
constexpr int MINB = BSP_NARROW_MINB;
static_assert(MINB == 1 || MINB == 2, "one or two CTAs per SM");
// shared memory of a CTA: all of it, or half of the SM's 228 KB less the
// 1 KB the driver reserves per resident CTA
constexpr int SMEM_MAX = MINB == 1 ? 227 * 1024 : 228 * 1024 / 2 - 1024;
constexpr int B_STAGE = BN * BK * 2;       // 2 KB
constexpr int OFF_B = 0;                   // 1024-B aligned regions first
constexpr int OFF_A = OFF_B + SB * B_STAGE;
constexpr int OFF_BAR = OFF_A + SA * A_BYTES;
// barriers: c_full[SC_MAX] c_empty[SC_MAX] c_scan[SC_MAX] b_full[SB] b_empty[SB] a_full[SA] a_empty[SA] acc
constexpr int NBAR = 3 * SC_MAX + 2 * SB + 2 * SA + 1;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;  // TMEM address (4 B), last-CTA flag (4 B)
constexpr int OFF_C = (OFF_TMEM + 16 + 127) & ~127;
constexpr int C_BYTES = SMEM_MAX - 1024 - OFF_C;  // 1024: slack to align the base to 1024 B
constexpr uint32_t TMEM_COLS = 32;                // the allocation minimum; the accumulator uses 16

// One C stage: two GT slots (512 B of bitmaps, then the 16-B chunks that
// hold the GT's value span), a 16-B header (the value shifts) and the row
// starts of the two GTs.  The slot is sized for the densest GT of the
// matrix, so the number of stages that fit follows the density.
constexpr uint32_t c_slot_bytes(uint32_t max_gt_nnz)
{
    return (512u + 16u * ((max_gt_nnz + 7u) / 8u + 1u) + 127u) & ~127u;
}
constexpr uint32_t c_stage_bytes(uint32_t slot)
{
    return (2u * slot + 16u + 2u * (uint32_t)RS_BYTES + 127u) & ~127u;
}
static_assert(C_BYTES >= 2 * (int)c_stage_bytes(c_slot_bytes(4096)), "two dense C stages");
static_assert((B_STAGE % 1024) == 0 && (A_BYTES % 1024) == 0, "swizzle atoms need 1024-B alignment");

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// M = 128, N = 16.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct NarrowArgs {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const uint8_t* values;
    __half* Y;
    int64_t M, N, K;           // logical: Y rows, columns, X row length
    int64_t Mp, KT;            // padded grid: rows (a multiple of 64), GT columns
    uint32_t c_slot, c_stage;  // C ring geometry (bytes): GT slot, stage
    int sc;                    // C stages in use, 2..SC_MAX
    // split-K over `splits` CTAs per tile: partial sums into the workspace
    // [N][M] fp32 (zero between calls) by atomic adds, or into the
    // deterministic slots [splits][N][M]; one arrival counter per tile (at
    // its first 64-row strip); the last CTA of a tile writes Y
    int splits;
    float* ws;
    float* ws_det;
    uint32_t* counters;
    int64_t ngt;            // GTs of the grid (self-checks)
    uint64_t values_bytes;  // bytes allocated for values, 0: unknown (self-checks)
    int* err;
    uint32_t spin_cap;
};

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

__device__ __forceinline__ int bt_local(int br, int bc)
{
    return (((br >> 1) * 4 + (bc >> 1)) << 2) + (br & 1) + ((bc & 1) << 1);
}

// One position of a row-byte, without a branch: if rbyte & bit, the next
// packed fp16 value (shared-memory byte address `addr`) zero-extended, and
// addr advances by one value; else 0.  Volatile: it reads shared memory,
// so it is neither duplicated nor moved across the ring-barrier waits.
__device__ __forceinline__ uint32_t take_f16(uint32_t& addr, uint32_t rbyte, uint32_t bit)
{
    uint32_t v;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 t;\n\t"
        "and.b32 t, %2, %3;\n\t"
        "setp.ne.b32 p, t, 0;\n\t"
        "mov.b32 %0, 0;\n\t"
        "@p ld.shared.u16 %0, [%1];\n\t"
        "@p add.u32 %1, %1, 2;\n\t}"
        : "=r"(v), "+r"(addr)
        : "r"(rbyte), "r"(bit));
    return v;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            bspx::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bspx::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accum)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bspx::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

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

// Grid: tiles x splits CTAs, split fastest; CTA (tile, part) takes the
// balanced share [part * KT / splits, (part + 1) * KT / splits) of the GT
// columns (at least one: the host keeps splits <= KT).
__global__ void __launch_bounds__(THREADS, MINB)
spmm_narrow_kernel(const __grid_constant__ CUtensorMap tmX, const NarrowArgs a)
{
    const int SC = a.sc;
    const uint32_t SLOT = a.c_slot, C_HDR = 2 * SLOT, C_RS = C_HDR + 16;
    const uint32_t vchunks = (SLOT - 512) / 16;  // value chunks a slot holds
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-B alignment of the shared-window offset (the 128-B swizzle atoms)
    uint8_t* smem = smem_raw + ((1024u - (bspx::smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr uint32_t FULL = 0xFFFFFFFFu;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint64_t* c_full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* c_empty = c_full + SC_MAX;
    uint64_t* c_scan = c_empty + SC_MAX;
    uint64_t* b_full = c_scan + SC_MAX;
    uint64_t* b_empty = b_full + SB;
    uint64_t* a_full = b_empty + SB;
    uint64_t* a_empty = a_full + SA;
    uint64_t* acc_bar = a_empty + SA;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    int* s_last = reinterpret_cast<int*>(smem + OFF_TMEM + 4);
    auto b_stage = [&](int s) { return smem + OFF_B + s * B_STAGE; };
    auto a_stage = [&](int s) { return smem + OFF_A + s * A_BYTES; };
    auto c_stage = [&](int s) { return smem + OFF_C + s * a.c_stage; };

    const int64_t M = a.M, N = a.N;
    const uint32_t KTA = (uint32_t)a.KT;  // GT columns of the grid (row pitch)
    const uint32_t part = blockIdx.x % (uint32_t)a.splits, nparts = (uint32_t)a.splits;
    const uint32_t k0 = (uint32_t)((uint64_t)part * KTA / nparts);             // first GT column
    const uint32_t KT = (uint32_t)((uint64_t)(part + 1) * KTA / nparts) - k0;  // GT columns of this CTA
    const int64_t mt = (int64_t)(blockIdx.x / (uint32_t)a.splits);              // tile
    const int64_t strip0 = 2 * mt, strip1 = 2 * mt + 1;
    const bool has_b = strip1 * 64 < a.Mp;  // second GT row strip of the tile exists
    const uint32_t cap = a.spin_cap;

    if (warp == 1) {  // 32 TMEM columns (the minimum) for the 128 x 16 accumulator
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         bspx::smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC; ++s) {
            bspx::mbar_init(c_full + s, 1);
            bspx::mbar_init(c_empty + s, DEC_WARPS);
            bspx::mbar_init(c_scan + s, 2 * 32);  // every scanner lane
        }
        for (int s = 0; s < SB; ++s) {
            bspx::mbar_init(b_full + s, 1);
            bspx::mbar_init(b_empty + s, 1);
        }
        for (int s = 0; s < SA; ++s) {
            bspx::mbar_init(a_full + s, DEC_WARPS);
            bspx::mbar_init(a_empty + s, 1);
        }
        bspx::mbar_init(acc_bar, 1);
        bspx::fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    bool failed = false;

    if (warp == 0) {
        // ---------------- C producer: the two GTs of each step, up to SC steps ahead
        const int64_t ta = strip0 * KTA + k0, tb = strip1 * KTA + k0;
        uint32_t offa = 0, offb = 0;
        uint32_t wbase = 0;
        uint32_t s = 0, ph = 0;  // stage and its phase parity
        uint32_t kc = 0;         // steps issued
        for (; kc < KT; ++kc) {
            if (kc >= (uint32_t)SC &&
                !__all_sync(FULL, bspx::mbar_wait_sleep(c_empty + s, ph ^ 1u, cap, kSleepNs))) {
                failed = true;
                break;
            }
            if (kc == 0 || kc - wbase >= 31) {  // window of offsets: lane i holds offsets[t + wbase + i]
                wbase = kc;
                const uint32_t i = wbase + lane;
                offa = offb = 0;
#if BSP_NW_CHECKS
                if ((i <= KT && ta + i > a.ngt) || (has_b && i <= KT && tb + i > a.ngt))
                    atomicCAS(a.err, 0, 101);
                else
#endif
                {
                    if (i <= KT) offa = __ldg(a.offsets + ta + i);
                    if (has_b && i <= KT) offb = __ldg(a.offsets + tb + i);
                }
            }
            const int w = (int)(kc - wbase);
            const uint32_t oa0 = __shfl_sync(FULL, offa, w), oa1 = __shfl_sync(FULL, offa, w + 1);
            const uint32_t ob0 = __shfl_sync(FULL, offb, w), ob1 = __shfl_sync(FULL, offb, w + 1);
            if (lane == 0) {
                uint8_t* st = c_stage(s);
                uint32_t* hdr = reinterpret_cast<uint32_t*>(st + C_HDR);
                const uint32_t cha = oa0 / 8, chb = ob0 / 8;
                uint32_t nca = (oa1 + 7) / 8 - cha, ncb = has_b ? (ob1 + 7) / 8 - chb : 0u;
                if (nca > vchunks || ncb > vchunks) {  // a GT denser than the handle recorded
                    atomicExch(a.err, (int)BSP_ERR_INTERNAL);
                    nca = min(nca, vchunks);
                    ncb = min(ncb, vchunks);
                }
#if BSP_NW_CHECKS
                if (a.values_bytes && ((uint64_t)(cha + nca) * 16 > a.values_bytes ||
                                       (uint64_t)(chb + ncb) * 16 > a.values_bytes)) {
                    atomicCAS(a.err, 0, 102);
                    nca = ncb = 0;
                }
#endif
                hdr[0] = oa0 - cha * 8;
                hdr[1] = ob0 - chb * 8;
                uint32_t bytes = 512 + nca * 16;
                if (has_b) bytes += 512 + ncb * 16;
                bspx::mbar_arrive_expect_tx(c_full + s, bytes);
                bspx::bulk_g2s(st, a.bitmaps + (ta + kc) * 64, 512, c_full + s);
                if (nca) bspx::bulk_g2s(st + 512, a.values + (int64_t)cha * 16, nca * 16, c_full + s);
                if (has_b) {
                    bspx::bulk_g2s(st + SLOT, a.bitmaps + (tb + kc) * 64, 512, c_full + s);
                    if (ncb) bspx::bulk_g2s(st + SLOT + 512, a.values + (int64_t)chb * 16, ncb * 16, c_full + s);
                }
            }
            if (++s == (uint32_t)SC) { s = 0; ph ^= 1u; }
        }
        // let the last copies land before the CTA can exit (bounded)
        for (uint32_t k = (kc > (uint32_t)SC ? kc - SC : 0); k < kc; ++k)
            bspx::mbar_wait_bounded(c_full + (k % SC), (k / SC) & 1u, cap);
    } else if (warp == BPROD) {
        // ---------------- B producer: one 16 x 64 X sub-tile per step by TMA
        uint32_t s = 0, ph = 0;
        uint32_t i = 0;
        for (; i < KT; ++i) {
            if (i >= (uint32_t)SB &&
                !__all_sync(FULL, bspx::mbar_wait_sleep(b_empty + s, ph ^ 1u, cap, kSleepNs))) {
                failed = true;
                break;
            }
            if (lane == 0) {
                bspx::mbar_arrive_expect_tx(b_full + s, (uint32_t)B_STAGE);
                tma_load_2d(b_stage(s), &tmX, (int)((k0 + i) * BK), 0, b_full + s);
            }
            if (++s == (uint32_t)SB) { s = 0; ph ^= 1u; }
        }
        for (uint32_t k = (i > (uint32_t)SB ? i - SB : 0); k < i; ++k)
            bspx::mbar_wait_bounded(b_full + (k % SB), (k / SB) & 1u, cap);
    } else if (warp == 1) {
        // ---------------- MMA issuer
        uint32_t sa = 0, pa = 0, sb = 0, pb = 0;
        for (uint32_t kb = 0; kb < KT && !failed; ++kb) {
            bool ok = bspx::mbar_wait_sleep(a_full + sa, pa, cap, kSleepNs);
            ok = ok && bspx::mbar_wait_sleep(b_full + sb, pb, cap, kSleepNs);
            if (!__all_sync(FULL, ok)) { failed = true; break; }
            tc_fence_after();
            if (lane == 0) {
                const uint64_t ad = smem_desc_sw128(bspx::smem_u32(a_stage(sa)));
                const uint64_t bd = smem_desc_sw128(bspx::smem_u32(b_stage(sb)));
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)  // K = 16 per MMA: 32 B along the swizzled row
                    umma_f16(tmem_base, ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j), (kb | j) ? 1u : 0u);
                umma_commit(b_empty + sb);  // fire once the MMAs above are done
                umma_commit(a_empty + sa);
            }
            __syncwarp();
            if (++sb == (uint32_t)SB) { sb = 0; pb ^= 1u; }
            if (++sa == (uint32_t)SA) { sa = 0; pa ^= 1u; }
        }
        if (lane == 0) umma_commit(acc_bar);  // fires once every MMA issued above is done
        __syncwarp();
        bspx::mbar_wait_bounded(acc_bar, 0, cap);
        __syncwarp();
    } else if (warp < DEC0) {
        // ---------------- scanners: row starts of GT (warp - 2)
        const int gsel = warp - 2;
        const bool active = gsel == 0 || has_b;
        uint32_t sc = 0, pc = 0;
        for (uint32_t kb = 0; kb < KT; ++kb) {
            const bool ok = bspx::mbar_wait_sleep(c_full + sc, pc, cap, kSleepNs);
            if (!__all_sync(FULL, ok)) { failed = true; break; }
            uint8_t* st = c_stage(sc);
            if (active) {
                // lane: BTs 2 lane and 2 lane + 1 (GT order = value order)
                const ulonglong2 bb = reinterpret_cast<const ulonglong2*>(st + gsel * SLOT)[lane];
                const uint32_t shift = reinterpret_cast<const uint32_t*>(st + C_HDR)[gsel];
                const uint32_t c0 = __popcll(bb.x), c1 = __popcll(bb.y);
                uint32_t incl = c0 + c1;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t o = __shfl_up_sync(FULL, incl, d);
                    if (lane >= d) incl += o;
                }
                const uint32_t base0 = incl - (c0 + c1) + shift;
                uint4* rs = reinterpret_cast<uint4*>(st + C_RS + gsel * RS_BYTES) + 2 * lane;
                rs[0] = bspx::row_starts(bb.x, base0);
                rs[1] = bspx::row_starts(bb.y, base0 + c0);
            }
            __syncwarp();
            bspx::mbar_arrive(c_scan + sc);  // release: the row starts above
            if (++sc == (uint32_t)SC) { sc = 0; pc ^= 1u; }
        }
    } else if (warp < BPROD) {
        // ---------------- decoders.  Row-byte j of a lane: row 16q + lane % 16
        // of the GT, octet bc = 2 p0 + 2 (lane / 16) + j; its eight positions
        // become one whole 16-B chunk of the A tile.  Each quarter-warp
        // writes the chunks of eight consecutive rows of one octet, which the
        // swizzle puts in distinct banks.
        const int dw = warp - DEC0;
        const int gsel = dw / WPG, wq = dw % WPG;
        const int q = wq / 2;         // TCTile row of the warp (16 GT rows)
        const int p0 = (wq % 2) * 2;  // first TCTile column (octet pair) of the warp
        const int row = 16 * q + (lane & 15);  // row inside the GT
        const int trow = 64 * gsel + row;      // row inside the 128-row tile
        int ent[NR];       // BT row entry: 8 g + row % 8 (bitmap byte / row start)
        uint32_t dst[NR];  // byte offset of the row-byte's 16-B chunk in A (128-B swizzle)
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int bc = 2 * p0 + 2 * (lane >> 4) + j;
            ent[j] = 8 * bt_local(row >> 3, bc) + (row & 7);
            dst[j] = (uint32_t)((trow >> 3) * 1024 + (trow & 7) * 128 + ((bc ^ (trow & 7)) << 4));
        }
        const bool active = gsel == 0 || has_b;
        uint32_t sc = 0, pc = 0, sa = 0, pa = 0;
        for (uint32_t kb = 0; kb < KT; ++kb) {
            // c_scan implies c_full: the scanners arrive only after they saw it
            bool ok = bspx::mbar_wait_sleep(c_scan + sc, pc, cap, kSleepNs);
            if (kb >= (uint32_t)SA) ok = ok && bspx::mbar_wait_sleep(a_empty + sa, pa ^ 1u, cap, kSleepNs);
            if (!__all_sync(FULL, ok)) { failed = true; break; }
            const uint8_t* st = c_stage(sc);
            uint8_t* at = a_stage(sa);
            if (active) {
                const uint8_t* bmb = st + gsel * SLOT;  // bitmap bytes: byte 8 g + r = row r of BT g
                const uint16_t* rst = reinterpret_cast<const uint16_t*>(st + C_RS + gsel * RS_BYTES);
                const uint32_t vbase = bspx::smem_u32(st + gsel * SLOT + 512);
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const uint32_t byte = bmb[ent[j]];
                    uint32_t start = (uint32_t)rst[ent[j]];
#if BSP_NW_CHECKS
                    if (2u * (start + 8u) > SLOT - 512u) { atomicCAS(a.err, 0, 110); start = 0; }
#endif
                    uint32_t addr = vbase + 2u * start;
                    uint32_t h[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) h[c] = take_f16(addr, byte, 1u << c);
                    *reinterpret_cast<uint4*>(at + dst[j]) =
                        make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
                }
            } else {
                // rows of a missing second strip: zeros, so that the MMA
                // reads defined values (their Y rows are not written)
#pragma unroll
                for (int j = 0; j < NR; ++j) *reinterpret_cast<uint4*>(at + dst[j]) = make_uint4(0u, 0u, 0u, 0u);
            }
            // make the generic-proxy writes of A visible to the tensor cores
            bspx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                bspx::mbar_arrive(a_full + sa);
                bspx::mbar_arrive(c_empty + sc);
            }
            if (++sc == (uint32_t)SC) { sc = 0; pc ^= 1u; }
            if (++sa == (uint32_t)SA) { sa = 0; pa ^= 1u; }
        }
    }

    // ---------------- epilogue: warps 4-7, one per TMEM lane quadrant, each
    // thread one row of the 16 columns; then split-K through the workspace
    const bool epi = warp >= DEC0 && warp < DEC0 + 4;
    const int trow = 32 * (warp & 3) + lane;
    const int64_t m = mt * BM + trow;
    float v[BN];
    bool ok = true;
    if (epi) {
        ok = __all_sync(FULL, bspx::mbar_wait_sleep(acc_bar, 0, cap, kSleepNs));
        if (!ok || failed) {
            failed = true;
            ok = false;
        } else {
            tc_fence_after();
            uint32_t r[16];
            tmem_ld16(tmem_base + ((uint32_t)(32 * (warp & 3)) << 16), r);
#pragma unroll
            for (int j = 0; j < BN; ++j) v[j] = __uint_as_float(r[j]);
        }
    }
    const bool mine = epi && ok && m < M;
    if (a.splits == 1) {
        if (mine)
#pragma unroll
            for (int j = 0; j < BN; ++j)
                if (j < N) a.Y[j * M + m] = __float2half_rn(v[j]);
    } else {
        // this split's partial sums: its own slot (deterministic) or an
        // atomic add; the last CTA of the tile to arrive writes Y
        float* det = a.ws_det ? a.ws_det + (int64_t)part * N * M : nullptr;
        if (mine)
#pragma unroll
            for (int j = 0; j < BN; ++j)
                if (j < N) {
                    if (det) det[j * M + m] = v[j];
                    else atomicAdd(a.ws + j * M + m, v[j]);
                }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) *s_last = atomicAdd(a.counters + strip0, 1u) == (uint32_t)(a.splits - 1);
        __syncthreads();
        if (*s_last) {
            __threadfence();
            if (epi && m < M)
                for (int j = 0; j < BN && j < N; ++j) {
                    float t = 0.f;
                    if (a.ws_det) {
                        for (int sp = 0; sp < a.splits; ++sp) t += __ldcg(a.ws_det + ((int64_t)sp * N + j) * M + m);
                    } else {
                        t = atomicExch(a.ws + j * M + m, 0.0f);
                    }
                    a.Y[j * M + m] = __float2half_rn(t);
                }
            if (threadIdx.x == 0) a.counters[strip0] = 0u;
        }
    }

    if (failed && lane == 0) atomicExch(a.err, (int)BSP_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
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

int bsp_narrow_splits_auto(const bsp_decode_problem& p)
{
    // the critical path: CTA waves (MINB CTAs per SM) times the GT columns
    // of a CTA plus a fixed cost per CTA (start, epilogue)
    const int64_t tiles = (p.Mp + BM - 1) / BM, KT = p.Kp / 64;
    const int64_t slots = (p.num_sms > 0 ? p.num_sms : 1) * MINB;
    int64_t best = 1, best_cost = INT64_MAX;
    for (int64_t sp = 1; sp <= KT && sp <= 64; ++sp) {
        const int64_t cost = ((tiles * sp + slots - 1) / slots) * ((KT + sp - 1) / sp + BSP_NARROW_CTA_COST);
        if (cost < best_cost) {
            best_cost = cost;
            best = sp;
        }
    }
    return (int)best;
}

int bsp_narrow_splits(const bsp_decode_problem& p)
{
    const int64_t KT = p.Kp / 64;
    int64_t best = bsp_narrow_splits_auto(p);
    if (const int64_t v = bsp_tune(BSP_TUNE_NARROW_SPLITK)) best = v;  // tests, tuning
    if (best > KT) best = KT;
    if (best < 1) best = 1;
    if (p.ws_det && best > p.det_slots) best = p.det_slots;
    return (int)best;
}

bsp_status_t bsp_run_spmm_narrow(const bsp_decode_problem& p, const void* X, int64_t N, void* Y, cudaStream_t s)
{
    if (p.dtype != BSP_FP16) return BSP_ERR_DTYPE;
    if (N < 1 || N > BN || p.K > (int64_t)0x7FFFFFFF) return BSP_ERR_INVALID_ARG;
    if (p.device < 0 || p.device >= 64) return BSP_ERR_INVALID_ARG;
    auto encode = get_encode_fn();
    if (!encode) return BSP_ERR_CUDA;
    // X: [N][K] fp16, K contiguous; boxes of 64 (K) x 16 rows, 128-B
    // swizzle; rows past N read as zeros
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BSP_ERR_INVALID_ARG;

    static bsp_attr_once attr;
    if (!attr.run(p.device, [] {
            return cudaFuncSetAttribute(spmm_narrow_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
        }))
        return BSP_ERR_CUDA;
    NarrowArgs a = {};
    a.bitmaps = p.bitmaps;
    a.offsets = p.offsets;
    a.values = (const uint8_t*)p.values;
    a.Y = (__half*)Y;
    a.M = p.M;
    a.N = N;
    a.K = p.K;
    a.Mp = p.Mp;
    a.KT = p.Kp / 64;
    a.splits = bsp_narrow_splits(p);
    if (a.splits < 1 || a.splits > a.KT) return BSP_ERR_INTERNAL;  // a split without GT columns
    a.ws = (float*)p.ws;
    a.ws_det = a.splits > 1 ? p.ws_det : nullptr;
    a.counters = p.counters;
    a.ngt = (p.Mp / 64) * (p.Kp / 64);
    a.values_bytes = p.values_bytes;
    a.err = p.err;
    a.spin_cap = bsp_spin_cap();
    // C ring: as many stages as fit, each sized for the densest GT
    a.c_slot = c_slot_bytes(std::min<uint32_t>(p.max_gt_nnz, 4096u));
    a.c_stage = c_stage_bytes(a.c_slot);
    a.sc = std::min<int>(SC_MAX, C_BYTES / (int)a.c_stage);
    const int smem = OFF_C + a.sc * (int)a.c_stage + 1024;
    const int64_t tiles = (p.Mp + BM - 1) / BM;
    const int64_t ctas = tiles * a.splits;
    if (ctas > 0x7FFFFFFF) return BSP_ERR_INVALID_ARG;
    spmm_narrow_kernel<<<(unsigned)ctas, THREADS, smem, s>>>(map, a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}
