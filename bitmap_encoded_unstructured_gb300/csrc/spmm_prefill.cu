// Prefill-path product Y = W * X for N > 16 on the 5th-generation tensor
// cores (tcgen05), fp16 inputs, fp32 accumulation in tensor memory.
//
// Method: "load as sparse, compute as dense" ("Unified Static-Dynamic
// Pruning for Efficient LLM Inference", section 4.3; "SpInfer: How bitmaps
// make sparse LLMs actually fast", sections "Shared Memory Bitmap Decoding
// (SMBD)" and "The async pipeline"): the compressed GroupTiles are streamed
// into shared memory, decoded into a dense fp16 tile there, and that tile
// feeds a dense tensor-core contraction.  Where the pages decode into mma
// register fragments (and SPDP adds a transpose stage), here the decoder
// warps write each 8-element row-byte of a BitmapTile as one 16-byte chunk
// straight into the K-major 128-byte-swizzled shared-memory layout that
// tcgen05.mma reads: a BT row-byte is exactly one swizzle chunk.
//
// CTA tile: 128 rows of W (two GT row strips) x 256 * NSUB columns of Y
// (tokens); one GT column (K = 64) per pipeline step, three rings:
//   C  compressed data  bitmaps + value spans of the two GTs (bulk copies),
//                       the rest of shared memory in stages sized for the
//                       densest GT (up to SC_MAX), producer -> decoders
//   A  decoded W tile   128 x 64 fp16, K-major, SWIZZLE_128B (16 KB),
//                       2 stages, decoders -> MMA
//   B  X sub-tiles      256 x 64 fp16 each, K-major, SWIZZLE_128B (TMA),
//                       4 stages (NSUB per step), producer -> MMA
// each with a "full" and an "empty" mbarrier per stage, so decoding step
// k+1 overlaps the MMAs of step k and the compressed data runs ahead.
// Warp roles (21 warps):
//   warp 0     C producer: bulk copies of the compressed GTs, up to SC
//              steps ahead of the decoders.
//   warp 20    B producer: TMA tensor loads of the X sub-tiles, up to 4
//              ahead of the MMAs (its own warp, so that neither ring waits
//              on the other).
//   warp 1     allocates 256 * NSUB TMEM columns; lane 0 issues NSUB x 4
//              tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16) per
//              step and commits them to the A and B "empty" barriers.
//   warps 2-3  scanners, one per GT: exclusive scan of the BT popcounts
//              (shfl) and per-byte popcounts give the first value index of
//              every BT row; the 512 row starts go into the C stage, then
//              "c_scan".
//   warps 4-19 decoders: eight per GT, each on 16 of its rows and half of
//              its columns; per half row-byte one byte of bitmap, one row
//              start and four predicated shared-memory loads (no branch per
//              position) give 8 bytes of A (with one 256-column sub-tile:
//              per whole row-byte, eight loads give a 16-B chunk); then
//              "a_full" / "c_empty".
//   warps 4-19 after the K loop: epilogue, tcgen05.ld of their TMEM lane
//              quadrant (warp % 4) and a quarter of the columns, fp32 ->
//              fp16, stores to Y[n][m].
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

namespace {

constexpr int BM = 128, BN = 256, BK = 64;    // BN: columns of one MMA / one TMEM accumulator
constexpr int A_BYTES = BM * BK * 2;          // 16384
// Decoder warps: 8 (four per GroupTile, eight half row-bytes per lane and
// step) or 16 (eight per GroupTile, four half row-bytes per lane and step).
#ifndef BSP_PF_DEC_WARPS
#define BSP_PF_DEC_WARPS 16
#endif
constexpr int DEC_WARPS = BSP_PF_DEC_WARPS;
static_assert(DEC_WARPS == 8 || DEC_WARPS == 16, "decoder warps");
constexpr int WPG = DEC_WARPS / 2;   // decoder warps per GroupTile
constexpr int NU = 32 / WPG;         // units (half row-bytes) per lane and step
constexpr int TCW = NU / 2;          // TCTile columns per warp
constexpr int DEC0 = 4;              // first decoder warp (after producer, MMA, 2 scanners)
constexpr int BPROD = DEC0 + DEC_WARPS;  // B (X tile) producer, the last warp
constexpr int WARPS = BPROD + 1;
constexpr int RS_BYTES = 64 * 8 * 2; // row starts of one GT: [BT][row] u16
#ifndef BSP_PF_SLEEP_NS
#define BSP_PF_SLEEP_NS 1000
#endif
constexpr uint32_t kSleepNs = BSP_PF_SLEEP_NS;  // suspend hint of the waiting polls
constexpr int THREADS = WARPS * 32;

// NSUB 256-column sub-tiles of N per CTA, each with its own TMEM
// accumulator: every decoded A tile feeds NSUB x 4 MMAs.
// X sub-tile ring depth with one 256-column sub-tile per CTA
#ifndef BSP_PF1_SB
#define BSP_PF1_SB 3
#endif
constexpr int SC_MAX = 12;        // barrier slots of the C ring
constexpr int SMEM_MAX = 227 * 1024;

// One C stage: two GT slots (512 B of bitmaps, then the 16-B chunks that
// hold the GT's value span), a 16-B header (the value shifts) and the row
// starts of the two GTs.  The slot is sized for the densest GT of the
// matrix, so the number of stages that fit follows the density.
__host__ __device__ constexpr uint32_t c_slot_bytes(uint32_t max_gt_nnz)
{
    return (512u + 16u * ((max_gt_nnz + 7u) / 8u + 1u) + 127u) & ~127u;
}
__host__ __device__ constexpr uint32_t c_stage_bytes(uint32_t slot)
{
    return (2u * slot + 16u + 2u * (uint32_t)RS_BYTES + 127u) & ~127u;
}

template <int NSUB>
struct PCfg {
    static constexpr int BN_CTA = BN * NSUB;
    // three rings with their own depths; the C ring takes the rest of the
    // shared memory, in stages sized at launch
    static constexpr int SB = NSUB == 1 ? BSP_PF1_SB : 4;  // X sub-tiles (TMA) -> MMA
    static constexpr int SA = 2;                             // decoded A tiles   -> MMA
    static constexpr int B_STAGE = BN * BK * 2;       // one sub-tile per stage
    static constexpr int OFF_B = 0;                   // 1024-B aligned regions first
    static constexpr int OFF_A = OFF_B + SB * B_STAGE;
    static constexpr int OFF_BAR = OFF_A + SA * A_BYTES;
    // barriers: c_full[SC_MAX] c_empty[SC_MAX] b_full[SB] b_empty[SB] a_full[SA] a_empty[SA] acc
    // c_scan[SC_MAX]
    static constexpr int NBAR = 3 * SC_MAX + 2 * SB + 2 * SA + 1;
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
    static constexpr int OFF_C = (OFF_TMEM + 16 + 127) & ~127;
    static constexpr int C_BYTES = SMEM_MAX - 1024 - OFF_C;  // 1024: slack to align the base to 1024 B
    static constexpr uint32_t TMEM_COLS = 256 * NSUB;
    static_assert(C_BYTES >= 2 * (int)c_stage_bytes(c_slot_bytes(4096)), "two dense C stages");
    static_assert((B_STAGE % 1024) == 0 && (A_BYTES % 1024) == 0, "swizzle atoms need 1024-B alignment");
};

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled canonical layout: rows of 128 B, 8-row atoms of 1 KB (stride
// 1024 B between atoms), atoms 1024-B aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);        // start address
    d |= (uint64_t)1u << 16;                         // leading offset (unused for swizzled K-major)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;   // stride offset: 1024 B between 8-row atoms
    d |= (uint64_t)1u << 46;                         // descriptor version of sm_100
    d |= (uint64_t)2u << 61;                         // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ int bt_local(int br, int bc)
{
    return (((br >> 1) * 4 + (bc >> 1)) << 2) + (br & 1) + ((bc & 1) << 1);
}

// One position of a row-byte, without a branch: if rbyte & bit, the next
// packed fp16 value (shared-memory byte address `addr`) zero-extended, and
// addr advances by one value; else 0.
__device__ __forceinline__ uint32_t take_f16(uint32_t& addr, uint32_t rbyte, uint32_t bit)
{
    uint32_t v;
    asm(
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

struct PrefillArgs {
    const uint64_t* bitmaps;
    const uint32_t* offsets;
    const uint8_t* values;
    __half* Y;
    int64_t M, N, K;  // logical: Y rows, columns, X row length
    int64_t Mp, KT;   // padded grid: rows (a multiple of 64), GT columns
    int64_t ntiles;   // N tiles of BN * NSUB columns
    uint32_t c_slot, c_stage;  // C ring geometry (bytes): GT slot, stage
    int sc;                    // C stages in use, 2..SC_MAX
    int* err;
    uint32_t spin_cap;
};

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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// KS: split-K over a cluster of two CTAs on one output tile.  Rank 0 takes
// the first ceil(KT / 2) GT columns, rank 1 the rest (at least one: the host
// launches KS only for KT >= 2); each accumulates in its own TMEM, then rank
// 1 stores its fp32 partial tile into rank 0's rings (idle by then) and
// rank 0 writes Y = RN(own + partner).
template <int NSUB, bool KS>
__global__ void __launch_bounds__(THREADS, 1)
spmm_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const PrefillArgs a)
{
    using P = PCfg<NSUB>;
    static_assert(!KS || NSUB == 1, "split-K: one 256-column sub-tile");
    static_assert(!KS || P::OFF_BAR >= BM * BN * 4, "split-K exchange buffer: the rings, below the barriers");
    constexpr int SA = P::SA, SB = P::SB;
    const int SC = a.sc;
    const uint32_t SLOT = a.c_slot, C_HDR = 2 * SLOT, C_RS = C_HDR + 16;
    const uint32_t vchunks = (SLOT - 512) / 16;  // value chunks a slot holds
    constexpr uint32_t TMEM_COLS = P::TMEM_COLS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-B alignment of the shared-window offset (the 128-B swizzle atoms)
    uint8_t* smem = smem_raw + ((1024u - (bspx::smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr uint32_t FULL = 0xFFFFFFFFu;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint64_t* c_full = reinterpret_cast<uint64_t*>(smem + P::OFF_BAR);
    uint64_t* c_empty = c_full + SC_MAX;
    uint64_t* b_full = c_empty + SC_MAX;
    uint64_t* b_empty = b_full + SB;
    uint64_t* a_full = b_empty + SB;
    uint64_t* a_empty = a_full + SA;
    uint64_t* acc_bar = a_empty + SA;
    uint64_t* c_scan = acc_bar + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::OFF_TMEM);
    auto b_stage = [&](int s) { return smem + P::OFF_B + s * P::B_STAGE; };
    auto a_stage = [&](int s) { return smem + P::OFF_A + s * A_BYTES; };
    auto c_stage = [&](int s) { return smem + P::OFF_C + s * a.c_stage; };

    const int64_t M = a.M, N = a.N;
    const uint32_t KTA = (uint32_t)a.KT;                 // GT columns of the grid (row pitch)
    const uint32_t krank = KS ? bspx::cluster_ctarank() : 0u;
    const uint32_t KT0 = KS ? (KTA + 1) / 2 : KTA;
    const uint32_t k0 = krank ? KT0 : 0u;                // first GT column of this CTA
    const uint32_t KT = krank ? KTA - KT0 : KT0;         // GT columns of this CTA
    // linear grid of clusters (one CTA, or the two K halves of one tile), N
    // tiles fastest, so that the CTAs streaming one W row strip run at about
    // the same time and share it in L2
    const int64_t cl = (int64_t)blockIdx.x / (KS ? 2 : 1);
    const int64_t mt = cl / a.ntiles;
    const int64_t n0 = (cl % a.ntiles) * P::BN_CTA;
    const int64_t strip0 = 2 * mt, strip1 = 2 * mt + 1;
    const bool has_b = strip1 * 64 < a.Mp;  // second GT row strip of the tile exists
    const uint32_t cap = a.spin_cap;

    if (warp == 1) {
        // allocate the accumulators: 128 lanes x 256*NSUB fp32 columns
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
        for (int s = 0; s < SC; ++s) bspx::mbar_init(c_scan + s, 2 * 32);  // every scanner lane
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
                offa = (i <= KT) ? __ldg(a.offsets + ta + i) : 0u;
                offb = (has_b && i <= KT) ? __ldg(a.offsets + tb + i) : 0u;
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
        // ---------------- B producer: X sub-tiles by TMA, (step, sub-tile) order,
        // up to SB sub-tiles ahead: a stage frees as soon as the MMAs of its
        // own sub-tile are done, half a step before those of the next one
        uint32_t s = 0, ph = 0;
        uint32_t i = 0;  // sub-tiles issued
        const uint32_t nb = KT * NSUB;
        for (; i < nb; ++i) {
            if (i >= (uint32_t)SB &&
                !__all_sync(FULL, bspx::mbar_wait_sleep(b_empty + s, ph ^ 1u, cap, kSleepNs))) {
                failed = true;
                break;
            }
            if (lane == 0) {
                const uint32_t kx = i / NSUB, u = i % NSUB;
                bspx::mbar_arrive_expect_tx(b_full + s, (uint32_t)P::B_STAGE);
                tma_load_2d(b_stage(s), &tmX, (int)((k0 + kx) * BK), (int)(n0 + u * BN), b_full + s);
            }
            if (++s == (uint32_t)SB) { s = 0; ph ^= 1u; }
        }
        for (uint32_t k = (i > (uint32_t)SB ? i - SB : 0); k < i; ++k)
            bspx::mbar_wait_bounded(b_full + (k % SB), (k / SB) & 1u, cap);
    } else if (warp == 1) {
        // ---------------- MMA issuer
        uint32_t sa = 0, pa = 0, sb = 0, pb = 0;
        for (uint32_t kb = 0; kb < KT && !failed; ++kb) {
            const bool oka = bspx::mbar_wait_sleep(a_full + sa, pa, cap, kSleepNs);
            if (!__all_sync(FULL, oka)) { failed = true; break; }
            const uint64_t ad = smem_desc_sw128(bspx::smem_u32(a_stage(sa)));
#pragma unroll
            for (int u = 0; u < NSUB; ++u) {
                const bool okb = bspx::mbar_wait_sleep(b_full + sb, pb, cap, kSleepNs);
                if (!__all_sync(FULL, okb)) { failed = true; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t bd = smem_desc_sw128(bspx::smem_u32(b_stage(sb)));
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)  // K = 16 per MMA: 32 B along the swizzled row
                        umma_f16(tmem_base + (uint32_t)(u * BN), ad + (uint64_t)(2 * j), bd + (uint64_t)(2 * j),
                                 (kb | j) ? 1u : 0u);
                    umma_commit(b_empty + sb);  // fires once the MMAs above are done
                }
                __syncwarp();
                if (++sb == (uint32_t)SB) { sb = 0; pb ^= 1u; }
            }
            if (failed) break;
            if (lane == 0) umma_commit(a_empty + sa);
            __syncwarp();
            if (++sa == (uint32_t)SA) { sa = 0; pa ^= 1u; }
        }
        if (lane == 0) umma_commit(acc_bar);  // fires once every MMA issued above is done
        __syncwarp();
        bspx::mbar_wait_bounded(acc_bar, 0, cap);
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
            bspx::mbar_arrive(c_scan + sc);  // release: the row starts above
            if (++sc == (uint32_t)SC) { sc = 0; pc ^= 1u; }
        }
    } else {
        // ---------------- decoders
        const int dw = warp - DEC0;
        const int gsel = dw / WPG, wq = dw % WPG;
        const int q = wq / (4 / TCW);             // TCTile row of the warp (16 GT rows)
        const int p0 = (wq % (4 / TCW)) * TCW;    // first TCTile column (octet pair)
        // Unit j of a lane: row 16q + 8 (lane / 16) + lane % 8 of the GT,
        // octet bc = 2 (p0 + j / 2) + j % 2, and of its 8 positions the low
        // (lane bit 3 clear) or the high half.  One unit of a warp thus reads
        // the values of two BTs adjacent in value order (TL and BL, or TR
        // and BR, of one TCTile): about 128 B at 50% density, where whole
        // row-bytes per lane would span four BTs.  Each half-warp writes
        // eight whole 16-B chunks of eight consecutive rows, which the
        // swizzle puts in distinct banks.
        //
        // One 256-column sub-tile (N <= 256): the decode, not shared-memory
        // bandwidth, sets the pace, so each lane takes whole row-bytes
        // instead: row 16q + lane % 16, octet 2 p0 + 2 (lane / 16) + j, its
        // eight positions one 16-B chunk (the same chunk addresses as the
        // two halves above; fewer instructions, loads spanning four BTs).
        constexpr bool FULLROW = NSUB == 1 && DEC_WARPS == 16;
        constexpr int NJ = FULLROW ? 2 : NU;  // row-bytes, or half row-bytes, per lane and step
        const int row = FULLROW ? 16 * q + (lane & 15) : 16 * q + 8 * (lane >> 4) + (lane & 7);  // row in the GT
        const int trow = 64 * gsel + row;                       // row inside the 128-row tile
        const int half = FULLROW ? 0 : (lane >> 3) & 1;
        const uint32_t nsh = 4u * (uint32_t)half;            // the lane's half of the row-byte
        const uint32_t lowm = half ? 0xFu : 0u;              // positions before it
        int ent[NJ];        // BT row entry: 8 g + row % 8 (bitmap byte / row start)
        uint32_t dst[NJ];   // byte offset of the unit's 8 (or 16) bytes in A (128-B swizzle)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int bc = FULLROW ? 2 * p0 + 2 * (lane >> 4) + j : 2 * (p0 + j / 2) + (j & 1);
            ent[j] = 8 * bt_local(row >> 3, bc) + (row & 7);
            dst[j] = (uint32_t)((trow >> 3) * 1024 + (trow & 7) * 128 + ((bc ^ (trow & 7)) << 4) + 8 * half);
        }
        const bool active = gsel == 0 || has_b;
        uint32_t sc = 0, pc = 0, sa = 0, pa = 0;
        for (uint32_t kb = 0; kb < KT; ++kb) {
            // c_scan implies c_full: the scanners arrive only after they saw it
            bool ok = bspx::mbar_wait_sleep(c_scan + sc, pc, cap, kSleepNs);
            if (kb >= (uint32_t)SA) ok = ok && bspx::mbar_wait_sleep(a_empty + sa, pa ^ 1u, cap, kSleepNs);
            if (!__all_sync(FULL, ok)) { failed = true; break; }
            const uint8_t* st = c_stage(sc);
            if (active) {
                const uint8_t* bmb = st + gsel * SLOT;  // bitmap bytes: byte 8 g + r = row r of BT g
                const uint16_t* rst = reinterpret_cast<const uint16_t*>(st + C_RS + gsel * RS_BYTES);
                const uint32_t vbase = bspx::smem_u32(st + gsel * SLOT + 512);
                uint8_t* at = a_stage(sa);
                if constexpr (FULLROW) {
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const uint32_t byte = bmb[ent[j]];
                        uint32_t addr = vbase + 2u * (uint32_t)rst[ent[j]];
                        uint32_t h[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) h[c] = take_f16(addr, byte, 1u << c);
                        *reinterpret_cast<uint4*>(at + dst[j]) = make_uint4(
                            h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const uint32_t byte = bmb[ent[j]];
                        const uint32_t start = (uint32_t)rst[ent[j]] + (uint32_t)__popc(byte & lowm);
                        const uint32_t nib = byte >> nsh;
                        uint32_t addr = vbase + 2u * start;
                        uint32_t h[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) h[c] = take_f16(addr, nib, 1u << c);
                        *reinterpret_cast<uint2*>(at + dst[j]) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
                    }
                }
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
        // ---------------- epilogue: every decoder warp; warp w reads TMEM lane
        // quadrant w % 4 (the lanes a warp may access), and the DEC_WARPS / 4
        // groups of four consecutive warps split the columns (split-K: below)
        if constexpr (!KS) {
            const bool ok = __all_sync(FULL, bspx::mbar_wait_sleep(acc_bar, 0, cap, kSleepNs));
            if (!ok) {
                failed = true;
            } else if (!failed) {
                tc_fence_after();
                constexpr int COLS = P::BN_CTA / (DEC_WARPS / 4);
                const int quad = warp & 3, cg = dw >> 2;  // warps 4-7, 8-11, ...: quadrants 0-3
                const int64_t m = mt * BM + 32 * quad + lane;
#pragma unroll 1
                for (int cb = cg * COLS; cb < (cg + 1) * COLS; cb += 16) {
                    uint32_t r[16];
                    tmem_ld16(tmem_base + ((uint32_t)(32 * quad) << 16) + (uint32_t)cb, r);
                    if (m < M) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int64_t n = n0 + cb + j;
                            if (n < N) a.Y[n * M + m] = __float2half_rn(__uint_as_float(r[j]));
                        }
                    }
                }
            }
        }
    }

    if constexpr (KS) {
        // ---------------- split-K exchange.  First barrier: every role of
        // both CTAs is past its rings, so rank 0's rings are free; the
        // decoder warps (the epilogue threads) have seen their MMAs complete.
        const bool dec = warp >= DEC0 && warp < BPROD;
        bool acc_ok = true;
        if (dec) {
            acc_ok = __all_sync(FULL, bspx::mbar_wait_sleep(acc_bar, 0, cap, kSleepNs));
            if (!acc_ok) failed = true;
        }
        tc_fence_before();
        bspx::cluster_sync();
        // exchange buffer [BN / 4][BM][4] fp32 over the idle rings (X first):
        // lane-consecutive 16-B chunks
        float* xbuf = reinterpret_cast<float*>(smem + P::OFF_B);
        constexpr int COLS = BN / (DEC_WARPS / 4);
        const int quad = warp & 3, cg = (warp - DEC0) >> 2;
        const int trow = 32 * quad + lane;
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * quad) << 16);
        if (dec && krank == 1 && acc_ok) {
            tc_fence_after();
            const uint32_t remote = bspx::mapa_shared(bspx::smem_u32(xbuf), 0);
#pragma unroll 1
            for (int cb = cg * COLS; cb < (cg + 1) * COLS; cb += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + (uint32_t)cb, r);
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    bspx::st_cluster_v4(remote + (uint32_t)((((cb + j) >> 2) * BM + trow) * 16), r[j], r[j + 1],
                                        r[j + 2], r[j + 3]);
            }
        }
        // second barrier: the partner's partial tile is in rank 0's memory
        bspx::cluster_sync();
        if (dec && krank == 0 && acc_ok) {
            tc_fence_after();
            const int64_t m = mt * BM + trow;
#pragma unroll 1
            for (int cb = cg * COLS; cb < (cg + 1) * COLS; cb += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + (uint32_t)cb, r);
                if (m < M) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 q = *reinterpret_cast<const float4*>(xbuf + (((cb + j) >> 2) * BM + trow) * 4);
                        const float pv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int64_t n = n0 + cb + j + e;
                            if (n < N) a.Y[n * M + m] = __float2half_rn(__uint_as_float(r[j + e]) + pv[e]);
                        }
                    }
                }
            }
        }
    }

    if (failed && lane == 0) atomicExch(a.err, (int)BSP_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

namespace {

template <int NSUB, bool KS>
bsp_status_t launch_prefill(const CUtensorMap& map, const PrefillArgs& a0, int64_t M, int64_t N,
                            uint32_t max_gt_nnz, int device, cudaStream_t s)
{
    using P = PCfg<NSUB>;
    static bsp_attr_once attr_once;
    if (!attr_once.run(device, [] {
            return cudaFuncSetAttribute(spmm_prefill_kernel<NSUB, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_MAX);
        }))
        return BSP_ERR_CUDA;
    if (KS && a0.KT < 2) return BSP_ERR_INTERNAL;  // rank 1 would have no GT column
    const int64_t bn_cta = (int64_t)BN * NSUB;
    const int64_t ntiles = (N + bn_cta - 1) / bn_cta;
    const int64_t ctas = ntiles * ((M + BM - 1) / BM) * (KS ? 2 : 1);
    if (ctas > 0x7FFFFFFF) return BSP_ERR_INVALID_ARG;
    PrefillArgs a = a0;
    a.ntiles = ntiles;
    // C ring: as many stages as fit, each sized for the densest GT
    a.c_slot = c_slot_bytes(std::min<uint32_t>(max_gt_nnz, 4096u));
    a.c_stage = c_stage_bytes(a.c_slot);
    a.sc = std::min<int>(SC_MAX, P::C_BYTES / (int)a.c_stage);
    if (const int64_t v = bsp_tune(BSP_TUNE_PREFILL_CSTAGES)) a.sc = std::max(2, std::min<int>(a.sc, (int)v));
    const int smem = P::OFF_C + a.sc * (int)a.c_stage + 1024;
    dim3 grid((unsigned)ctas, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (KS) {  // two consecutive CTAs form a cluster: the two K halves of a tile
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, spmm_prefill_kernel<NSUB, KS>, map, a) == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

}  // namespace

// Split K over two CTAs (N <= 256: one tile column) when that shortens the
// critical path: CTA waves times GT columns per CTA, plus a fixed cost per
// CTA (start, epilogue; about 4 GT columns) and the exchange (about 2).
// BSP_TUNE_PREFILL_KSPLIT = 0 / 1 forces the choice (tests), for KT >= 2.
static bool prefill_split_k(int64_t tiles, int64_t KT, int num_sms)
{
    if (KT < 2) return false;
    if (const int64_t v = bsp_tune(BSP_TUNE_PREFILL_KSPLIT); v >= 0) return v == 1;
    const int64_t slots = num_sms > 0 ? num_sms : 1;  // one CTA per SM (shared memory)
    const int64_t one = ((tiles + slots - 1) / slots) * (KT + 4);
    const int64_t two = ((2 * tiles + slots - 1) / slots) * ((KT + 1) / 2 + 6);
    return two < one;
}

bsp_status_t bsp_run_spmm_prefill(const bsp_decode_problem& p, const void* X, int64_t N, void* Y, cudaStream_t s)
{
    if (p.dtype != BSP_FP16) return BSP_ERR_DTYPE;
    if (N < 1 || N > (int64_t)0x7FFFFFFF || p.K > (int64_t)0x7FFFFFFF) return BSP_ERR_INVALID_ARG;
    auto encode = get_encode_fn();
    if (!encode) return BSP_ERR_CUDA;
    if (p.device < 0 || p.device >= 64) return BSP_ERR_INVALID_ARG;
    // X: [N][K] fp16, K contiguous; box = 64 (K) x 256 (N) rows, with the
    // 128-B swizzle
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BSP_ERR_INVALID_ARG;
    PrefillArgs a;
    a.bitmaps = p.bitmaps;
    a.offsets = p.offsets;
    a.values = (const uint8_t*)p.values;
    a.Y = (__half*)Y;
    a.M = p.M;
    a.N = N;
    a.K = p.K;
    a.Mp = p.Mp;
    a.KT = p.Kp / 64;
    a.err = p.err;
    a.spin_cap = bsp_spin_cap();
    // one 256-column sub-tile per CTA for N <= 256, two (512 columns) above
    if (N > BN) return launch_prefill<2, false>(map, a, p.Mp, N, p.max_gt_nnz, p.device, s);
    if (prefill_split_k(p.Mp / BM + (p.Mp % BM ? 1 : 0), a.KT, p.num_sms))
        return launch_prefill<1, true>(map, a, p.Mp, N, p.max_gt_nnz, p.device, s);
    return launch_prefill<1, false>(map, a, p.Mp, N, p.max_gt_nnz, p.device, s);
}
