// score_tc.cu -- sub-key scores and per-half top-W on the tensor cores (bf16 layers).
//
// Product-key addressing ("Sparse Delta Memory" blog, "Write & Read": two sub-keys ->
// outer sum -> top-k) scores every query half against its sub-key table:
//   s_h[q][i] = <K_h[i], q_h>   for the n rows of K_h, both halves, write and read queries.
// Over all tokens that is a dense GEMM [2*ntok, dk/2] x [dk/2, n] per half, and this
// kernel runs it on the 5th-generation tensor cores:
//  * one CTA per SM works on one half; the half's sub-key table (n <= 512 rows) is
//    loaded once by TMA into shared memory in the 128-byte-swizzled K-major layout the
//    MMA reads, and 128-query tiles stream through two TMA stages;
//  * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M = 128, N = 256
//    twice) into a 512-column TMEM accumulator: row r of the tile in TMEM lane r;
//  * sixteen epilogue warps (four per TMEM lane quadrant, one column group each) keep,
//    per row, the W largest scores by (score desc, row asc), in three passes over TMEM:
//    the row's range, mean and spread; counting passes of six probes narrowing a
//    bracket [lo, hi) of the W-th largest score (the first around mean + z sd -- scores
//    of a row are near normal, z the normal quantile of 1 - W/n -- later ones, run only
//    while a row of the warp keeps too many scores inside its bracket, around the
//    interpolated place of the W-th score and the midpoint of the bracket's order keys);
//    and a pass that writes the scores kept outright and lists the bracket's scores
//    (with their columns) in shared memory, where each thread ranks its own entries
//    against the row's list to find the W-th largest, t. The kept bracket scores are
//    then written from the list: those above t, then those equal to t by ascending row.
// The per-half lists are written in ascending row order among equal scores; the
// candidate kernel sorts them by score.
// Every wait is bounded (status SDM_ETIMEOUT); on time-out a role stops issuing, the
// CTA waits (bounded) for its copies and MMAs in flight and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kTileM = 128;               // queries per tile
constexpr int kKAtom = 64;                // bf16 elements per 128-byte swizzle row
constexpr int kBRows = 512;               // sub-key rows staged (n padded)
constexpr int kTmemCols = 512;
constexpr int kEpiWarps = 16;             // four per TMEM lane quadrant, one column group each
constexpr int kThreads = 32 * (2 + kEpiWarps);  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr uint32_t kBBytes = kBRows * 128 * 2;        // two K atoms of 512 rows
constexpr uint32_t kABytes = kTileM * 128 * 2;        // two K atoms of 128 rows
// Top-W epilogue: probes a counting pass, their places around the expected W-th score in
// rows (multiples of dz), and the capacity of a row's list of the scores inside its final
// bracket (odd: the rows of a warp hit different banks)
constexpr int kProbes = 6;
constexpr int kLCap = 31;
// Counting passes at most: each pass at least halves a bracket's order-key range, so
// real scores need far fewer. A row still over the list capacity after them (reached
// only by constructed scores) keeps its ties at lo, possibly fewer than W, and the
// kernel reports SDM_EUNSUPPORTED.
constexpr int kMaxPasses = 40;
__constant__ float kProbeAt[kProbes] = {-35.f, -15.f, -7.f, 7.f, 15.f, 35.f};
// exchange area after the barriers and the TMEM address: the bracket lists [128][kLCap]
// of scores (the row statistics of the first pass alias their start) and of their
// columns, probe counts [kProbes][512] (the emission counts alias the first two), list
// sizes [512], counts of scores kept outright [512], W-th scores [128]
constexpr uint32_t kXBytes = 128 * kLCap * (4 + 2) + kProbes * 512 * 2 + 2 * 512 * 2 + 128 * 4;

struct ScoreArgs {
    int ntok, n, khalf, W, tiles_per_kind, ctas_per_half;
    int rep;               // 1: a tile holds 128 queries; 4: 32 queries, each in all four
                           // TMEM lane quadrants, so all 16 epilogue warps share its rows
    int qrows;             // queries a tile: 128 / rep
    float z;               // standard normal quantile of 1 - W/n (bracket of the W-th score)
    float dz;              // 1 / (n phi(z)): standard deviations a score a row apart near z
    float* hv;
    int32_t* hi;
    int* status;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// the mbarrier arrives once every MMA this thread issued so far has completed
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void bar_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// barrier over n threads that also returns whether `ok` holds in all of them
__device__ __forceinline__ bool bar_all(int id, int n, bool ok)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout
// (8-row groups of 1024 bytes, rows of 128 bytes), start address 16-byte units.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Order-preserving integer image of an fp32 score (larger score, larger key; -0 folds
// to +0). Every real score maps to a key >= 0x007FFFFF, so 0 marks padding columns.
__device__ __forceinline__ uint32_t order_key(uint32_t bits)
{
    const uint32_t u = __float_as_uint(__uint_as_float(bits) + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_score(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ------------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kThreads, 1) score_tc_kernel(
    const __grid_constant__ CUtensorMap map_qw, const __grid_constant__ CUtensorMap map_qr,
    const __grid_constant__ CUtensorMap map_k1, const __grid_constant__ CUtensorMap map_k2,
    ScoreArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base for the swizzled operands
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sp = smem_raw + (base - raw);
    const uint32_t sB = base, sA0 = base + kBBytes, sA1 = base + kBBytes + kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sp + kBBytes + 2 * kABytes);
    // bars: 0 B loaded, 1..2 A stage full, 3..4 A stage empty, 5 TMEM full, 6 TMEM empty
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
    // exchange between the epilogue warps sharing rows; per-thread slots [quadrant][group][lane]
    float* xl = reinterpret_cast<float*>(tmem_slot + 4);   // [row slot][kLCap] bracket lists
    float* xfmin = xl;                                     // [512] each: row minimum, maximum,
    float* xfmax = xl + 512;                               // sum and sum of squares (first pass)
    float* xs = xl + 1024;
    float* xs2 = xl + 1536;
    unsigned short* xlc = reinterpret_cast<unsigned short*>(xl + 128 * kLCap);  // [row slot][kLCap]
    unsigned short* xpb = xlc + 128 * kLCap;               // [kProbes][512]
    unsigned short* xa = xpb;                              // [512] emission counts: kept, ties
    unsigned short* xt = xpb + 512;
    unsigned short* xln = xpb + kProbes * 512;             // [512] list entries a thread
    unsigned short* xab = xln + 512;                       // [512] scores kept outright
    float* xtr = reinterpret_cast<float*>(xab + 512);      // [row slot] W-th score
    __shared__ int dead;                 // a role gave up: the others stop at their next wait

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x / a.ctas_per_half;
    const int cta = blockIdx.x % a.ctas_per_half;
    const int ntiles = 2 * a.tiles_per_kind;
    const int my_tiles = cta < ntiles ? (ntiles - cta + a.ctas_per_half - 1) / a.ctas_per_half : 0;
    const int NP = (a.n + 15) & ~15;     // MMA N over all chunks
    const int katoms = a.khalf / kKAtom;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bars + 0), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(bars + 1 + s), 1);
            mbar_init(smem_u32(bars + 3 + s), 1);
        }
        mbar_init(smem_u32(bars + 5), 1);
        mbar_init(smem_u32(bars + 6), kEpiWarps);
        dead = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int* stat = a.status;
    auto waitb = [&](uint32_t bar, uint32_t parity) -> bool {
        // bounded, and gives up early once another role has given up
        if (mbar_try_wait(bar, parity))
            return true;
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, parity)) {
            if (*(volatile int*)&dead)
                return false;
            if (clock64() - t0 > kSpinLimitCycles) {
                report(stat, SDM_ETIMEOUT);
                *(volatile int*)&dead = 1;
                return false;
            }
        }
        return true;
    };

    if (warp == 0) {
        // ---------------- TMA producer: the sub-key table once, then query tiles
        if (lane == 0 && my_tiles > 0) {
            const CUtensorMap* mk = half ? &map_k2 : &map_k1;
            const uint32_t bB = smem_u32(bars + 0);
            mbar_arrive_expect_tx(bB, (uint32_t)katoms * 2 * 256 * 128);
            for (int kb = 0; kb < katoms; ++kb)
                for (int nc = 0; nc < 2; ++nc)
                    tma_load_2d(sB + kb * (kBBytes / 2) + nc * 256 * 128, mk, kb * kKAtom, nc * 256, bB);
            int armed[2] = {-1, -1};
            for (int i = 0; i < my_tiles; ++i) {
                const int s = i & 1;
                if (i >= 2 && !waitb(smem_u32(bars + 3 + s), ((i - 2) >> 1) & 1))
                    break;
                const int tl = cta + i * a.ctas_per_half;
                const int kind = tl / a.tiles_per_kind;
                const int row0 = (tl % a.tiles_per_kind) * a.qrows;
                const CUtensorMap* mq = kind ? &map_qr : &map_qw;
                const uint32_t fb = smem_u32(bars + 1 + s);
                const uint32_t dst = s ? sA1 : sA0;
                mbar_arrive_expect_tx(fb, (uint32_t)katoms * kTileM * 128);
                // (the 1024-byte swizzle period divides a 32-row slice, so slices of
                // a replicated tile land exactly as rows of a full one would)
                for (int kb = 0; kb < katoms; ++kb)
                    for (int r = 0; r < a.rep; ++r)
                        tma_load_2d(dst + kb * (kABytes / 2) + r * a.qrows * 128, mq,
                                    half * a.khalf + kb * kKAtom, row0, fb);
                armed[s] = i;
            }
            // copies in flight land before the CTA may end
            mbar_wait(bB, 0, nullptr, stat);
            for (int s = 0; s < 2; ++s)
                if (armed[s] >= 0)
                    mbar_wait(smem_u32(bars + 1 + s), (armed[s] >> 1) & 1, nullptr, stat);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0 && my_tiles > 0) {
            bool ok = waitb(smem_u32(bars + 0), 0);
            int issued = -1;
            for (int i = 0; ok && i < my_tiles; ++i) {
                const int s = i & 1;
                ok = waitb(smem_u32(bars + 1 + s), (i >> 1) & 1);
                // the accumulator is free once the epilogue has read the previous tile
                if (ok && i >= 1)
                    ok = waitb(smem_u32(bars + 6), (i - 1) & 1);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t aBase = s ? sA1 : sA0;
                for (int nc = 0; nc * 256 < NP; ++nc) {
                    const int N = min(256, NP - nc * 256);
                    const uint32_t idesc = idesc_bf16(kTileM, N);
                    for (int kb = 0; kb < katoms; ++kb)
                        for (int kk = 0; kk < kKAtom / 16; ++kk) {
                            const uint64_t ad = sw128_desc(aBase + kb * (kABytes / 2) + kk * 32);
                            const uint64_t bd =
                                sw128_desc(sB + kb * (kBBytes / 2) + nc * 256 * 128 + kk * 32);
                            tc_mma(tmem + nc * 256, ad, bd, idesc, (kb | kk) ? 1u : 0u);
                        }
                }
                tc_commit(smem_u32(bars + 3 + s));   // the A stage may be refilled
                tc_commit(smem_u32(bars + 5));       // the scores are in TMEM
                issued = i;
            }
            // MMAs in flight complete before TMEM is freed
            if (issued >= 0)
                mbar_wait(smem_u32(bars + 5), issued & 1, nullptr, stat);
        }
    } else {
        // ---------------- epilogue: per-row top-W of the scores. Warp e = warp - 2 reads
        // TMEM lane quadrant q = warp % 4 (the quadrant a warp may access). With 128
        // queries a tile, the four warps of a quadrant share its 32 rows, one column group
        // g = e / 4 each, and add up their counts per row through shared memory at a
        // named barrier (id 1 + q, 128 threads). With replicated queries every quadrant
        // holds the same 32 rows, and all 16 warps share them, column group g = e, at one
        // barrier of 512 threads. The warps at a barrier run the same number of rounds
        // (same rows, same totals) and leave together, so none can be left waiting.
        const int q = warp & 3;
        const int G = a.rep == 1 ? 4 : 16;                          // column groups a row
        const int g = a.rep == 1 ? (warp - 2) >> 2 : warp - 2;
        const int xs0 = a.rep == 1 ? q : 0;                         // exchange block
        const int bid = a.rep == 1 ? 1 + q : 1;
        const int bn = 32 * G;                                      // threads at the barrier
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
        const int W = a.W;
        const int CW = ((NP + G * 32 - 1) / (G * 32)) * 32;         // columns a group reads
        const int cb = min(NP, g * CW), ce = min(NP, cb + CW);
        const int xi = (xs0 * G + g) * 32 + lane;                   // own exchange slot
        const int xq = xs0 * G * 32 + lane;                         // group 0 of this lane
        for (int i = 0; i < my_tiles; ++i) {
            const bool got = waitb(smem_u32(bars + 5), i & 1);
            if (!bar_all(bid, bn, got))
                break;
            tc_fence_after();
            const int tl = cta + i * a.ctas_per_half;
            const int kind = tl / a.tiles_per_kind;
            const int tok = (tl % a.tiles_per_kind) * a.qrows + (a.rep == 1 ? q * 32 : 0) + lane;
            uint32_t v[32];
            const int nv_own = max(0, min(ce, a.n) - cb);          // valid columns here
            // 32 columns into v; in a chunk past the n-th column, -inf in the columns
            // beyond it, below every probe and threshold
            auto load = [&](int c0) {
                tmem_ld32(trow + c0, v);
                if (c0 + 32 > a.n) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j >= a.n)
                            v[j] = 0xFF800000u;
                }
            };
            // the row's range, mean and spread
            float fmn = INFINITY, fmx = -INFINITY, sum = 0.f, sum2 = 0.f;
            for (int c0 = cb; c0 < ce; c0 += 32) {
                tmem_ld32(trow + c0, v);
                if (c0 + 32 <= a.n) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = __uint_as_float(v[j]);
                        fmn = fminf(fmn, f);
                        fmx = fmaxf(fmx, f);
                        sum += f;
                        sum2 = fmaf(f, f, sum2);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < a.n) {
                            const float f = __uint_as_float(v[j]);
                            fmn = fminf(fmn, f);
                            fmx = fmaxf(fmx, f);
                            sum += f;
                            sum2 = fmaf(f, f, sum2);
                        }
                    }
                }
            }
            xfmin[xi] = fmn;
            xfmax[xi] = fmx;
            xs[xi] = sum;
            xs2[xi] = sum2;
            bar_sync(bid, bn);
            sum = 0.f;
            sum2 = 0.f;
            for (int h = 0; h < G; ++h) {
                fmn = fminf(fmn, xfmin[xq + h * 32]);
                fmx = fmaxf(fmx, xfmax[xq + h * 32]);
                sum += xs[xq + h * 32];
                sum2 += xs2[xq + h * 32];
            }
            // Bracket [lo, hi) of the W-th largest score: c_lo >= W scores lie at or above
            // lo (o_lo of them in this thread's columns), c_hi < W at or above hi (o_hi);
            // exact: exactly W at or above lo. Counting passes narrow it with kProbes probes
            // each: the first around mean + z sd (scores of a row are near normal), later
            // ones around the interpolated place of the W-th score inside the bracket, one
            // of them the midpoint of the bracket's order keys, which at least halves it.
            // The passes end once every row of the warp's rows has exactly W, a bracket of
            // one value, or at most kLCap scores inside its bracket.
            float lo = fmn, hi = INFINITY;
            int c_lo = a.n, c_hi = 0, o_lo = nv_own, o_hi = 0;
            bool exact = false;
            float pr[kProbes];
            {
                const float mean = sum / a.n;
                const float sd = sqrtf(fmaxf(sum2 / a.n - mean * mean, 0.f));
#pragma unroll
                for (int k = 0; k < kProbes; ++k)
                    pr[k] = mean + (a.z + a.dz * kProbeAt[k]) * sd;
            }
            for (int pass = 0;; ++pass) {
                unsigned short* xp = xpb;
                if (pass > 0)
                    bar_sync(bid, bn);   // everyone has read the previous pass's counts
                // (counted in floats, exact here: the additions go to the FMA pipe, the
                // comparisons to the ALU pipe)
                float cf[kProbes];
#pragma unroll
                for (int k = 0; k < kProbes; ++k)
                    cf[k] = 0.f;
                for (int c0 = cb; c0 < ce; c0 += 32) {
                    load(c0);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = __uint_as_float(v[j]);
#pragma unroll
                        for (int k = 0; k < kProbes; ++k)
                            cf[k] += f >= pr[k] ? 1.f : 0.f;
                    }
                }
                int cp[kProbes];
#pragma unroll
                for (int k = 0; k < kProbes; ++k) {
                    cp[k] = (int)cf[k];
                    xp[k * 512 + xi] = (unsigned short)cp[k];
                }
                bar_sync(bid, bn);
#pragma unroll
                for (int k = 0; k < kProbes; ++k) {
                    int c = 0;
                    for (int h = 0; h < G; ++h)
                        c += xp[k * 512 + xq + h * 32];
                    if (!exact && pr[k] > lo && pr[k] < hi) {
                        if (c >= W) {
                            lo = pr[k];
                            c_lo = c;
                            o_lo = cp[k];
                            exact = c == W;
                        } else {
                            hi = pr[k];
                            c_hi = c;
                            o_hi = cp[k];
                        }
                    }
                }
                const uint32_t klo = order_key(__float_as_uint(lo));
                const uint32_t khi = hi < INFINITY ? order_key(__float_as_uint(hi))
                                                   : order_key(__float_as_uint(fmx)) + 1u;
                // one value in the bracket: no float strictly between lo and its top
                const bool single =
                    !(nextafterf(lo, INFINITY) < (hi < INFINITY ? hi : nextafterf(fmx, INFINITY)));
                const bool over = !exact && !single && c_lo - c_hi > kLCap;
                // (the same rows in every warp at this barrier: all leave together)
                if (!__any_sync(0xFFFFFFFFu, over))
                    break;
                if (pass + 1 >= kMaxPasses) {
                    if (over)
                        report(stat, SDM_EUNSUPPORTED);
                    break;
                }
                const float top = hi < INFINITY ? hi : fmx;
                const float step = (top - lo) / (float)(c_lo - c_hi);
                const float est = top - step * ((float)(W - c_hi) - 0.5f);
                // the midpoint of the bracket's order keys (-0 and +0 share a key: where the
                // midpoint's float is not strictly inside, the float just above lo is)
                pr[0] = key_to_score(klo + ((khi - klo) >> 1));
                if (!(pr[0] > lo && pr[0] < hi))
                    pr[0] = nextafterf(lo, INFINITY);
#pragma unroll
                for (int k = 1; k < kProbes; ++k)
                    pr[k] = est + step * (0.25f * kProbeAt[k]);
            }
            // The W-th largest score t. Keep: ex ? scores >= t : scores > t, and then the
            // lowest-numbered rows among the scores equal to t up to W in all (ties are
            // taken in column order, so a group takes ties only after lower columns' groups).
            const bool single_v =
                !(nextafterf(lo, INFINITY) < (hi < INFINITY ? hi : nextafterf(fmx, INFINITY)));
            // rank inside the bracket's list (a row left over the capacity after the last
            // pass keeps ties at lo instead)
            const bool listed = !exact && !single_v && c_lo - c_hi <= kLCap;
            const int m = c_lo - c_hi;
            // Scores at or above ta are kept outright: all of the row's W when exact (ta =
            // lo), else those at or above hi. The list pass writes them out (after the
            // kept scores of lower groups: ab of them here) and lists the bracket's.
            const float ta = exact ? lo : hi;
            const int ab = exact ? o_lo : o_hi;
            xln[xi] = (unsigned short)(listed ? o_lo - o_hi : 0);
            xab[xi] = (unsigned short)ab;
            bar_sync(bid, bn);
            int off = 0, pre_ab = 0;
            for (int h = 0; h < g; ++h) {
                off += xln[xq + h * 32];
                pre_ab += xab[xq + h * 32];
            }
            const int rslot = xs0 * 32 + lane;
            float* L = xl + (size_t)rslot * kLCap;
            unsigned short* Lc = xlc + (size_t)rslot * kLCap;
            const int own_end = off + (listed ? o_lo - o_hi : 0);
            const size_t ob = (((size_t)kind * a.ntok + tok) * 2 + half) * W;
            const int pmax = tok < a.ntok ? W : 0;
            float* hv_row = a.hv + ob;
            int32_t* hi_row = a.hi + ob;
            {
                // scores kept outright to the output, in column order; the bracket's into
                // this group's run of the list (own_end = off where the row has no list)
                int e = off, pos = pre_ab;
                for (int c0 = cb; c0 < ce; c0 += 32) {
                    load(c0);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = __uint_as_float(v[j]);
                        if (f >= lo) {
                            if (f >= ta) {
                                if (pos < pmax) {
                                    hv_row[pos] = f + 0.0f;   // (-0 as +0)
                                    hi_row[pos] = c0 + j;
                                }
                                ++pos;
                            } else {
                                if (e < own_end) {
                                    L[e] = f;
                                    Lc[e] = (unsigned short)(c0 + j);
                                }
                                ++e;
                            }
                        }
                    }
                }
            }
            bar_sync(bid, bn);
            const int need_b = W - c_hi;    // scores to take from inside the bracket
            if (listed) {
                // t is the listed score with fewer than need_b listed above it and at
                // least need_b at or above it
                for (int e = off; e < own_end; ++e) {
                    const float x = L[e];
                    int gt = 0, ge = 0;
                    for (int e2 = 0; e2 < m; ++e2) {
                        const float y = L[e2];
                        gt += y > x ? 1 : 0;
                        ge += y >= x ? 1 : 0;
                    }
                    if (gt < need_b && need_b <= ge)
                        xtr[rslot] = x;
                }
            }
            bar_sync(bid, bn);
            // Inside the bracket: kept outright ka (ex ? scores >= t : scores > t), ties kt
            // (scores equal to t, taken by ascending row up to W in all). A row with one
            // value in its bracket (not listed) keeps ties of lo.
            float t = lo;
            bool ex = exact;
            int ka = 0, kt = 0, cnt_above = c_hi;
            if (exact) {
                cnt_above = W;
            } else if (!listed) {
                kt = o_lo - o_hi;
            } else {
                t = xtr[rslot];
                int gt = 0, ge = 0, og = 0, oe = 0;
                for (int e2 = 0; e2 < m; ++e2) {
                    const float y = L[e2];
                    gt += y > t ? 1 : 0;
                    ge += y >= t ? 1 : 0;
                }
                for (int e = off; e < own_end; ++e) {
                    og += L[e] > t ? 1 : 0;
                    oe += L[e] == t ? 1 : 0;
                }
                ex = c_hi + ge == W;
                ka = ex ? og + oe : og;
                kt = ex ? 0 : oe;
                cnt_above = c_hi + gt;
            }
            xa[xi] = (unsigned short)ka;
            xt[xi] = (unsigned short)kt;
            bar_sync(bid, bn);
            int pre_a = 0, pre_t = 0;
            for (int h = 0; h < g; ++h) {
                pre_a += xa[xq + h * 32];
                pre_t += xt[xq + h * 32];
            }
            const int need = ex ? 0 : W - cnt_above;
            // after the c_hi outright scores of the row (the list pass wrote them)
            int pos = c_hi + pre_a + min(pre_t, need);
            const int allow = max(0, min(kt, need - pre_t));
            int ties = 0;
            if (listed) {
                // this group's kept bracket scores from its run of the list, column order
                for (int e = off; e < own_end; ++e) {
                    const float f = L[e];
                    const bool keep = ex ? f >= t : f > t;
                    const bool tie = !keep && f == t && ties < allow;
                    if (keep || tie) {
                        ties += tie ? 1 : 0;
                        if (pos < pmax) {
                            hv_row[pos] = f + 0.0f;
                            hi_row[pos] = Lc[e];
                        }
                        ++pos;
                    }
                }
            }
            if (__any_sync(0xFFFFFFFFu, !exact && !listed)) {
                // rows whose bracket holds one value: its first ties by column order
                // (rare: rows of equal scores, such as the zero queries of a last tile's
                // rows past the tokens)
                for (int c0 = cb; c0 < ce; c0 += 32) {
                    load(c0);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = __uint_as_float(v[j]);
                        if (!exact && !listed && f == lo && ties < allow) {
                            ++ties;
                            if (pos < pmax) {
                                hv_row[pos] = f + 0.0f;
                                hi_row[pos] = c0 + j;
                            }
                            ++pos;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(bars + 6));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
}

// ------------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D bf16 row-major tensor [rows, cols], box {64 columns, box_rows}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    auto enc = encode_fn();
    if (enc == nullptr)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKAtom, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// z with P(Z > z) = p for a standard normal Z: bisection on the upper tail
// 0.5 erfc(z / sqrt 2), which falls as z grows. Only a starting bracket for an exact
// search, so a float is plenty.
float normal_upper_quantile(double p)
{
    if (p <= 0.0 || p >= 1.0)
        return 0.0f;
    double lo = -10.0, hi = 10.0;
    for (int i = 0; i < 60; ++i) {
        const double mid = 0.5 * (lo + hi);
        if (0.5 * std::erfc(mid / std::sqrt(2.0)) > p)
            lo = mid;
        else
            hi = mid;
    }
    return (float)(0.5 * (lo + hi));
}


bool score_tc_supported(const sdm_cfg& c)
{
    const int h = c.dk / 2;
    return c.dtype == SDM_BF16 && (h == 64 || h == 128) && c.n_sub <= kBRows && c.w <= 64 &&
           encode_fn() != nullptr;
}

cudaError_t launch_score_tc(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                            const void* q_r, int64_t ntok, float* hv, int32_t* hi, int* status,
                            cudaStream_t s)
{
    if (ntok <= 0)
        return cudaSuccess;
    const int h = c.dk / 2;
    // Replicated queries when the tiles of 128 would leave most SMs idle: four times the
    // CTAs, a quarter of the columns per epilogue thread.
    const int sms = num_sms_current_device();
    const int64_t full_tiles = 2 * 2 * ((ntok + kTileM - 1) / kTileM);
    const int rep_ = full_tiles * 2 < sms ? 4 : 1;
    const int qrows = kTileM / rep_;
    CUtensorMap mqw, mqr, mk1, mk2;
    if (!make_map(&mqw, q_w, (uint64_t)c.dk, (uint64_t)ntok, (uint32_t)qrows) ||
        !make_map(&mqr, q_r, (uint64_t)c.dk, (uint64_t)ntok, (uint32_t)qrows) ||
        !make_map(&mk1, K1, (uint64_t)h, (uint64_t)c.n_sub, 256) ||
        !make_map(&mk2, K2, (uint64_t)h, (uint64_t)c.n_sub, 256))
        return cudaErrorInvalidValue;
    ScoreArgs a;
    a.ntok = (int)ntok;
    a.n = c.n_sub;
    a.khalf = h;
    a.W = c.w;
    a.z = normal_upper_quantile((double)c.w / c.n_sub);
    a.dz = (float)(1.0 / (c.n_sub * std::exp(-0.5 * (double)a.z * a.z) / std::sqrt(2.0 * M_PI)));
    a.rep = rep_;
    a.qrows = qrows;
    a.tiles_per_kind = (int)((ntok + qrows - 1) / qrows);
    int per_half = sms / 2;
    if (per_half > 2 * a.tiles_per_kind)
        per_half = 2 * a.tiles_per_kind;
    if (per_half < 1)
        per_half = 1;
    a.ctas_per_half = per_half;
    a.hv = hv;
    a.hi = hi;
    a.status = status;
    const size_t smem = 1024 + kBBytes + 2 * kABytes + 8 * sizeof(uint64_t) + 16 + kXBytes;
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    score_tc_kernel<<<2 * per_half, kThreads, smem, s>>>(mqw, mqr, mk1, mk2, a);
    return cudaGetLastError();
}

}  // namespace sdm
