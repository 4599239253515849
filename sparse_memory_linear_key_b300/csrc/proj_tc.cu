// proj_tc.cu -- step P, the three projections of every token ("Sparse Delta Memory" blog,
// "Write & Read": the token embedding is projected to write keys; a separate query
// projection selects the read slots):
//   q_w = x W_qw [ntok, dk],  q_r = x W_qr [ntok, dk],  v = x W_v [ntok, d]
// fp32 accumulation, rounded once to the I/O type.
//
// bf16 layers run on the 5th-generation tensor cores, one launch for all three products:
//  * tiles of 128 tokens x 256 output columns of one product; x tiles are K-major
//    (token rows), weight tiles N-major (W is stored [d, n], n contiguous), both staged
//    by TMA in the 128-byte swizzle the MMA reads, four stages of 64 K-columns deep;
//  * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M = 128, N = 256,
//    B transposed) into a TMEM accumulator; four epilogue warps read it back with
//    tcgen05.ld (one token row per thread), round to bf16 and store;
//  * a persistent kernel, one CTA per SM walking the tiles, two TMEM accumulators so
//    that a tile's epilogue overlaps the next tile's MMAs, every tile over the whole K
//    (one accumulation order, so the same shape always gives the same bits);
//  * many tokens (prefill): tiles of 256 output columns, four 48 KB stages;
//  * few tokens (decode), where 256-column tiles would leave most SMs idle: tiles of 64
//    columns, eight 24 KB stages, and each tile split along K over a cluster of two
//    CTAs (64 tokens, d = 2048, dk = 256: 40 tiles, 80 CTAs). Rows [r R, (r+1) R)
//    of a tile belong to rank r: once its MMAs are done, each CTA puts the rows of its
//    fp32 partial that others own into its own shared memory and sends each owner its
//    rows with one bulk copy into a receive buffer of the owner's (no partial ever
//    lands on memory its owner still uses), and each owner sums its rows over the
//    ranks in rank order (the same shape always gives the same bits).
// fp32 layers (exact fp32 products are wanted there, which the tensor cores' tf32 path
// does not give) use a tiled SIMT fp32 GEMM.
// Every wait is bounded (status SDM_ETIMEOUT); on time-out a role stops, the CTA waits
// (bounded) for its copies and MMAs in flight and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kBM = 128;                 // tokens a tile (TMEM lanes)
constexpr int kBK = 64;                  // K columns a stage: one 128-byte swizzle row
constexpr uint32_t kAStage = kBM * kBK * 2;            // 16 KB
constexpr uint32_t kBChunk = kBK * 64 * 2;             // 64 K-rows x 64 columns: 8 KB
constexpr uint32_t kStageBudget = 192 * 1024;          // shared memory for the stages
constexpr int kThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
// CTAs of a cluster sharing a 64-column tile: two, so that the projections of a decode
// step (40 tiles, 80 CTAs) leave room for the addressing kernel's 64 CTAs, which launch
// while the projections run and stage their sub-key tables
constexpr int kMaxSplit = 2;
constexpr int kXStride = 64 + 4;         // fp32 per partial row in an exchange buffer
constexpr uint32_t kXRow = kXStride * 4; // bytes of that row (a multiple of 16)
// receive buffers: (split - 1) sources x the rows one rank owns
constexpr uint32_t kRecvBytes = (kMaxSplit - 1) * ((kBM + kMaxSplit - 1) / kMaxSplit) * kXRow;

// A tile of BN output columns (the MMA's N): the stage holds the x tile and BN / 64
// weight chunks; as many stages as the budget takes.
template <int BN>
struct Tile {
    static constexpr uint32_t kBStage = kBChunk * (BN / 64);
    static constexpr uint32_t kStageBytes = kAStage + kBStage;
    static constexpr int kStages = (int)(kStageBudget / kStageBytes);
    static constexpr uint32_t kTmemCols = 2 * BN;      // two accumulators
};

struct ProjMat {
    void* out;      // [M, n] bf16
    int n;          // output columns
    int ntiles;     // ceil(n / BN)
};

struct ProjArgs {
    ProjMat mat[3];
    int M, K, kblocks, mtiles, tiles;
    int abox;       // token rows an x copy brings (all kBM once there are that many tokens)
    int split;      // CTAs per tile (a cluster along K; 64-column tiles only), else 1
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

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
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

// Shared-memory matrix descriptor, 128-byte swizzle. K-major operand (x): rows of 128
// bytes (64 K-columns), 8-row groups 1024 bytes apart (stride offset); the leading offset
// is unused. N-major operand (W): each 64-column chunk holds one 128-byte row per K-row,
// 8-K-row groups 1024 bytes apart (stride offset), chunks kBChunk bytes apart (leading
// offset).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;       // leading byte offset
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16, bf16 A (K-major) and B (N-major: transposed), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_bt(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// bulk copy from this CTA's shared memory into another CTA's of the cluster, completing
// on that CTA's barrier
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// tile t -> product j, its column tile and its token tile. 256-column tiles: the column
// tiles of all three products innermost, so that the CTAs working at one time share each
// x tile (read from DRAM once instead of once a column tile: at 4 x 4,096 tokens, d =
// 2048, 137 -> 127 us a launch from a cold L2; 2 x 16,384 tokens, d = 3840, 915 -> 726 us).
// 64-column tiles (few tokens): token tiles innermost.
template <int BN>
__device__ __forceinline__ void tile_coords(const ProjArgs& a, int t, int& j, int& n0, int& m0)
{
    if (BN == 256) {
        const int per = a.mat[0].ntiles + a.mat[1].ntiles + a.mat[2].ntiles;
        m0 = (t / per) * kBM;
        int c = t % per;
        j = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (c >= a.mat[j].ntiles) {
                c -= a.mat[j].ntiles;
                ++j;
            }
        }
        n0 = c * BN;
        return;
    }
    j = 0;
    int rem = t;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int cnt = a.mtiles * a.mat[j].ntiles;
        if (rem >= cnt) {
            rem -= cnt;
            ++j;
        }
    }
    n0 = (rem / a.mtiles) * BN;
    m0 = (rem % a.mtiles) * kBM;
}

// ------------------------------------------------------------------------ kernel

// split == 1: CTA b takes tiles b, b + grid, ... over the whole K, two accumulators.
// split > 1 (BN = 64): rank r of cluster c takes tile c over its share of the K blocks,
// one accumulator, then the cluster exchanges and sums the partials.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1) proj_tc_kernel(
    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w0,
    const __grid_constant__ CUtensorMap map_w1, const __grid_constant__ CUtensorMap map_w2,
    ProjArgs a)
{
    using TL = Tile<BN>;
    constexpr int kStages = TL::kStages;
    constexpr uint32_t kStageBytes = TL::kStageBytes;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sp = smem_raw + (base - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sp + kStages * kStageBytes);
    // bars: [0, S) full, [S, 2S) empty, 2S + {0, 1} accumulator full, 2S + {2, 3} empty
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    uint64_t* rx = bars + 2 * kStages + 6;             // partials received (split > 1)
    unsigned char* recv = sp + kStages * kStageBytes + (2 * kStages + 8) * 8;   // 16-aligned
    __shared__ int dead;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool split = BN == 64 && a.split > 1;
    const uint32_t rank = split ? cluster_rank() : 0u;
    const int first_tile = split ? (int)(blockIdx.x / a.split) : (int)blockIdx.x;
    const int tile_step = split ? a.tiles : (int)gridDim.x;      // split: one tile a cluster
    const int kb0 = split ? (int)((long long)a.kblocks * rank / a.split) : 0;
    const int kb1 = split ? (int)((long long)a.kblocks * (rank + 1) / a.split) : a.kblocks;
    constexpr int naccs = 2;
    constexpr uint32_t tmem_cols = TL::kTmemCols;
    // split: the tile's rows, R of them a rank, and how many this rank owns
    int rows = 0, R = 1, mine = 0;
    if (split) {
        int j_, n0_, m0_;
        tile_coords<BN>(a, first_tile, j_, n0_, m0_);
        rows = min(kBM, a.M - m0_);
        R = (rows + a.split - 1) / a.split;
        mine = max(0, min(R, rows - (int)rank * R));
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(bars + s), 1);
            mbar_init(smem_u32(bars + kStages + s), 1);
        }
        for (int c = 0; c < 2; ++c) {
            mbar_init(smem_u32(bars + 2 * kStages + c), 1);
            mbar_init(smem_u32(bars + 2 * kStages + 2 + c), 4);
        }
        dead = 0;
        if (split) {
            // every other rank sends this one its rows: armed before the cluster barrier
            // below lets any of them send
            mbar_init(smem_u32(rx), 1);
            fence_mbarrier_init();
            mbar_arrive_expect_tx(smem_u32(rx), (uint32_t)((a.split - 1) * mine) * kXRow);
        }
        fence_mbarrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (split)
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    // inputs are read and outputs written only after the kernel before has completed (a
    // programmatic launch starts earlier); the next kernel may then start its own prologue
    griddep_wait();
    griddep_launch();
    const uint32_t tmem = *tmem_slot;
    int* stat = a.status;
    auto waitb = [&](uint32_t bar, uint32_t parity) -> bool {
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
    const int nkb = kb1 - kb0;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0 && nkb > 0) {
            int it = 0;   // stage fills so far
            bool ok = true;
            for (int t = first_tile; ok && t < a.tiles; t += tile_step) {
                int j, n0, m0;
                tile_coords<BN>(a, t, j, n0, m0);
                const CUtensorMap* mw = j == 0 ? &map_w0 : j == 1 ? &map_w1 : &map_w2;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages && !waitb(smem_u32(bars + kStages + s), ((it / kStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(bars + s);
                    const uint32_t sa = base + s * kStageBytes;
                    mbar_arrive_expect_tx(fb, (uint32_t)a.abox * (kBK * 2) + TL::kBStage);
                    tma_load_2d(sa, &map_x, kb * kBK, m0, fb);
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_2d(sa + kAStage + c * kBChunk, mw, n0 + c * 64, kb * kBK, fb);
                }
            }
            // copies in flight land before the CTA may end
            for (int q = (it > kStages ? it - kStages : 0); q < it; ++q)
                mbar_wait(smem_u32(bars + q % kStages), (q / kStages) & 1, nullptr, stat);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0 && nkb > 0) {
            const uint32_t idesc = idesc_bf16_bt(kBM, BN);
            int it = 0, tl = 0;
            bool ok = true;
            int last_acc = -1;
            for (int t = first_tile; ok && t < a.tiles; t += tile_step, ++tl) {
                const int acc = tl % naccs;
                // the accumulator is free once the epilogue has read its previous tile
                if (tl >= naccs && !waitb(smem_u32(bars + 2 * kStages + 2 + acc), ((tl / naccs) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!waitb(smem_u32(bars + s), (it / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t ad = sw128_desc(sa + kk * 32, 16);
                        const uint64_t bd = sw128_desc(sa + kAStage + kk * 16 * 128, kBChunk);
                        tc_mma(d, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(bars + kStages + s));   // stage s may be refilled
                }
                if (!ok)
                    break;
                tc_commit(smem_u32(bars + 2 * kStages + acc));   // accumulator ready
                last_acc = tl;
            }
            // MMAs in flight complete before TMEM is freed
            if (last_acc >= 0)
                mbar_wait(smem_u32(bars + 2 * kStages + (last_acc % naccs)), (last_acc / naccs) & 1,
                          nullptr, stat);
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lane quadrant w % 4, one token row
        // a thread
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
        int tl = 0;
        for (int t = first_tile; t < a.tiles && nkb > 0; t += tile_step, ++tl) {
            const int acc = tl % naccs;
            const bool got = waitb(smem_u32(bars + 2 * kStages + acc), (tl / naccs) & 1);
            if (!__all_sync(0xFFFFFFFFu, got))
                break;
            tc_fence_after();
            if (split)
                break;                   // (the partial is exchanged below)
            int j, n0, m0;
            tile_coords<BN>(a, t, j, n0, m0);
            const ProjMat& mat = a.mat[j];
            const int m = m0 + row;
            uint32_t v[32];
            for (int c0 = 0; c0 < BN; c0 += 32) {
                tmem_ld32(trow + acc * BN + c0, v);
                if (m >= a.M || n0 + c0 >= mat.n)
                    continue;
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(mat.out) + (size_t)m * mat.n + n0 + c0);
                const int left = mat.n - (n0 + c0);   // a multiple of 8 columns
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (8 * i < left)
                        __stcs(dst + i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(bars + 2 * kStages + 2 + acc));
        }
    }
    if (split) {
        // Every rank's partial is in its TMEM once its MMAs are done (the epilogue warps
        // have seen the accumulator barrier), and its stages are free. The epilogue
        // threads put the rows other ranks own into the stages ([owner][row - owner R]),
        // thread 0 sends each owner its block with one bulk copy into the owner's receive
        // buffer (slot of this rank among the others), and the owners sum in rank order.
        __syncwarp();
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        int j, n0, m0;
        tile_coords<BN>(a, first_tile, j, n0, m0);
        const ProjMat& mat = a.mat[j];
        const int q = warp & 3, row = q * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
        const int owner = row / R;
        const bool have = warp >= 2 && nkb > 0 && !*(volatile int*)&dead;
        float own[BN];
        if (warp >= 2 && q * 32 < rows) {                         // (warp-uniform)
            uint32_t v[32];
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
                if (have) {
                    tmem_ld32(trow + c0, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = 0u;                                // (no K blocks: zeros)
                }
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    own[c0 + i] = __uint_as_float(v[i]);
            }
            if (row < rows && owner != (int)rank) {
                float4* dst = reinterpret_cast<float4*>(sp + (size_t)(owner * R + row - owner * R) * kXRow);
#pragma unroll
                for (int i = 0; i < BN / 4; ++i)
                    dst[i] = make_float4(own[4 * i], own[4 * i + 1], own[4 * i + 2], own[4 * i + 3]);
            }
        }
        fence_proxy_async_shared();
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int o = 0; o < a.split; ++o) {
                const int orows = max(0, min(R, rows - o * R));
                if (o == (int)rank || orows == 0)
                    continue;
                const uint32_t slot = (uint32_t)((int)rank < o ? rank : rank - 1);
                bulk_s2cluster(cluster_addr(smem_u32(recv) + slot * (uint32_t)R * kXRow, (uint32_t)o),
                               smem_u32(sp) + (uint32_t)(o * R) * kXRow, (uint32_t)orows * kXRow,
                               cluster_addr(smem_u32(rx), (uint32_t)o));
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (warp >= 2 && q * 32 < rows) {
            bool ok = mine == 0 || waitb(smem_u32(rx), 0);
            if (row < rows && owner == (int)rank && ok) {
                const int rl = row - (int)rank * R;
                float sum[BN];
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    sum[c] = 0.f;
                for (int src = 0; src < a.split; ++src) {
                    if (src == (int)rank) {
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            sum[c] += own[c];
                    } else {
                        const int slot = src < (int)rank ? src : src - 1;
                        const float4* pp = reinterpret_cast<const float4*>(recv + (size_t)(slot * R + rl) * kXRow);
#pragma unroll
                        for (int i = 0; i < BN / 4; ++i) {
                            const float4 f = pp[i];
                            sum[4 * i] += f.x;
                            sum[4 * i + 1] += f.y;
                            sum[4 * i + 2] += f.z;
                            sum[4 * i + 3] += f.w;
                        }
                    }
                }
                const int m = m0 + row;
                if (m < a.M && n0 < mat.n) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(mat.out) + (size_t)m * mat.n + n0);
                    const int left = mat.n - n0;          // a multiple of 8 columns
#pragma unroll
                    for (int i = 0; i < BN / 8; ++i)
                        if (8 * i < left)
                            __stcs(dst + i, make_uint4(pack_bf16x2(sum[8 * i], sum[8 * i + 1]),
                                                       pack_bf16x2(sum[8 * i + 2], sum[8 * i + 3]),
                                                       pack_bf16x2(sum[8 * i + 4], sum[8 * i + 5]),
                                                       pack_bf16x2(sum[8 * i + 6], sum[8 * i + 7])));
                }
            }
            if (!ok && lane == 0)
                mbar_drain(smem_u32(rx), 0, kSpinLimitCycles);   // (late copies land first)
        }
        // this CTA's copies are done (read and written) before it may end
        if (threadIdx.x == 0)
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols)
                     : "memory");
}

// ---------------------------------------------------------------- fp32 layers

// C [M, n] = x [M, K] W [K, n], fp32 FMAs in K order; 64 x 64 tiles, 4 x 4 a thread.
// blockIdx.z: which product.
struct F32Mats {
    const float* w[3];
    float* out[3];
    int n[3];
};

__global__ void __launch_bounds__(256) proj_f32_kernel(const float* __restrict__ x, F32Mats mats,
                                                       int M, int K)
{
    __shared__ float xs[16][64 + 4];   // [k][m]
    __shared__ float ws[16][64 + 4];   // [k][n]
    const int j = blockIdx.z;
    const int n = mats.n[j];
    const float* W = mats.w[j];
    float* out = mats.out[j];
    const int n0 = blockIdx.x * 64, m0 = blockIdx.y * 64;
    if (n0 >= n)
        return;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int e = threadIdx.x; e < 64 * 16; e += 256) {
            const int mm = e / 16, kk = e % 16;            // x: consecutive threads along k
            const int m = m0 + mm, k = k0 + kk;
            xs[kk][mm] = (m < M && k < K) ? x[(size_t)m * K + k] : 0.f;
            const int kk2 = e / 64, nn = e % 64;           // W: consecutive threads along n
            const int k2 = k0 + kk2, nc = n0 + nn;
            ws[kk2][nn] = (k2 < K && nc < n) ? W[(size_t)k2 * n + nc] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float xv[4], wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[i] = xs[kk][ty * 4 + i];
                wv[i] = ws[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    acc[i][c] = fmaf(xv[i], wv[c], acc[i][c]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M)
            continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int nc = n0 + tx * 4 + c;
            if (nc < n)
                out[(size_t)m * n + nc] = acc[i][c];
        }
    }
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

// 2D bf16 row-major [rows, cols] tensor, box {64 columns, box_rows}, 128-byte swizzle,
// zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    auto enc = encode_fn();
    if (enc == nullptr)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <int BN>
static size_t proj_smem_bytes()
{
    using TL = Tile<BN>;
    return 1024 + (size_t)TL::kStages * TL::kStageBytes + (2 * TL::kStages + 8) * 8 +
           (BN == 64 ? kRecvBytes : 0);
}

// Tile width: 64 columns once 256-column tiles would leave most SMs idle (few tokens),
// else 256. A function of the layer's shape and the token count only (all three products
// counted, whichever a launch computes), so that the same shape always takes the same
// path and gives the same bits.
static bool proj_narrow(const sdm_cfg& c, int64_t ntok)
{
    const int64_t mtiles = (ntok + kBM - 1) / kBM;
    const int64_t tiles = mtiles * (2 * ((c.dk + 255) / 256) + (c.d + 255) / 256);
    return tiles * 2 < num_sms_current_device();
}

template <int BN>
static cudaError_t launch_tc(const CUtensorMap& mx, const CUtensorMap (&mw)[3], ProjArgs a,
                             cudaStream_t s, bool early, long long full_tiles)
{
    int ntiles = 0;
    for (int q = 0; q < 3; ++q) {
        a.mat[q].ntiles = a.mat[q].ntiles > 0 ? (a.mat[q].n + BN - 1) / BN : 0;
        ntiles += a.mat[q].ntiles;
    }
    a.tiles = a.mtiles * ntiles;
    // 64-column tiles: split along K while the clusters still fit the SMs (at least two K
    // blocks a CTA); the count follows from the shape alone (all three products)
    a.split = 1;
    if (BN == 64) {
        const int sms = num_sms_current_device();
        for (int sp = kMaxSplit; sp > 1; --sp)
            if ((long long)full_tiles * sp <= sms && a.kblocks >= 2 * sp) {
                a.split = sp;
                break;
            }
    }
    const size_t smem = proj_smem_bytes<BN>();
    auto kern = proj_tc_kernel<BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int grid = num_sms_current_device();
    if (grid > a.tiles)
        grid = a.tiles;
    if (a.split > 1)
        grid = a.tiles * a.split;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)a.split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (early) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    return cudaLaunchKernelEx(&cfg, kern, mx, mw[0], mw[1], mw[2], a);
}

cudaError_t launch_project_tc(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                              void* q_w, void* q_r, void* v, cudaStream_t s, int which, bool early)
{
    if (ntok <= 0 || (which & 7) == 0)
        return cudaSuccess;
    const void* wts[3] = {w.W_qw, w.W_qr, w.W_v};
    void* outs[3] = {q_w, q_r, v};
    const int ns[3] = {c.dk, c.dk, c.d};
    int sel[3], nsel = 0;                  // the products this launch computes, in order
    for (int j = 0; j < 3; ++j)
        if (which & (1 << j))
            sel[nsel++] = j;
    if (c.dtype != SDM_BF16) {
        F32Mats fm;
        int nmax = 0;
        for (int q = 0; q < 3; ++q) {
            const int j = sel[q < nsel ? q : 0];
            fm.w[q] = (const float*)wts[j];
            fm.out[q] = (float*)outs[j];
            fm.n[q] = ns[j];
            nmax = ns[j] > nmax ? ns[j] : nmax;
        }
        dim3 grid((unsigned)((nmax + 63) / 64), (unsigned)((ntok + 63) / 64), (unsigned)nsel);
        if (grid.y > 65535u)
            return cudaErrorInvalidValue;
        proj_f32_kernel<<<grid, 256, 0, s>>>((const float*)x, fm, (int)ntok, c.d);
        return cudaGetLastError();
    }
    // Fewer tokens than a tile: the x copies bring only the token rows (rounded up to the
    // 8-row swizzle period); the MMA's other rows read whatever the stage holds, and the
    // rows of the result they give are never stored (a row of the product depends on
    // the same row of x alone).
    CUtensorMap mx, mw[3];
    const int abox = ntok >= kBM ? kBM : (int)((ntok + 7) / 8 * 8);
    if (!make_map(&mx, x, (uint64_t)c.d, (uint64_t)ntok, (uint32_t)abox))
        return cudaErrorInvalidValue;
    ProjArgs a;
    for (int q = 0; q < 3; ++q) {
        const bool used = q < nsel;
        const int j = sel[used ? q : 0];
        if (!make_map(&mw[q], wts[j], (uint64_t)ns[j], (uint64_t)c.d, kBK))
            return cudaErrorInvalidValue;
        a.mat[q].out = outs[j];
        a.mat[q].n = ns[j];
        a.mat[q].ntiles = used ? 1 : 0;   // (counted per tile width at launch)
    }
    a.M = (int)ntok;
    a.K = c.d;
    a.kblocks = (c.d + kBK - 1) / kBK;
    a.mtiles = (int)((ntok + kBM - 1) / kBM);
    a.abox = abox;
    a.tiles = 0;
    a.status = nullptr;
    // tiles of all three products, whichever this launch computes (the split count)
    const long long full64 = (long long)a.mtiles * (2 * ((c.dk + 63) / 64) + (c.d + 63) / 64);
    return proj_narrow(c, ntok) ? launch_tc<64>(mx, mw, a, s, early, full64)
                                : launch_tc<256>(mx, mw, a, s, early, 0);
}

}  // namespace sdm
