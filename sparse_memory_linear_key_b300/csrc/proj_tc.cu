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
//  * many tokens (prefill): a persistent kernel, one CTA per SM walking the tiles, two
//    TMEM accumulators so that a tile's epilogue overlaps the next tile's MMAs;
//  * few tokens (decode): too few tiles to fill the SMs, so each tile is split along K
//    over a cluster of up to 8 CTAs; after a cluster barrier every CTA pushes each row
//    of its fp32 partial tile into the shared memory of the CTA that owns the row
//    (distributed shared memory stores), and after a second one each CTA sums its rows
//    over the cluster's partials in rank order (the same shape always gives the same
//    bits).
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
constexpr int kBN = 256;                 // output columns a tile (MMA N)
constexpr int kBK = 64;                  // K columns a stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr uint32_t kAStage = kBM * kBK * 2;            // 16 KB
constexpr uint32_t kBChunk = kBK * 64 * 2;             // 64 K-rows x 64 columns: 8 KB
constexpr uint32_t kBStage = kBChunk * (kBN / 64);     // 32 KB
constexpr uint32_t kStageBytes = kAStage + kBStage;    // 48 KB
constexpr int kThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kMaxSplit = 8;             // CTAs of a cluster sharing one tile along K
constexpr int kRedStride = kBN + 4;      // fp32 per partial-tile row in shared memory

struct ProjMat {
    void* out;      // [M, n] bf16
    int n;          // output columns
    int ntiles;     // ceil(n / kBN)
};

struct ProjArgs {
    ProjMat mat[3];
    int M, K, kblocks, mtiles, tiles;
    int split;      // CTAs per tile (cluster size); 1: persistent, whole K per CTA
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

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// tile t -> product j, its column tile and its token tile (token tiles innermost)
__device__ __forceinline__ void tile_coords(const ProjArgs& a, int t, int& j, int& n0, int& m0)
{
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
    n0 = (rem / a.mtiles) * kBN;
    m0 = (rem % a.mtiles) * kBM;
}

// ------------------------------------------------------------------------ kernel

// One kernel for both modes. split == 1: persistent, CTA b takes tiles b, b + grid, ...
// over the whole K, two accumulators. split > 1: CTA rank r of cluster c takes tile c over
// its share of the K blocks, one accumulator, then the cluster reduces the partials.
__global__ void __launch_bounds__(kThreads, 1) proj_tc_kernel(
    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w0,
    const __grid_constant__ CUtensorMap map_w1, const __grid_constant__ CUtensorMap map_w2,
    ProjArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sp = smem_raw + (base - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sp + kStages * kStageBytes);
    // bars: [0, S) full, [S, 2S) empty, 2S + {0, 1} accumulator full, 2S + {2, 3} empty
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    __shared__ int dead;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool split = a.split > 1;
    const uint32_t rank = split ? cluster_rank() : 0u;
    const int first_tile = split ? (int)(blockIdx.x / a.split) : (int)blockIdx.x;
    const int tile_step = split ? a.tiles : (int)gridDim.x;     // split: one tile a cluster
    const int kb0 = split ? (int)((long long)a.kblocks * rank / a.split) : 0;
    const int kb1 = split ? (int)((long long)a.kblocks * (rank + 1) / a.split) : a.kblocks;
    const int naccs = split ? 1 : 2;
    const uint32_t tmem_cols = split ? 256u : 512u;

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
                tile_coords(a, t, j, n0, m0);
                const CUtensorMap* mw = j == 0 ? &map_w0 : j == 1 ? &map_w1 : &map_w2;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages && !waitb(smem_u32(bars + kStages + s), ((it / kStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(bars + s);
                    const uint32_t sa = base + s * kStageBytes;
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    tma_load_2d(sa, &map_x, kb * kBK, m0, fb);
#pragma unroll
                    for (int c = 0; c < kBN / 64; ++c)
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
            const uint32_t idesc = idesc_bf16_bt(kBM, kBN);
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
                const uint32_t d = tmem + acc * kBN;
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
                break;                   // (the partial is read after the cluster barrier)
            int j, n0, m0;
            tile_coords(a, t, j, n0, m0);
            const ProjMat& mat = a.mat[j];
            const int m = m0 + row;
            uint32_t v[32];
            for (int c0 = 0; c0 < kBN; c0 += 32) {
                tmem_ld32(trow + acc * kBN + c0, v);
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
        // Every CTA's MMAs are done once all have reached the barrier, so their stage
        // memory is free. Rows [r R, (r+1) R) of the tile belong to rank r: each epilogue
        // thread pushes its row of the fp32 partial, 32 columns at a time, into the owning
        // rank's shared memory, slot [this rank][row - r R]; after a second barrier each rank
        // sums its rows over the slots in rank order and stores them.
        __syncthreads();
        cluster_sync();
        tc_fence_after();
        int j, n0, m0;
        tile_coords(a, first_tile, j, n0, m0);
        const ProjMat& mat = a.mat[j];
        const int rows = min(kBM, a.M - m0);
        const int R = (rows + a.split - 1) / a.split;
        const uint32_t red0 = base;                     // [split][R][kRedStride] fp32
        if (warp >= 2) {
            const int q = warp & 3, row = q * 32 + lane;
            const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
            if (q * 32 < rows) {                        // (warp-uniform)
                const uint32_t owner = (uint32_t)(row / R);
                const uint32_t slot =
                    red0 + (uint32_t)((rank * R + (row - (int)owner * R)) * kRedStride) * 4u;
                uint32_t remote = 0;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(slot), "r"(owner));
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    uint32_t v[32];
                    if (nkb > 0) {
                        tmem_ld32(trow + c0, v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = 0u;                  // (a CTA without K blocks adds zeros)
                    }
                    if (row < rows) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             remote + (uint32_t)(c0 + 4 * i) * 4u),
                                         "r"(v[4 * i]), "r"(v[4 * i + 1]), "r"(v[4 * i + 2]),
                                         "r"(v[4 * i + 3])
                                         : "memory");
                    }
                }
            }
        }
        cluster_sync();
        const float* red = reinterpret_cast<const float*>(sp);
        const int r0 = (int)rank * R, r1 = min(rows, r0 + R);
        const int cols = min(kBN, mat.n - n0);          // a multiple of 8
        const int groups = cols / 8;
        for (int e = threadIdx.x; e < (r1 - r0) * groups; e += kThreads) {
            const int rl = e / groups, c = (e % groups) * 8;
            float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int src = 0; src < a.split; ++src) {
                const float4* pp = reinterpret_cast<const float4*>(red + (size_t)(src * R + rl) * kRedStride + c);
                const float4 p0 = pp[0], p1 = pp[1];
                sum[0] += p0.x; sum[1] += p0.y; sum[2] += p0.z; sum[3] += p0.w;
                sum[4] += p1.x; sum[5] += p1.y; sum[6] += p1.z; sum[7] += p1.w;
            }
            uint4 o = make_uint4(pack_bf16x2(sum[0], sum[1]), pack_bf16x2(sum[2], sum[3]),
                                 pack_bf16x2(sum[4], sum[5]), pack_bf16x2(sum[6], sum[7]));
            __stcs(reinterpret_cast<uint4*>(static_cast<bf16*>(mat.out) + (size_t)(m0 + r0 + rl) * mat.n + n0 + c), o);
        }
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

static size_t proj_smem_bytes() { return 1024 + (size_t)kStages * kStageBytes + (2 * kStages + 4) * 8 + 16; }

// CTAs per tile: a cluster per tile along K once the tiles of the whole-K kernel would
// leave most SMs idle (few tokens). A function of the layer's shape and the token count
// only (all three products counted, whichever a launch computes), so that the same shape
// always takes the same path and gives the same bits.
static int proj_split_for(const sdm_cfg& c, int64_t ntok)
{
    const int sms = num_sms_current_device();
    const int64_t mtiles = (ntok + kBM - 1) / kBM;
    const int64_t tiles = mtiles * (2 * ((c.dk + kBN - 1) / kBN) + (c.d + kBN - 1) / kBN);
    const int kblocks = (c.d + kBK - 1) / kBK;
    if (tiles * 2 >= sms)
        return 1;
    int s = kMaxSplit;
    while (s > 1 && (s > kblocks || tiles * s > 2 * sms))
        s /= 2;
    return s;
}

cudaError_t launch_project_tc(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                              void* q_w, void* q_r, void* v, cudaStream_t s, int which)
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
    CUtensorMap mx, mw[3];
    if (!make_map(&mx, x, (uint64_t)c.d, (uint64_t)ntok, kBM))
        return cudaErrorInvalidValue;
    ProjArgs a;
    int ntiles = 0;
    for (int q = 0; q < 3; ++q) {
        const bool used = q < nsel;
        const int j = sel[used ? q : 0];
        if (!make_map(&mw[q], wts[j], (uint64_t)ns[j], (uint64_t)c.d, kBK))
            return cudaErrorInvalidValue;
        a.mat[q].out = outs[j];
        a.mat[q].n = ns[j];
        a.mat[q].ntiles = used ? (ns[j] + kBN - 1) / kBN : 0;
        ntiles += a.mat[q].ntiles;
    }
    a.M = (int)ntok;
    a.K = c.d;
    a.kblocks = (c.d + kBK - 1) / kBK;
    a.mtiles = (int)((ntok + kBM - 1) / kBM);
    a.tiles = a.mtiles * ntiles;
    a.status = nullptr;
    a.split = proj_split_for(c, ntok);
    const size_t smem = proj_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    if (a.split == 1) {
        int grid = num_sms_current_device();
        if (grid > a.tiles)
            grid = a.tiles;
        proj_tc_kernel<<<grid, kThreads, smem, s>>>(mx, mw[0], mw[1], mw[2], a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.tiles * a.split), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, proj_tc_kernel, mx, mw[0], mw[1], mw[2], a);
}

}  // namespace sdm
