// address.cu -- product-key addressing of every token, run up front because it
// depends only on the input ("Sparse Delta Memory" blog, "Write & Read": two sub-keys
// -> outer sum -> top-k; softmax-weighted).
//
//   score_tc_kernel        (score_tc.cu) s_h = K_h q_h for both halves of both queries
//                          on the tensor cores, and the top-W of each half (bf16 layers)
//   subkey_topw_kernel     the same on the SIMT cores in fp32 (fp32 layers and shapes
//                          the tensor path does not take), lists sorted
//                          (score desc, row asc)
//   address_small_kernel   few tokens (a decode step): a cluster of two blocks per group
//                          of queries, one per half, scores from the sub-key table staged
//                          in shared memory on the SIMT cores, keeps each half's top-W, and
//                          merges the halves through distributed shared memory
//   candidate_select_kernel  sorts each half's list, then forms the outer sums of the
//                          pairs of half-ranks (a, b) with (a+1)(b+1) <= W -- the only
//                          pairs that can reach the top-W of all n^2 sums -- keeps their
//                          top-W (bisection over the sums), takes the softmax, and reports
//                          the set in ascending slot order.
#include <algorithm>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

// ------------------------------------------------------------------ half top-W

// Block: 8 warps; blockIdx.y = half (0: K1 on q[0:h], 1: K2 on q[h:dk]). The half's
// sub-key table is staged transposed ([h][P], zero-padded to P = 32*E columns) in
// shared memory; each warp then takes (token, kind) queries in turn.
template <typename IO, int E>
__global__ void __launch_bounds__(256) subkey_topw_kernel(
    const IO* __restrict__ q_w, const IO* __restrict__ q_r, const IO* __restrict__ K1,
    const IO* __restrict__ K2, int64_t ntok, int dk, int n, int W, float* __restrict__ hv,
    int32_t* __restrict__ hi)
{
    constexpr int P = 32 * E;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int h = dk / 2;
    const int half = blockIdx.y;
    IO* KT = reinterpret_cast<IO*>(smem_raw);                     // [h][P]
    float* qs = reinterpret_cast<float*>(smem_raw + (size_t)h * P * sizeof(IO));  // [8][h]
    const IO* K = half ? K2 : K1;
    for (int e = threadIdx.x; e < h * P; e += blockDim.x) {
        const int k = e / P, r = e % P;
        KT[e] = (r < n) ? K[(size_t)r * h + k] : IO(0.0f);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* qw = qs + warp * h;
    const int64_t nq = 2 * ntok;
    for (int64_t qi = (int64_t)blockIdx.x * 8 + warp; qi < nq; qi += (int64_t)gridDim.x * 8) {
        const int kind = (int)(qi / ntok);
        const int64_t tok = qi % ntok;
        const IO* q = (kind ? q_r : q_w) + tok * dk + half * h;
        __syncwarp();
        for (int k = lane; k < h; k += 32)
            qw[k] = to_f32(q[k]);
        __syncwarp();
        float acc[E];
#pragma unroll
        for (int i = 0; i < E; ++i)
            acc[i] = 0.0f;
        for (int k = 0; k < h; ++k) {
            const float qk = qw[k];
            const IO* row = KT + (size_t)k * P + lane;
#pragma unroll
            for (int i = 0; i < E; ++i)
                acc[i] = fmaf(to_f32(row[32 * i]), qk, acc[i]);
        }
        uint64_t key[E];
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int r = lane + 32 * i;
            key[i] = (r < n) ? desc_key(acc[i], (uint32_t)r) : ~0ull;
        }
        warp_bitonic_sort<E>(key);
        const size_t base = (((size_t)kind * ntok + tok) * 2 + half) * W;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int e = lane * E + i;
            if (e < W) {
                hv[base + e] = key_score(key[i]);
                hi[base + e] = (int32_t)key_id(key[i]);
            }
        }
    }
}

// --------------------------------------------------------- candidates + softmax

// One warp per (token, kind). Candidate pairs (a, b) of half-ranks come from a table
// built in shared memory at block start.
__device__ __forceinline__ float __reduce_add_sync_f(float x)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1)
        x += __shfl_xor_sync(0xFFFFFFFFu, x, m);
    return x;
}

// Pairs (a, b) of half-ranks with (a+1)(b+1) <= W, row a's run after the runs of rows < a;
// built by the first W threads of a block. Returns nothing; the count is in *npairs.
__device__ __forceinline__ void build_pairs(unsigned short* pairs, int* npairs, int W)
{
    if (threadIdx.x < W) {
        const int a = threadIdx.x;
        int start = 0;
        for (int a2 = 0; a2 < a; ++a2)
            start += W / (a2 + 1);
        for (int b = 0; b < W / (a + 1); ++b)
            pairs[start + b] = (unsigned short)((a << 8) | b);
        if (a == W - 1)
            *npairs = start + W / (a + 1);
    }
}

// One warp: given each half's W best (score, row) sorted by (score desc, row asc) in
// lv0/li0 and lv1/li1, the W largest outer sums over the candidate pairs by (sum desc,
// slot asc) -- a bisection over the order-preserving keys of the sums, NC candidates a
// lane, stopping once exactly W keys lie at or above the probe, equal sums at the
// threshold to the lower slot -- then the softmax over them, and the set in ascending
// slot order with its weights into idx[0..W) / wsel[0..W). sel: W entries of scratch.
template <int NC, int EW>
__device__ __forceinline__ void select_candidates(const float* lv0, const int* li0, const float* lv1,
                                                  const int* li1, const unsigned short* pairs, int C,
                                                  int n, int W, uint64_t* sel, int32_t* idx,
                                                  float* wsel)
{
    const int lane = threadIdx.x & 31;
    uint32_t ck[NC], cs[NC];
    float cv[NC];
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = lane + 32 * i;
        ck[i] = 0u;                                    // below every real key
        cv[i] = 0.0f;
        cs[i] = 0xFFFFFFFFu;
        if (c < C) {
            const int a = pairs[c] >> 8, b = pairs[c] & 0xFF;
            cv[i] = lv0[a] + lv1[b];
            cs[i] = (uint32_t)li0[a] * (uint32_t)n + (uint32_t)li1[b];
            ck[i] = float_order_bits(cv[i]);
            kmin = min(kmin, ck[i]);
            kmax = max(kmax, ck[i]);
        }
    }
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    uint32_t lo = kmin, hi = kmax + 1;
    int cnt_hi = 0;
    bool exact = false;
    while (!exact && hi - lo > 1) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        int c = 0;
#pragma unroll
        for (int i = 0; i < NC; ++i)
            c += ck[i] >= mid ? 1 : 0;
        c = __reduce_add_sync(0xFFFFFFFFu, c);
        if (c == W) {
            lo = mid;
            exact = true;
        } else if (c > W) {
            lo = mid;
        } else {
            hi = mid;
            cnt_hi = c;
        }
    }
    bool keep[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i)
        keep[i] = exact ? ck[i] >= lo : ck[i] >= hi;
    for (int need = exact ? 0 : W - cnt_hi; need > 0; --need) {
        // the lowest slot among the equal sums not yet kept
        uint32_t best = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < NC; ++i)
            if (!keep[i] && ck[i] == lo)
                best = min(best, cs[i]);
        best = __reduce_min_sync(0xFFFFFFFFu, best);
#pragma unroll
        for (int i = 0; i < NC; ++i)
            if (!keep[i] && ck[i] == lo && cs[i] == best)
                keep[i] = true;
    }
    // softmax over the kept sums (the largest one is the largest of all)
    const float mx = float_from_order_bits(kmax);
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < NC; ++i)
        part += keep[i] ? expf(cv[i] - mx) : 0.0f;
    part = __reduce_add_sync_f(part);
    int base_pos = 0;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep[i]);
        if (keep[i]) {
            const int pos = base_pos + __popc(bal & ((1u << lane) - 1u));
            sel[pos] = ((uint64_t)cs[i] << 32) | __float_as_uint(expf(cv[i] - mx) / part);
        }
        base_pos += __popc(bal);
    }
    __syncwarp();
    // report the set in ascending slot order, weights alongside
    uint64_t k2[EW];
#pragma unroll
    for (int i = 0; i < EW; ++i) {
        const int e = lane * EW + i;
        k2[i] = (e < W) ? sel[e] : ~0ull;
    }
    warp_bitonic_sort<EW>(k2);
#pragma unroll
    for (int i = 0; i < EW; ++i) {
        const int e = lane * EW + i;
        if (e < W) {
            idx[e] = (int32_t)(k2[i] >> 32);
            wsel[e] = __uint_as_float((uint32_t)k2[i]);
        }
    }
}

// One warp per (token, kind). Candidate pairs (a, b) of half-ranks come from a table
// built in shared memory at block start.
template <int NC, int EW, int EH>
__global__ void __launch_bounds__(256) candidate_select_kernel(
    const float* __restrict__ hv, const int32_t* __restrict__ hi, int64_t ntok, int n, int W,
    int32_t* __restrict__ idx, float* __restrict__ wsel)
{
    __shared__ unsigned short pairs[32 * NC];     // (a << 8) | b
    __shared__ int npairs;
    __shared__ float lv[8][2][64];
    __shared__ int li[8][2][64];
    __shared__ uint64_t sel[8][64];
    build_pairs(pairs, &npairs, W);
    __syncthreads();
    const int C = npairs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nq = 2 * ntok;
    for (int64_t qi = (int64_t)blockIdx.x * 8 + warp; qi < nq; qi += (int64_t)gridDim.x * 8) {
        const int kind = (int)(qi / ntok);
        const int64_t tok = qi % ntok;
        const size_t base = ((size_t)kind * ntok + tok) * 2 * W;
        // each half's W best rows, sorted (score desc, row asc): the tensor-core scoring
        // writes them in row order
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint64_t hk[EH];
#pragma unroll
            for (int i = 0; i < EH; ++i) {
                const int e = lane * EH + i;
                hk[i] = e < W ? desc_key(hv[base + h * W + e], (uint32_t)hi[base + h * W + e]) : ~0ull;
            }
            warp_bitonic_sort<EH>(hk);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < EH; ++i) {
                const int e = lane * EH + i;
                if (e < W) {
                    lv[warp][h][e] = key_score(hk[i]);
                    li[warp][h][e] = (int)key_id(hk[i]);
                }
            }
        }
        __syncwarp();
        const size_t ob = ((size_t)tok * 2 + kind) * W;
        select_candidates<NC, EW>(lv[warp][0], li[warp][0], lv[warp][1], li[warp][1], pairs, C, n, W,
                                  sel[warp], idx + ob, wsel + ob);
    }
}

// ---------------------------------------------- few tokens: a block pair a query group

constexpr int kQG = 4;    // queries (token, kind) a cluster

__device__ __forceinline__ uint32_t cluster_rank_u()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t local, uint32_t rank)
{
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// <K row chunk, q chunk> of 16 bytes each, in fp32 FMAs in element order
__device__ __forceinline__ float dot16(const uint4& k, const uint4& q, float acc, bf16)
{
    const uint32_t kw[4] = {k.x, k.y, k.z, k.w}, qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(kw[i] << 16), __uint_as_float(qw[i] << 16), acc);
        acc = fmaf(__uint_as_float(kw[i] & 0xFFFF0000u), __uint_as_float(qw[i] & 0xFFFF0000u), acc);
    }
    return acc;
}

__device__ __forceinline__ float dot16(const uint4& k, const uint4& q, float acc, float)
{
    acc = fmaf(__uint_as_float(k.x), __uint_as_float(q.x), acc);
    acc = fmaf(__uint_as_float(k.y), __uint_as_float(q.y), acc);
    acc = fmaf(__uint_as_float(k.z), __uint_as_float(q.z), acc);
    return fmaf(__uint_as_float(k.w), __uint_as_float(q.w), acc);
}

// One warp: the W best of the n scores s[0..n) by (score desc, row asc), sorted, into
// lv[0..W) / li[0..W). A bisection over the order-preserving keys finds the W-th largest;
// ties at the threshold go to the lower rows. It starts from whatever holds of a bracket
// mean + (z -+ 1/2) sd around the W-th score (the scores of a row are near normal; z is
// the standard normal quantile of 1 - W/n), checked by one counting pass; the search is
// exact either way. out: 64 entries of scratch.
template <int KPL>
__device__ __forceinline__ void warp_topw(const float* s, int n, int W, float z, uint64_t* out,
                                          float* lv, int* li)
{
    const int lane = threadIdx.x & 31;
    uint32_t key[KPL];
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    float sum = 0.f, sum2 = 0.f;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int r = lane + 32 * i;
        const float f = r < n ? s[r] : 0.f;
        key[i] = r < n ? float_order_bits(f) : 0u;     // 0 is below every real key
        if (r < n) {
            kmin = min(kmin, key[i]);
            kmax = max(kmax, key[i]);
            sum += f;
            sum2 = fmaf(f, f, sum2);
        }
    }
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    sum = __reduce_add_sync_f(sum);
    sum2 = __reduce_add_sync_f(sum2);
    uint32_t lo = kmin, hi = kmax + 1;
    int cnt_hi = 0;
    bool exact = false;
    {
        const float mean = sum / n;
        const float sd = sqrtf(fmaxf(sum2 / n - mean * mean, 0.f));
        const uint32_t bl = float_order_bits(mean + (z - 0.5f) * sd);
        const uint32_t bh = float_order_bits(mean + (z + 0.5f) * sd);
        int cl = 0, ch = 0;
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            cl += key[i] >= bl ? 1 : 0;
            ch += key[i] >= bh ? 1 : 0;
        }
        cl = __reduce_add_sync(0xFFFFFFFFu, cl);
        ch = __reduce_add_sync(0xFFFFFFFFu, ch);
        // at least W keys lie at or above lo, fewer than W at or above hi
        if (bl > lo && bl < hi) {
            if (cl == W) {
                lo = bl;
                exact = true;
            } else if (cl > W) {
                lo = bl;
            } else {
                hi = bl;
                cnt_hi = cl;
            }
        }
        if (!exact && bh > lo && bh < hi) {
            if (ch == W) {
                lo = bh;
                exact = true;
            } else if (ch > W) {
                lo = bh;
            } else {
                hi = bh;
                cnt_hi = ch;
            }
        }
    }
    while (!exact && hi - lo > 1) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        int c = 0;
#pragma unroll
        for (int i = 0; i < KPL; ++i)
            c += key[i] >= mid ? 1 : 0;
        c = __reduce_add_sync(0xFFFFFFFFu, c);
        if (c == W) {
            lo = mid;
            exact = true;
        } else if (c > W) {
            lo = mid;
        } else {
            hi = mid;
            cnt_hi = c;
        }
    }
    // kept: keys >= lo when exactly W lie there, else keys >= hi and the lowest rows
    // among those equal to lo (rows ascend with i, then with the lane)
    const int need = exact ? 0 : W - cnt_hi;
    int ties_before = 0, pos = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const bool tie = !exact && key[i] == lo && key[i] != 0u;
        const unsigned tb = __ballot_sync(0xFFFFFFFFu, tie);
        const int trank = ties_before + __popc(tb & ((1u << lane) - 1u));
        const bool keep = key[i] != 0u && ((exact ? key[i] >= lo : key[i] >= hi) ||
                                           (tie && trank < need));
        const unsigned kb = __ballot_sync(0xFFFFFFFFu, keep);
        const int at = pos + __popc(kb & ((1u << lane) - 1u));
        if (keep && at < 64) {
            const int r = lane + 32 * i;
            out[at] = desc_key(s[r], (uint32_t)r);
        }
        pos += __popc(kb);
        ties_before += __popc(tb);
    }
    __syncwarp();
    uint64_t k2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int e = lane * 2 + i;
        k2[i] = e < W ? out[e] : ~0ull;
    }
    warp_bitonic_sort<2>(k2);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int e = lane * 2 + i;
        if (e < W) {
            lv[e] = key_score(k2[i]);
            li[e] = (int)key_id(k2[i]);
        }
    }
    __syncwarp();
}

// the scores of a bf16 half on the tensor cores when its width is a multiple of 16
template <typename IO>
__device__ __forceinline__ bool score_mma(int h)
{
    return sizeof(IO) == 2 && h % 16 == 0;
}

// s[j][r] = <K[r], q_j> for the rows r < n of a bf16 table in shared memory (rows rs bytes
// apart, whole 16-row tiles) and the kQG queries (8 rows rs bytes apart, the rest zero):
// warp w takes the 16-row tiles w, w + 16, ...; per tile and 16 columns one
// mma.sync.m16n8k16 (bf16 x bf16 -> fp32) with fragments from ldmatrix.
__device__ __forceinline__ void score_tiles_mma(uint32_t ktab, uint32_t qs, int rs, int n, int h,
                                                float* sc, int sc_stride)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    const int tiles = (n + 15) / 16;
    for (int mt = warp; mt < tiles; mt += nwarps) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        // lane i addresses row (i % 8) of 8x8 matrix i / 8: A matrices are (rows 0-7 | 8-15)
        // x (columns 0-7 | 8-15); B matrices are the 8 query rows x (columns 0-7 | 8-15)
        const uint32_t arow = ktab + (uint32_t)((mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * rs) +
                              (uint32_t)(16 * (lane >> 4));
        const uint32_t brow = qs + (uint32_t)((lane & 7) * rs) + (uint32_t)(16 * ((lane >> 3) & 1));
        for (int k0 = 0; k0 < h; k0 += 16) {
            uint32_t a0, a1, a2, a3, b0, b1;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(arow + (uint32_t)(k0 * 2)));
            asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                         : "=r"(b0), "=r"(b1)
                         : "r"(brow + (uint32_t)(k0 * 2)));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
        // c0, c1: row gid, queries 2 tig and 2 tig + 1; c2, c3: row gid + 8
        const int r0 = mt * 16 + gid;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 2 * tig + (e & 1), r = r0 + 8 * (e >> 1);
            if (j < kQG && r < n)
                sc[j * sc_stride + r] = c[e];
        }
    }
}

struct SmallSmem {
    // offsets in the dynamic shared memory of address_small_kernel; rows of the sub-key
    // table and of the queries are rs bytes apart (one row plus 16 bytes, so that eight
    // rows read at one column fall in different banks)
    uint32_t rs, ktab, qs, sc, lv, li, lv1, li1, hk, total;
};

__host__ __device__ inline SmallSmem small_layout(int n, int h, int es, int kpl)
{
    SmallSmem L;
    uint32_t o = 0;
    L.rs = (uint32_t)(h * es + 16);
    L.ktab = o; o += (uint32_t)((n + 15) / 16 * 16) * L.rs;     // whole 16-row tiles
    L.qs = o; o += 8u * L.rs;                                   // 8 rows: the MMA's N
    L.sc = o; o += (uint32_t)(kQG * 32 * kpl * 4);
    L.lv = o; o += kQG * 64 * 4;
    L.li = o; o += kQG * 64 * 4;
    L.lv1 = o; o += kQG * 64 * 4;
    L.li1 = o; o += kQG * 64 * 4;
    L.hk = o; o += kQG * 64 * 8;
    L.total = o;
    return L;
}

// Few tokens (a decode step): a cluster of two blocks takes kQG queries (token, kind),
// block 0 the first half of each query against K1, block 1 the second against K2:
//  1. the block stages its sub-key table in shared memory with one bulk copy a row and
//     its queries' halves with plain loads;
//  2. the scores s[r] = <K[r], q_half>, fp32 sums of exact products: bf16 tables whose
//     half-width is a multiple of 16 on the tensor cores (mma.sync m16n8k16, the table as
//     A in 16-row tiles, the kQG queries padded to 8 as B), others on the SIMT cores
//     (thread t takes row t, its 16-byte chunks in a rotated order, products in element
//     order);
//  3. warp j keeps query j's W best rows of this half (warp_topw);
//  4. after a cluster barrier, block 0's warp j reads block 1's list of query j through
//     distributed shared memory and merges the two exactly as the candidate kernel does
//     (select_candidates): the set and its softmax weights.
constexpr int kSmallThreads = 512;

template <typename IO, int NC, int EW, int KPL>
__global__ void __launch_bounds__(kSmallThreads) address_small_kernel(
    const IO* __restrict__ q_w, const IO* __restrict__ q_r, const IO* __restrict__ K1,
    const IO* __restrict__ K2, int64_t ntok, int dk, int n, int W, float z,
    int32_t* __restrict__ idx, float* __restrict__ wsel, int* status)
{
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ unsigned short pairs[32 * NC];
    __shared__ int npairs;
    __shared__ __align__(8) uint64_t kbar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t half = cluster_rank_u();
    const int64_t q0 = (int64_t)(blockIdx.x >> 1) * kQG;      // first query of the group
    const int64_t nq = 2 * ntok;
    const int h = dk / 2;
    const int rowb = h * (int)sizeof(IO);
    const int nch = rowb / 16;
    const SmallSmem L = small_layout(n, h, (int)sizeof(IO), KPL);
    const int rs = (int)L.rs;
    const uint32_t base = smem_u32(sm);
    float* sc = reinterpret_cast<float*>(sm + L.sc);
    float* lv = reinterpret_cast<float*>(sm + L.lv);
    int* li = reinterpret_cast<int*>(sm + L.li);
    const uint32_t tbytes = (uint32_t)(n * rowb);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&kbar), 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // 1. the half's sub-key table (one bulk copy a row, issued by every thread) and the
    //    queries' halves (rows kQG..7 zero)
    if (threadIdx.x == 0)
        mbar_arrive_expect_tx(smem_u32(&kbar), tbytes);
    __syncthreads();
    {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(half ? K2 : K1);
        for (int r = threadIdx.x; r < n; r += blockDim.x)
            bulk_g2s(base + L.ktab + (uint32_t)(r * rs), src + (size_t)r * rowb, (uint32_t)rowb,
                     smem_u32(&kbar));
        for (int e = threadIdx.x; e < 8 * h; e += blockDim.x) {
            const int j = e / h, k = e % h;
            const int64_t qi = q0 + j;                          // token-major: tok * 2 + kind
            IO val = IO(0.0f);
            if (j < kQG && qi < nq)
                val = ((qi & 1) ? q_r : q_w)[(qi >> 1) * dk + half * h + k];
            reinterpret_cast<IO*>(sm + L.qs + j * rs)[k] = val;
        }
        // rows of the last 16-row tile past the table: zero (read by the MMA, never kept)
        for (int e = threadIdx.x; e < ((n + 15) / 16 * 16 - n) * h; e += blockDim.x)
            reinterpret_cast<IO*>(sm + L.ktab + (n + e / h) * rs)[e % h] = IO(0.0f);
    }
    build_pairs(pairs, &npairs, W);
    __syncthreads();
    bool ok = mbar_wait(smem_u32(&kbar), 0, nullptr, status);
    ok = __syncthreads_and(ok) != 0;
    // 2. scores of this half
    if (ok && score_mma<IO>(h)) {
        score_tiles_mma(base + L.ktab, base + L.qs, rs, n, h, sc, 32 * KPL);
    } else if (ok) {
        for (int r = threadIdx.x; r < n; r += blockDim.x) {
            float acc[kQG];
#pragma unroll
            for (int j = 0; j < kQG; ++j)
                acc[j] = 0.f;
            const unsigned char* kr = sm + L.ktab + (size_t)r * rs;
            for (int c = 0; c < nch; ++c) {
                const int cc = (c + r) % nch;
                const uint4 kv = *reinterpret_cast<const uint4*>(kr + cc * 16);
#pragma unroll
                for (int j = 0; j < kQG; ++j) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sm + L.qs + j * rs + cc * 16);
                    acc[j] = dot16(kv, qv, acc[j], IO(0.0f));
                }
            }
#pragma unroll
            for (int j = 0; j < kQG; ++j)
                sc[j * 32 * KPL + r] = acc[j];
        }
    }
    __syncthreads();
    // 3. query j's W best rows of this half
    if (ok && warp < kQG && q0 + warp < nq)
        warp_topw<KPL>(sc + warp * 32 * KPL, n, W, z,
                       reinterpret_cast<uint64_t*>(sm + L.hk) + warp * 64, lv + warp * 64,
                       li + warp * 64);
    __syncthreads();
    cluster_sync_all();
    // 4. block 0 merges each query's halves
    if (ok && half == 0 && warp < kQG && q0 + warp < nq) {
        float* lv1 = reinterpret_cast<float*>(sm + L.lv1) + warp * 64;
        int* li1 = reinterpret_cast<int*>(sm + L.li1) + warp * 64;
        for (int e = lane; e < W; e += 32) {
            lv1[e] = __uint_as_float(ld_dsmem_u32(base + L.lv + (warp * 64 + e) * 4, 1));
            li1[e] = (int)ld_dsmem_u32(base + L.li + (warp * 64 + e) * 4, 1);
        }
        __syncwarp();
        const int64_t qi = q0 + warp;
        const size_t ob = ((size_t)(qi >> 1) * 2 + (qi & 1)) * W;
        select_candidates<NC, EW>(lv + warp * 64, li + warp * 64, lv1, li1, pairs, npairs, n, W,
                                  reinterpret_cast<uint64_t*>(sm + L.hk) + warp * 64, idx + ob,
                                  wsel + ob);
    }
    // block 1 stays until block 0 has read its lists
    cluster_sync_all();
}

static int candidate_count(int W)
{
    int c = 0;
    for (int a = 1; a <= W; ++a)
        c += W / a;
    return c;
}

size_t address_ws_bytes(const sdm_cfg& c, int64_t ntok)
{
    // half lists: [2 kinds][ntok][2 halves][W] x (fp32 score + int32 row)
    const size_t n = (size_t)2 * ntok * 2 * c.w;
    return ((n * 8) + 255) / 256 * 256;
}

template <typename IO, int E>
static cudaError_t run_topw(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                            const void* q_r, int64_t ntok, float* hv, int32_t* hi,
                            cudaStream_t s)
{
    const int h = c.dk / 2;
    const size_t smem = (size_t)h * 32 * E * sizeof(IO) + 8 * h * sizeof(float);
    auto kern = subkey_topw_kernel<IO, E>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    const int sms = num_sms_current_device();
    int64_t blocks = (2 * ntok + 7) / 8;
    if (blocks > (int64_t)sms * 2)
        blocks = (int64_t)sms * 2;
    dim3 grid((unsigned)blocks, 2);
    kern<<<grid, 256, smem, s>>>((const IO*)q_w, (const IO*)q_r, (const IO*)K1, (const IO*)K2,
                                 ntok, c.dk, c.n_sub, c.w, hv, hi);
    return cudaGetLastError();
}

template <typename IO>
static cudaError_t run_topw_e(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                              const void* q_r, int64_t ntok, float* hv, int32_t* hi,
                              cudaStream_t s)
{
    const int n = c.n_sub;
    if (n <= 32) return run_topw<IO, 1>(c, K1, K2, q_w, q_r, ntok, hv, hi, s);
    if (n <= 64) return run_topw<IO, 2>(c, K1, K2, q_w, q_r, ntok, hv, hi, s);
    if (n <= 128) return run_topw<IO, 4>(c, K1, K2, q_w, q_r, ntok, hv, hi, s);
    if (n <= 256) return run_topw<IO, 8>(c, K1, K2, q_w, q_r, ntok, hv, hi, s);
    return run_topw<IO, 16>(c, K1, K2, q_w, q_r, ntok, hv, hi, s);
}

template <int NC, int EW, int EH>
static cudaError_t run_cand(const sdm_cfg& c, int64_t ntok, const float* hv, const int32_t* hi,
                            int32_t* idx, float* wsel, cudaStream_t s)
{
    const int sms = num_sms_current_device();
    int64_t blocks = (2 * ntok + 7) / 8;
    if (blocks > (int64_t)sms * 4)
        blocks = (int64_t)sms * 4;
    candidate_select_kernel<NC, EW, EH><<<(unsigned)blocks, 256, 0, s>>>(hv, hi, ntok, c.n_sub, c.w,
                                                                    idx, wsel);
    return cudaGetLastError();
}

// Few tokens (a decode step): a block pair per group of queries does everything
// (address_small_kernel). The choice depends on the shape only, so a shape always gives
// the same bits.
constexpr int64_t kSmallAddressTokens = 256;

static int small_kpl(int n) { return n <= 32 ? 1 : n <= 64 ? 2 : n <= 128 ? 4 : n <= 256 ? 8 : 16; }

bool address_small_path(const sdm_cfg& c, int64_t ntok)
{
    const int es = c.dtype == SDM_BF16 ? 2 : 4;
    const int h = c.dk / 2;
    return ntok <= kSmallAddressTokens && (h * es) % 16 == 0 &&
           small_layout(c.n_sub, h, es, small_kpl(c.n_sub)).total <= 200u * 1024u;
}

template <typename IO, int NC, int EW, int KPL>
static cudaError_t run_small_kpl(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                                 const void* q_r, int64_t ntok, int32_t* idx, float* wsel,
                                 int* status, cudaStream_t s)
{
    auto kern = address_small_kernel<IO, NC, EW, KPL>;
    const SmallSmem L = small_layout(c.n_sub, c.dk / 2, (int)sizeof(IO), KPL);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L.total);
    if (e != cudaSuccess)
        return e;
    const int64_t groups = (2 * ntok + kQG - 1) / kQG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * groups), 1, 1);
    cfg.blockDim = dim3(kSmallThreads, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float z = normal_upper_quantile((double)c.w / c.n_sub);
    return cudaLaunchKernelEx(&cfg, kern, (const IO*)q_w, (const IO*)q_r, (const IO*)K1,
                              (const IO*)K2, ntok, c.dk, c.n_sub, c.w, z, idx, wsel, status);
}

template <typename IO, int NC, int EW>
static cudaError_t run_small_k(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                               const void* q_r, int64_t ntok, int32_t* idx, float* wsel,
                               int* status, cudaStream_t s)
{
    switch (small_kpl(c.n_sub)) {
    case 1: return run_small_kpl<IO, NC, EW, 1>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    case 2: return run_small_kpl<IO, NC, EW, 2>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    case 4: return run_small_kpl<IO, NC, EW, 4>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    case 8: return run_small_kpl<IO, NC, EW, 8>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    default: return run_small_kpl<IO, NC, EW, 16>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    }
}

template <typename IO>
static cudaError_t run_small(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                             const void* q_r, int64_t ntok, int32_t* idx, float* wsel,
                             int* status, cudaStream_t s)
{
    switch (c.w) {
    case 8: return run_small_k<IO, 1, 1>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    case 16: return run_small_k<IO, 2, 1>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    case 32: return run_small_k<IO, 4, 1>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    case 64: return run_small_k<IO, 9, 2>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_address(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                           const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                           int* status, cudaStream_t s)
{
    if (ntok <= 0)
        return cudaSuccess;
    if (address_small_path(c, ntok))
        return c.dtype == SDM_BF16
                   ? run_small<bf16>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s)
                   : run_small<float>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s);
    float* hv = (float*)ws;
    int32_t* hi = (int32_t*)((char*)ws + (size_t)2 * ntok * 2 * c.w * sizeof(float));
    // bf16 layers score on the tensor cores; fp32 layers (exact fp32 products) and other
    // shapes on the SIMT kernel
    cudaError_t e = score_tc_supported(c)
                        ? launch_score_tc(c, K1, K2, q_w, q_r, ntok, hv, hi, status, s)
                        : (c.dtype == SDM_BF16)
                              ? run_topw_e<bf16>(c, K1, K2, q_w, q_r, ntok, hv, hi, s)
                              : run_topw_e<float>(c, K1, K2, q_w, q_r, ntok, hv, hi, s);
    if (e != cudaSuccess)
        return e;
    const int C = candidate_count(c.w);
    switch (c.w) {
    case 8: return run_cand<1, 1, 1>(c, ntok, hv, hi, idx, wsel, s);      // 20 candidates
    case 16: return run_cand<2, 1, 1>(c, ntok, hv, hi, idx, wsel, s);     // 50
    case 32: return run_cand<4, 1, 1>(c, ntok, hv, hi, idx, wsel, s);     // 119
    case 64: return run_cand<9, 2, 2>(c, ntok, hv, hi, idx, wsel, s);     // 280
    default: (void)C; return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
