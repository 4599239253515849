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
//                          in shared memory, keeps each half's top-W, and merges the
//                          halves through distributed shared memory
//   candidate_select_kernel  orders each half's list, then forms the outer sums of the
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
        const int kind = qi >= ntok ? 1 : 0;             // (qi < 2 ntok)
        const int64_t tok = kind ? qi - ntok : qi;
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

// ----------------------------------------------- exact top-W: shared pieces

// An element's composite key: ascending = larger order key first, then smaller id.
__device__ __forceinline__ uint64_t comp_key(uint32_t key, uint32_t id)
{
    return ((uint64_t)(~key) << 32) | id;
}

// Which elements group_kth keeps: exact ? key >= lo : comp_key(key, id) <= e.
struct KthSel {
    bool exact;
    uint32_t lo;
    uint64_t e;
};

// Narrow the bracket [lo, hi) with a probe p that c elements reach (key >= p).
__device__ __forceinline__ void kth_narrow(uint32_t p, int c, int W, uint32_t& lo, uint32_t& hi,
                                           int& cnt_lo, int& cnt_hi)
{
    if (c >= W) {
        if (p > lo) {
            lo = p;
            cnt_lo = c;
        }
    } else if (p < hi) {
        hi = p;
        cnt_hi = c;
    }
}

// One warp: given each half's W best (score, row) sorted by (score desc, row asc) in
// lv0/li0 and lv1/li1, the W largest outer sums over the candidate pairs by (sum desc,
// slot asc) -- a bisection over the order-preserving keys of the sums, NC candidates a
// lane, stopping once exactly W keys lie at or above the probe, equal sums at the
// threshold to the lower slot -- then the softmax over them, and the set in ascending
// slot order with its weights into idx[0..W) / wsel[0..W). sel: W entries of scratch.
// The bisection starts at a sum the W-th largest cannot be below: for ranks a, b with
// (a+1)(b+1) >= W, the (a+1)(b+1) pairs of ranks at most a and at most b all sum to at
// least lv0[a] + lv1[b].
template <int NC, int EW>
__device__ __forceinline__ void select_candidates(const float* lv0, const int* li0, const float* lv1,
                                                  const int* li1, const unsigned short* pairs, int C,
                                                  const unsigned char* fpart, int n, int W,
                                                  uint64_t* sel, int32_t* idx, float* wsel)
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
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    {
        // floor: the largest lv0[a] + lv1[ceil(W / (a+1)) - 1] over the ranks a < W (the
        // partner ranks from fpart)
        uint32_t fl = 0u;
        for (int a = lane; a < W; a += 32)
            fl = max(fl, float_order_bits(lv0[a] + lv1[fpart[a]]));
        kmin = max(kmin, __reduce_max_sync(0xFFFFFFFFu, fl));
        kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    }
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
    for (int i = 0; i < NC; ++i) {
        cv[i] = keep[i] ? expf(cv[i] - mx) : 0.0f;
        part += cv[i];
    }
    part = __reduce_add_sync_f(part);
    const float inv = 1.0f / part;   // (one division a query; a weight is within an ulp of
                                     // the quotient)
    // kept weights by position in sel (as floats); sort keys (slot << 6) | position (slots
    // below 2^18, positions below 64)
    float* selw = reinterpret_cast<float*>(sel);
    uint32_t k2[EW];
#pragma unroll
    for (int i = 0; i < EW; ++i)
        k2[i] = ~0u;
    int base_pos = 0;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep[i]);
        if (keep[i]) {
            const int pos = base_pos + __popc(bal & ((1u << lane) - 1u));
            selw[pos] = cv[i] * inv;
            reinterpret_cast<uint32_t*>(selw + 64)[pos] = (cs[i] << 6) | (uint32_t)pos;
        }
        base_pos += __popc(bal);
    }
    __syncwarp();
    // report the set in ascending slot order, weights alongside
#pragma unroll
    for (int i = 0; i < EW; ++i) {
        const int e = lane * EW + i;
        if (e < W)
            k2[i] = reinterpret_cast<const uint32_t*>(selw + 64)[e];
    }
    warp_bitonic_sort<EW>(k2);
#pragma unroll
    for (int i = 0; i < EW; ++i) {
        const int e = lane * EW + i;
        if (e < W) {
            idx[e] = (int32_t)(k2[i] >> 6);
            wsel[e] = selw[k2[i] & 63u];
        }
    }
}

// One warp per (token, kind). Candidate pairs (a, b) of half-ranks come from a table
// built in shared memory at block start.
template <int NC>
__global__ void __launch_bounds__(256, 4) candidate_select_kernel(
    const float* __restrict__ hv, const int32_t* __restrict__ hi, int64_t ntok, int n, int W,
    int32_t* __restrict__ idx, float* __restrict__ wsel)
{
    __shared__ unsigned short pairs[32 * NC];     // (a << 8) | b
    __shared__ int npairs;
    __shared__ float lv[8][2][64];
    __shared__ int li[8][2][64];
    __shared__ uint64_t sel[8][64];     // kept weights [64] and sort keys [64] a warp
    __shared__ unsigned char fpart[64]; // ceil(W / (a+1)) - 1: the floor's partner rank of a
    build_pairs(pairs, &npairs, W);
    if (threadIdx.x < W)
        fpart[threadIdx.x] = (unsigned char)((W + (int)threadIdx.x) / ((int)threadIdx.x + 1) - 1);
    __syncthreads();
    const int C = npairs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nq = 2 * ntok;
    for (int64_t qi = (int64_t)blockIdx.x * 8 + warp; qi < nq; qi += (int64_t)gridDim.x * 8) {
        const int kind = qi >= ntok ? 1 : 0;             // (qi < 2 ntok)
        const int64_t tok = kind ? qi - ntok : qi;
        const size_t base = ((size_t)kind * ntok + tok) * 2 * W;
        // each half's W best rows sorted by (score desc, row asc). The lists come in
        // ascending row order (the tensor-core scoring writes them so; the SIMT one
        // already sorted), so a sort on the score's descending order key with its 6 low
        // bits replaced by the list position keeps equal scores in row order. Only
        // scores that differ in those 6 bits alone can come out of order; a list where
        // that happened is sorted again on full (score, row) keys.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float* hvl = hv + base + h * W;
            const int32_t* hil = hi + base + h * W;
            uint32_t sk[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = lane * 2 + i;
                sk[i] = e < W ? ((~float_order_bits(hvl[e])) & ~63u) | (uint32_t)e : ~0u;
            }
            warp_bitonic_sort<2>(sk);
            float sv[2];
            int si[2];
            uint32_t ok[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = lane * 2 + i;
                const int src = e < W ? (int)(sk[i] & 63u) : 0;
                sv[i] = hvl[src];
                si[i] = hil[src];
                ok[i] = float_order_bits(sv[i]);
            }
            const uint32_t nxt = __shfl_down_sync(0xFFFFFFFFu, ok[0], 1);
            const bool bad = (lane * 2 + 1 < W && ok[0] < ok[1]) ||
                             (lane < 31 && lane * 2 + 2 < W && ok[1] < nxt);
            if (__any_sync(0xFFFFFFFFu, bad)) {
                uint64_t hk[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int e = lane * 2 + i;
                    hk[i] = e < W ? desc_key(hvl[e], (uint32_t)hil[e]) : ~0ull;
                }
                warp_bitonic_sort<2>(hk);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    sv[i] = key_score(hk[i]);
                    si[i] = (int)key_id(hk[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = lane * 2 + i;
                if (e < W) {
                    lv[warp][h][e] = sv[i];
                    li[warp][h][e] = si[i];
                }
            }
        }
        __syncwarp();
        const size_t ob = ((size_t)tok * 2 + kind) * W;
        select_candidates<NC, 2>(lv[warp][0], li[warp][0], lv[warp][1], li[warp][1], pairs, C, fpart,
                                 n, W, sel[warp], idx + ob, wsel + ob);
    }
}

// ------------------------------------- few tokens: a query's selection on a warp group

constexpr int kGW = 4;                 // warps a query group
constexpr int kGT = kGW * 32;          // threads a query group
constexpr int kKList = 40;             // entries of a group's bracket list (32 + the pick)

// A query group (kGW warps at named barrier `bar`) exchanging partial results through
// shared memory: xs holds two halves of kGW x 4 words, used in turn, so that one barrier
// per exchange suffices (a half is written again only after the barrier of the exchange
// in between, which every reader of its last use has passed).
struct Group {
    int bar;          // named barrier (1 + the group's index)
    int gw;           // warp within the group
    int tid;          // thread within the group
    uint32_t* xs;     // [2][kGW][4]
    int ph;           // the half the next exchange uses
};

__device__ __forceinline__ void grp_sync(const Group& g)
{
    asm volatile("bar.sync %0, %1;" ::"r"(g.bar), "n"(kGT) : "memory");
}

// this warp's words w[0..NV) into the exchange, then every thread reads all warps'
template <int NV>
__device__ __forceinline__ const uint32_t* grp_post(Group& g, const uint32_t (&w)[NV])
{
    uint32_t* x = g.xs + g.ph * kGW * 4;
    g.ph ^= 1;
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i)
            x[g.gw * 4 + i] = w[i];
    }
    grp_sync(g);
    return x;
}

// group sums of NV ints
template <int NV>
__device__ __forceinline__ void grp_sum(Group& g, int (&v)[NV])
{
    uint32_t w[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i)
        w[i] = (uint32_t)__reduce_add_sync(0xFFFFFFFFu, v[i]);
    const uint32_t* x = grp_post<NV>(g, w);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        int s = 0;
#pragma unroll
        for (int q = 0; q < kGW; ++q)
            s += (int)x[q * 4 + i];
        v[i] = s;
    }
}

// offset of this warp's c elements in the group's order (warps in turn) and the total
__device__ __forceinline__ int grp_offset(Group& g, int c, int& total)
{
    const uint32_t w[1] = {(uint32_t)c};
    const uint32_t* x = grp_post<1>(g, w);
    int off = 0;
    total = 0;
#pragma unroll
    for (int q = 0; q < kGW; ++q) {
        off += q < g.gw ? (int)x[q * 4] : 0;
        total += (int)x[q * 4];
    }
    return off;
}

// Exact top-W for a query group of kGW warps, NK elements a thread: order keys key[] (0: no
// element) with distinct ids id[]. Finds the W best elements by (key desc, id asc) from a
// bracket [lo, hi) that holds cnt_lo = #{key >= lo} >= W > cnt_hi = #{key >= hi}. Each
// round counts three probes over the group (one exchange): two where a count falling
// linearly in the score between the ends of the bracket would reach W, 12 elements'
// worth either side, and the middle of the key range, which at least halves it. It stops
// when exactly W keys lie at or above lo, or at most 32 in the bracket: those are gathered
// in list (kKList entries, warps in turn) and ranked by the group's first warp, and the
// e of the result is the (W - cnt_hi)-th of them. Should more than 32 share one key value,
// the same rank among their ids comes from a bisection over the ids.
template <int NK>
__device__ __forceinline__ KthSel group_kth(Group& g, const uint32_t (&key)[NK],
                                            const uint32_t (&id)[NK], int W, uint32_t lo,
                                            uint32_t hi, int cnt_lo, int cnt_hi, uint64_t* list)
{
    const int lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    auto count_ge = [&](uint32_t p) {
        int c = 0;
#pragma unroll
        for (int i = 0; i < NK; ++i)
            c += key[i] >= p ? 1 : 0;
        return c;
    };
    for (int round = 0; round < 40 && cnt_lo != W && cnt_lo - cnt_hi > 32 && hi - lo > 1; ++round) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        const float vlo = float_from_order_bits(lo), vhi = float_from_order_bits(hi);
        const float span = (float)(cnt_lo - cnt_hi);
        const float f = (float)(cnt_lo - W) / span, dl = 12.0f / span;
        const uint32_t pa = min(max(float_order_bits(vlo + (vhi - vlo) * (f - dl)), lo + 1), hi - 1);
        const uint32_t pb = min(max(float_order_bits(vlo + (vhi - vlo) * (f + dl)), lo + 1), hi - 1);
        int c[3] = {count_ge(pa), count_ge(pb), count_ge(mid)};
        grp_sum<3>(g, c);
        kth_narrow(pa, c[0], W, lo, hi, cnt_lo, cnt_hi);
        kth_narrow(pb, c[1], W, lo, hi, cnt_lo, cnt_hi);
        kth_narrow(mid, c[2], W, lo, hi, cnt_lo, cnt_hi);
    }
    KthSel r{cnt_lo == W, lo, 0ull};
    if (r.exact)
        return r;
    const int m = cnt_lo - cnt_hi, need = W - cnt_hi;
    if (m <= 32) {
        // the bracket's elements into list[0..m), warps in turn
        int at = 0;
        uint64_t mine[NK];
        int pos[NK];
#pragma unroll
        for (int i = 0; i < NK; ++i) {
            const bool in = key[i] >= lo && key[i] < hi;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
            pos[i] = in ? at + __popc(bal & below) : -1;
            mine[i] = comp_key(key[i], id[i]);
            at += __popc(bal);
        }
        int total = 0;
        const int off = grp_offset(g, at, total);
#pragma unroll
        for (int i = 0; i < NK; ++i)
            if (pos[i] >= 0)
                list[off + pos[i]] = mine[i];
        grp_sync(g);
        if (g.gw == 0) {
            // (a fixed trip count, so that the loads are issued together)
            const uint64_t e = lane < m ? list[lane] : ~0ull;
            int rank = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                rank += (j < m && list[j] < e) ? 1 : 0;
            const unsigned who = __ballot_sync(0xFFFFFFFFu, lane < m && rank == need - 1);
            const uint64_t pick = __shfl_sync(0xFFFFFFFFu, e, __ffs(who) - 1);
            if (lane == 0)
                list[32] = pick;
        }
        grp_sync(g);
        r.e = list[32];
        return r;
    }
    // more than 32 left, all with key lo: the need-th lowest id among them
    uint32_t ia = 0u, ib = 0xFFFFFFFFu;
    for (int round = 0; round < 33 && ia < ib; ++round) {
        const uint32_t md = ia + ((ib - ia) >> 1);
        int c[1] = {0};
#pragma unroll
        for (int i = 0; i < NK; ++i)
            c[0] += (key[i] == lo && id[i] <= md) ? 1 : 0;
        grp_sum<1>(g, c);
        if (c[0] >= need)
            ib = md;
        else
            ia = md + 1u;
    }
    r.e = comp_key(lo, ia);
    return r;
}

// the group's kept elements (keep[i]) into dst[0..), warps in turn; returns how many
template <int NK>
__device__ __forceinline__ int grp_compact(Group& g, const bool (&keep)[NK], const uint64_t (&val)[NK],
                                           uint64_t* dst)
{
    const int lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    int at = 0, pos[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) {
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep[i]);
        pos[i] = keep[i] ? at + __popc(bal & below) : -1;
        at += __popc(bal);
    }
    int total = 0;
    const int off = grp_offset(g, at, total);
#pragma unroll
    for (int i = 0; i < NK; ++i)
        if (pos[i] >= 0)
            dst[off + pos[i]] = val[i];
    grp_sync(g);
    return total;
}

// One query group: the W best of the n scores s[0..n) by (score desc, row asc), sorted,
// into lv[0..W) / li[0..W), NK scores a thread (rows tid + kGT i). The first bracket comes
// from probes around mean + z sd (the scores of a row are near normal; z is the standard
// normal quantile of 1 - W/n), checked by one counting pass; group_kth's search is exact
// either way. out: 64 entries, list: kKList entries of scratch.
template <int NK, int W>
__device__ __forceinline__ void group_topw(Group& g, const float* s, int n, float z, uint64_t* out,
                                           uint64_t* list, float* lv, int* li)
{
    uint32_t key[NK], id[NK];
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    float sum = 0.f, sum2 = 0.f;
#pragma unroll
    for (int i = 0; i < NK; ++i) {
        const int r = g.tid + kGT * i;
        const float f = r < n ? s[r] : 0.f;
        key[i] = r < n ? float_order_bits(f) : 0u;     // 0 is below every real key
        id[i] = (uint32_t)r;
        if (r < n) {
            kmin = min(kmin, key[i]);
            kmax = max(kmax, key[i]);
            sum += f;
            sum2 = fmaf(f, f, sum2);
        }
    }
    {
        const uint32_t w[4] = {__reduce_min_sync(0xFFFFFFFFu, kmin), __reduce_max_sync(0xFFFFFFFFu, kmax),
                               __float_as_uint(__reduce_add_sync_f(sum)),
                               __float_as_uint(__reduce_add_sync_f(sum2))};
        const uint32_t* x = grp_post<4>(g, w);
        sum = 0.f;
        sum2 = 0.f;
#pragma unroll
        for (int q = 0; q < kGW; ++q) {
            kmin = min(kmin, x[q * 4]);
            kmax = max(kmax, x[q * 4 + 1]);
            sum += __uint_as_float(x[q * 4 + 2]);
            sum2 += __uint_as_float(x[q * 4 + 3]);
        }
    }
    uint32_t lo = kmin, hi = kmax + 1u;
    int cnt_lo = n, cnt_hi = 0;
    {
        // four probes, mean + (z -+ 1/2) sd and mean + (z -+ 1/10) sd: the W-th score lies
        // within 1/10 sd of mean + z sd more often than not, and then at most about 20
        // scores lie between the inner two, few enough to rank at once
        const float mean = sum / n;
        const float sd = sqrtf(fmaxf(sum2 / n - mean * mean, 0.f));
        uint32_t pb[4];
        const float off[4] = {-0.5f, -0.1f, 0.1f, 0.5f};
        int c[4] = {0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            pb[q] = float_order_bits(mean + (z + off[q]) * sd);
#pragma unroll
            for (int i = 0; i < NK; ++i)
                c[q] += key[i] >= pb[q] ? 1 : 0;
        }
        grp_sum<4>(g, c);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            kth_narrow(pb[q], c[q], W, lo, hi, cnt_lo, cnt_hi);
    }
    const KthSel ks = group_kth<NK>(g, key, id, W, lo, hi, cnt_lo, cnt_hi, list);
    bool keep[NK];
    uint64_t ck[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) {
        ck[i] = comp_key(key[i], id[i]);
        keep[i] = key[i] != 0u && (ks.exact ? key[i] >= ks.lo : ck[i] <= ks.e);
    }
    grp_compact<NK>(g, keep, ck, out);
    // in order of (score desc, row asc): each entry's place is the number before it
    if (g.tid < W) {
        const uint64_t e = out[g.tid];
        int place = 0;
#pragma unroll
        for (int j = 0; j < W; ++j)
            place += out[j] < e ? 1 : 0;
        lv[place] = key_score(e);
        li[place] = (int)key_id(e);
    }
    grp_sync(g);
}

// One query group: select_candidates' merge, NC candidates a thread (candidate tid + kGT i);
// the softmax normaliser is summed in a fixed order (each warp's butterfly, then the warps
// in turn). sel: 64 entries, list: kKList entries of scratch.
template <int NC, int W>
__device__ __forceinline__ void group_merge(Group& g, const float* lv0, const int* li0, const float* lv1,
                                            const int* li1, const unsigned short* pairs, int C, int n,
                                            uint64_t* sel, uint64_t* list, int32_t* idx, float* wsel)
{
    uint32_t ck[NC], cs[NC];
    float cv[NC];
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = g.tid + kGT * i;
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
    {
        const uint32_t w[2] = {__reduce_min_sync(0xFFFFFFFFu, kmin), __reduce_max_sync(0xFFFFFFFFu, kmax)};
        const uint32_t* x = grp_post<2>(g, w);
#pragma unroll
        for (int q = 0; q < kGW; ++q) {
            kmin = min(kmin, x[q * 4]);
            kmax = max(kmax, x[q * 4 + 1]);
        }
    }
    const KthSel ks = group_kth<NC>(g, ck, cs, W, kmin, kmax + 1u, C, 0, list);
    // softmax over the kept sums (the largest one is the largest of all)
    const float mx = float_from_order_bits(kmax);
    bool keep[NC];
    float ev[NC];
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        keep[i] = ck[i] != 0u && (ks.exact ? ck[i] >= ks.lo : comp_key(ck[i], cs[i]) <= ks.e);
        ev[i] = keep[i] ? expf(cv[i] - mx) : 0.0f;
        part += ev[i];
    }
    {
        const uint32_t w[1] = {__float_as_uint(__reduce_add_sync_f(part))};
        const uint32_t* x = grp_post<1>(g, w);
        part = 0.0f;
#pragma unroll
        for (int q = 0; q < kGW; ++q)
            part += __uint_as_float(x[q * 4]);
    }
    uint64_t val[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i)
        val[i] = ((uint64_t)cs[i] << 32) | __float_as_uint(keep[i] ? ev[i] / part : 0.0f);
    grp_compact<NC>(g, keep, val, sel);
    // the set in ascending slot order, weights alongside
    if (g.tid < W) {
        const uint64_t e = sel[g.tid];
        int place = 0;
#pragma unroll
        for (int j = 0; j < W; ++j)
            place += sel[j] < e ? 1 : 0;
        idx[place] = (int32_t)(e >> 32);
        wsel[place] = __uint_as_float((uint32_t)e);
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
    uint32_t rs, ktab, qs, sc, lv, li, lv1, li1, hk, kl, xs, total;
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
    L.kl = o; o += kQG * kKList * 8;
    L.xs = o; o += kQG * 2 * kGW * 4 * 4;
    L.total = o;
    return L;
}

// Few tokens (a decode step): a cluster of two blocks takes kQG queries (token, kind),
// block 0 the first half of each query against K1, block 1 the second against K2:
//  1. the block stages its sub-key table in shared memory with one bulk copy a row;
//  2. it waits for the kernel before it (the projections, when launched early: the table
//     copy then overlaps them) and loads its queries' halves with plain loads;
//  3. the scores s[r] = <K[r], q_half>, fp32 sums of exact products: bf16 tables whose
//     half-width is a multiple of 16 on the tensor cores (mma.sync m16n8k16, the table as
//     A in 16-row tiles, the kQG queries padded to 8 as B), others on the SIMT cores
//     (thread t takes row t, its 16-byte chunks in a rotated order, products in element
//     order);
//  4. warp group j (warps 4j .. 4j+3) keeps query j's W best rows of this half
//     (group_topw);
//  5. after a cluster barrier, block 0's group j reads block 1's list of query j through
//     distributed shared memory and merges the two as the candidate kernel does, on the
//     group (group_merge): the set and its softmax weights.
constexpr int kSmallThreads = 512;

template <typename IO, int NC, int KPL>
__global__ void __launch_bounds__(kSmallThreads) address_small_kernel(
    const IO* __restrict__ q_w, const IO* __restrict__ q_r, const IO* __restrict__ K1,
    const IO* __restrict__ K2, int64_t ntok, int dk, int n, int W, float z,
    int32_t* __restrict__ idx, float* __restrict__ wsel, int* status, uint32_t* clear,
    long long clear_words)
{
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ unsigned short pairs[32 * NC];
    __shared__ int npairs;
    __shared__ __align__(8) uint64_t kbar;
    const int warp = threadIdx.x >> 5;
    // the set size, fixed by the candidate count a lane the launch picked
    constexpr int WC = NC == 9 ? 64 : NC == 4 ? 32 : NC == 2 ? 16 : 8;
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
    // 1. the half's sub-key table (one bulk copy a row, issued by every thread)
    if (threadIdx.x == 0)
        mbar_arrive_expect_tx(smem_u32(&kbar), tbytes);
    __syncthreads();
    {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(half ? K2 : K1);
        for (int r = threadIdx.x; r < n; r += blockDim.x)
            bulk_g2s(base + L.ktab + (uint32_t)(r * rs), src + (size_t)r * rowb, (uint32_t)rowb,
                     smem_u32(&kbar));
        // rows of the last 16-row tile past the table: zero (read by the MMA, never kept)
        for (int e = threadIdx.x; e < ((n + 15) / 16 * 16 - n) * h; e += blockDim.x)
            reinterpret_cast<IO*>(sm + L.ktab + (n + e / h) * rs)[e % h] = IO(0.0f);
    }
    build_pairs(pairs, &npairs, W);
    __syncthreads();
    bool ok = mbar_wait(smem_u32(&kbar), 0, nullptr, status);
    ok = __syncthreads_and(ok) != 0;
    // 2. the queries' halves (rows kQG..7 zero), once the projections that write them
    //    are done (a programmatic launch starts before)
    griddep_wait();
    griddep_launch();
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < clear_words;
         e += (long long)gridDim.x * blockDim.x)
        clear[e] = 0u;
    {
        // 16-byte pieces: a query half is a whole number of them on this path ((h * es) %
        // 16 == 0) and the q buffers are 16-byte aligned, so every piece is too; one load
        // a thread, all in flight together
        const int pieces = rowb / 16;
        for (int e = threadIdx.x; e < 8 * pieces; e += blockDim.x) {
            const int j = e / pieces, k = e - j * pieces;
            const int64_t qi = q0 + j;                      // token-major: tok * 2 + kind
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (j < kQG && qi < nq)
                val = reinterpret_cast<const uint4*>(((qi & 1) ? q_r : q_w) + (qi >> 1) * dk + half * h)[k];
            *reinterpret_cast<uint4*>(sm + L.qs + j * rs + k * 16) = val;
        }
    }
    ok = __syncthreads_and(ok) != 0;
    // 3. scores of this half
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
    // 4. query j's W best rows of this half, on warp group j
    const int grp = warp / kGW;
    Group g{1 + grp, warp % kGW, (int)threadIdx.x - grp * kGT,
            reinterpret_cast<uint32_t*>(sm + L.xs) + grp * 2 * kGW * 4, 0};
    uint64_t* gout = reinterpret_cast<uint64_t*>(sm + L.hk) + grp * 64;
    uint64_t* glist = reinterpret_cast<uint64_t*>(sm + L.kl) + grp * kKList;
    constexpr int KPG = KPL >= 4 ? KPL / 4 : 1;      // scores a thread of the group
    if (ok && grp < kQG && q0 + grp < nq)
        group_topw<KPG, WC>(g, sc + grp * 32 * KPL, n, z, gout, glist, lv + grp * 64, li + grp * 64);
    __syncthreads();
    cluster_sync_all();
    // 5. block 0 merges each query's halves: group j reads block 1's list of query j
    if (ok && half == 0 && grp < kQG && q0 + grp < nq) {
        float* lv1 = reinterpret_cast<float*>(sm + L.lv1) + grp * 64;
        int* li1 = reinterpret_cast<int*>(sm + L.li1) + grp * 64;
        if (g.tid < W) {
            lv1[g.tid] = __uint_as_float(ld_dsmem_u32(base + L.lv + (grp * 64 + g.tid) * 4, 1));
            li1[g.tid] = (int)ld_dsmem_u32(base + L.li + (grp * 64 + g.tid) * 4, 1);
        }
        grp_sync(g);
        const int64_t qi = q0 + grp;
        const size_t ob = ((size_t)(qi >> 1) * 2 + (qi & 1)) * W;
        group_merge<(NC + 3) / 4, WC>(g, lv + grp * 64, li + grp * 64, lv1, li1, pairs, npairs, n,
                                      gout, glist, idx + ob, wsel + ob);
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

template <int NC>
static cudaError_t run_cand(const sdm_cfg& c, int64_t ntok, const float* hv, const int32_t* hi,
                            int32_t* idx, float* wsel, cudaStream_t s)
{
    const int sms = num_sms_current_device();
    int64_t blocks = (2 * ntok + 7) / 8;
    if (blocks > (int64_t)sms * 4)
        blocks = (int64_t)sms * 4;
    candidate_select_kernel<NC><<<(unsigned)blocks, 256, 0, s>>>(hv, hi, ntok, c.n_sub, c.w,
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

template <typename IO, int NC, int KPL>
static cudaError_t run_small_kpl(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                                 const void* q_r, int64_t ntok, int32_t* idx, float* wsel,
                                 int* status, cudaStream_t s, bool early, void* clear,
                                 size_t clear_bytes)
{
    auto kern = address_small_kernel<IO, NC, KPL>;
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 2 : 1;
    const float z = normal_upper_quantile((double)c.w / c.n_sub);
    return cudaLaunchKernelEx(&cfg, kern, (const IO*)q_w, (const IO*)q_r, (const IO*)K1,
                              (const IO*)K2, ntok, c.dk, c.n_sub, c.w, z, idx, wsel, status,
                              (uint32_t*)clear, (long long)(clear_bytes / 4));
}

template <typename IO, int NC>
static cudaError_t run_small_k(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                               const void* q_r, int64_t ntok, int32_t* idx, float* wsel,
                               int* status, cudaStream_t s, bool early, void* clear,
                               size_t clear_bytes)
{
    switch (small_kpl(c.n_sub)) {
    case 1: return run_small_kpl<IO, NC, 1>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early,
                                             clear, clear_bytes);
    case 2: return run_small_kpl<IO, NC, 2>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early,
                                             clear, clear_bytes);
    case 4: return run_small_kpl<IO, NC, 4>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early,
                                             clear, clear_bytes);
    case 8: return run_small_kpl<IO, NC, 8>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early,
                                             clear, clear_bytes);
    default: return run_small_kpl<IO, NC, 16>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early,
                                              clear, clear_bytes);
    }
}

template <typename IO>
static cudaError_t run_small(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                             const void* q_r, int64_t ntok, int32_t* idx, float* wsel,
                             int* status, cudaStream_t s, bool early, void* clear,
                             size_t clear_bytes)
{
    switch (c.w) {
    case 8: return run_small_k<IO, 1>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early, clear,
                                       clear_bytes);
    case 16: return run_small_k<IO, 2>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early, clear,
                                       clear_bytes);
    case 32: return run_small_k<IO, 4>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early, clear,
                                       clear_bytes);
    case 64: return run_small_k<IO, 9>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early, clear,
                                       clear_bytes);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_address(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                           const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                           int* status, cudaStream_t s, bool early, void* clear,
                           size_t clear_bytes)
{
    if (ntok <= 0)
        return clear_bytes > 0 ? cudaMemsetAsync(clear, 0, clear_bytes, s) : cudaSuccess;
    if (address_small_path(c, ntok))
        return c.dtype == SDM_BF16
                   ? run_small<bf16>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early, clear,
                                     clear_bytes)
                   : run_small<float>(c, K1, K2, q_w, q_r, ntok, idx, wsel, status, s, early, clear,
                                      clear_bytes);
    if (clear_bytes > 0) {
        const cudaError_t ec = cudaMemsetAsync(clear, 0, clear_bytes, s);
        if (ec != cudaSuccess)
            return ec;
    }
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
    case 8: return run_cand<1>(c, ntok, hv, hi, idx, wsel, s);      // 20 candidates
    case 16: return run_cand<2>(c, ntok, hv, hi, idx, wsel, s);     // 50
    case 32: return run_cand<4>(c, ntok, hv, hi, idx, wsel, s);     // 119
    case 64: return run_cand<9>(c, ntok, hv, hi, idx, wsel, s);     // 280
    default: (void)C; return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
