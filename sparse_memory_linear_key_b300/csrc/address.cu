// address.cu -- product-key addressing of every token, run up front because it
// depends only on the input ("Sparse Delta Memory" blog, "Write & Read": two sub-keys
// -> outer sum -> top-k; softmax-weighted).
//
//   score_tc_kernel        (score_tc.cu) s_h = K_h q_h for both halves of both queries
//                          on the tensor cores, and the top-W of each half (bf16 layers)
//   subkey_topw_kernel     the same on the SIMT cores in fp32 (fp32 layers and shapes
//                          the tensor path does not take), lists sorted
//                          (score desc, row asc)
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
    // pairs (a, b) with (a+1)(b+1) <= W, row a's run starting after the runs of rows < a
    if (threadIdx.x < W) {
        const int a = threadIdx.x;
        int start = 0;
        for (int a2 = 0; a2 < a; ++a2)
            start += W / (a2 + 1);
        for (int b = 0; b < W / (a + 1); ++b)
            pairs[start + b] = (unsigned short)((a << 8) | b);
        if (a == W - 1)
            npairs = start + W / (a + 1);
    }
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
        // The W largest candidate sums by (sum desc, slot asc): bisection over the
        // order-preserving keys of the sums (NC candidates a lane), stopping once exactly W
        // keys lie at or above the probe; equal sums at the threshold go to the lower slot.
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
                cv[i] = lv[warp][0][a] + lv[warp][1][b];
                cs[i] = (uint32_t)li[warp][0][a] * (uint32_t)n + (uint32_t)li[warp][1][b];
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
                sel[warp][pos] = ((uint64_t)cs[i] << 32) | __float_as_uint(expf(cv[i] - mx) / part);
            }
            base_pos += __popc(bal);
        }
        __syncwarp();
        // report the set in ascending slot order, weights alongside
        uint64_t k2[EW];
#pragma unroll
        for (int i = 0; i < EW; ++i) {
            const int e = lane * EW + i;
            k2[i] = (e < W) ? sel[warp][e] : ~0ull;
        }
        warp_bitonic_sort<EW>(k2);
        const size_t ob = ((size_t)tok * 2 + kind) * W;
#pragma unroll
        for (int i = 0; i < EW; ++i) {
            const int e = lane * EW + i;
            if (e < W) {
                idx[ob + e] = (int32_t)(k2[i] >> 32);
                wsel[ob + e] = __uint_as_float((uint32_t)k2[i]);
            }
        }
    }
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

cudaError_t launch_address(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                           const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                           int* status, cudaStream_t s)
{
    if (ntok <= 0)
        return cudaSuccess;
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
