// address.cu -- product-key addressing of every token, run up front because it
// depends only on the input ("Sparse Delta Memory" blog, "Write & Read": two sub-keys
// -> outer sum -> top-k; softmax-weighted).
//
//   score_tc_kernel        (score_tc.cu) s_h = K_h q_h for both halves of both queries
//                          on the tensor cores, and the top-W of each half (bf16 layers)
//   subkey_topw_kernel     the same on the SIMT cores in fp32 (fp32 layers and shapes
//                          the tensor path does not take), lists sorted
//                          (score desc, row asc)
//   candidate_select_kernel  sorts each half's list, then outer sums of the pairs of
//                          half-ranks (a, b) with
//                          (a+1)(b+1) <= W -- the only pairs that can reach the top-W
//                          of all n^2 sums -- their top-W, softmax, and the set in
//                          ascending slot order.
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
template <int EC, int EW, int EH>
__global__ void __launch_bounds__(256) candidate_select_kernel(
    const float* __restrict__ hv, const int32_t* __restrict__ hi, int64_t ntok, int n, int W,
    int32_t* __restrict__ idx, float* __restrict__ wsel)
{
    __shared__ unsigned short pairs[32 * EC];     // (a << 8) | b
    __shared__ int npairs;
    __shared__ float lv[8][2][64];
    __shared__ int li[8][2][64];
    __shared__ uint64_t sel[8][64];
    if (threadIdx.x == 0) {
        int c = 0;
        for (int a = 0; a < W; ++a)
            for (int b = 0; (a + 1) * (b + 1) <= W; ++b)
                pairs[c++] = (unsigned short)((a << 8) | b);
        npairs = c;
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
        uint64_t key[EC];
#pragma unroll
        for (int i = 0; i < EC; ++i) {
            const int c = lane * EC + i;
            if (c < C) {
                const int a = pairs[c] >> 8, b = pairs[c] & 0xFF;
                const float s = lv[warp][0][a] + lv[warp][1][b];
                const uint32_t slot = (uint32_t)li[warp][0][a] * (uint32_t)n + (uint32_t)li[warp][1][b];
                key[i] = desc_key(s, slot);
            } else {
                key[i] = ~0ull;
            }
        }
        warp_bitonic_sort<EC>(key);
        // softmax over the W kept scores (elements 0..W-1); element 0 is the max
        const float mx = __shfl_sync(0xFFFFFFFFu, key_score(key[0]), 0);
        float ex[EC];
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < EC; ++i) {
            const int e = lane * EC + i;
            ex[i] = (e < W) ? expf(key_score(key[i]) - mx) : 0.0f;
            part += ex[i];
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1)
            part += __shfl_xor_sync(0xFFFFFFFFu, part, m);
#pragma unroll
        for (int i = 0; i < EC; ++i) {
            const int e = lane * EC + i;
            if (e < W)
                sel[warp][e] = ((uint64_t)key_id(key[i]) << 32) | __float_as_uint(ex[i] / part);
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

template <int EC, int EW, int EH>
static cudaError_t run_cand(const sdm_cfg& c, int64_t ntok, const float* hv, const int32_t* hi,
                            int32_t* idx, float* wsel, cudaStream_t s)
{
    const int sms = num_sms_current_device();
    int64_t blocks = (2 * ntok + 7) / 8;
    if (blocks > (int64_t)sms * 4)
        blocks = (int64_t)sms * 4;
    candidate_select_kernel<EC, EW, EH><<<(unsigned)blocks, 256, 0, s>>>(hv, hi, ntok, c.n_sub, c.w,
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
    case 64: return run_cand<16, 2, 2>(c, ntok, hv, hi, idx, wsel, s);    // 280
    default: (void)C; return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
