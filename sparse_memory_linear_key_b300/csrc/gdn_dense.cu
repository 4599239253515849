// gdn_dense.cu -- the dense-state comparator: the same gated delta rule on a state of W
// columns that every token updates ("Sparse Delta Memory" blog, "Background" and "How
// does SDM work?": SDM's 64 active slot vectors per token are exactly the size of a
// gated-delta-net's whole dense state, at identical FLOPs per token; the difference is
// the state the active vectors are drawn from).
//
// Per sequence, state S [d][W] fp32 (column j plays slot j), per token t with write
// weights k [W], read weights r [W], value v [d], gates alpha, beta:
//   u = S k;  S <- alpha S + beta (v - alpha u) k^T;  y = S r      (fp32 throughout)
// Rows are independent, so a row's W columns live in the registers of four threads (16
// columns each) for the whole sequence; u and y are summed over the four by shuffles.
// Nothing but the per-token inputs and y crosses HBM: the block stages 32 tokens of
// weights, gates and its rows of v in shared memory (cp.async, double-buffered) while
// it computes the previous 32.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kGdnCols = 64;                  // W: the dense state's columns
constexpr int kGdnPer = 16;                   // columns a thread
constexpr int kGdnTpr = kGdnCols / kGdnPer;   // threads a row
constexpr int kGdnRows = 32;                  // rows a block
constexpr int kGdnThreads = kGdnRows * kGdnTpr;
constexpr int kGdnChunk = 32;                 // tokens staged in shared memory at a time

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <typename IO>
struct GdnStage {
    float kr[kGdnChunk][2][kGdnCols];   // write weights, then read weights
    IO v[kGdnChunk][kGdnRows];          // this block's rows of v
    float ab[kGdnChunk][2];             // alpha, beta
};

__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

// sum over the kGdnTpr threads of a row (adjacent lanes)
__device__ __forceinline__ float row_sum(float x)
{
#pragma unroll
    for (int o = 1; o < kGdnTpr; o <<= 1)
        x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

// Stage tokens [t0, t0 + n) of sequence b: weights and v by 16-byte cp.async, gates by
// plain loads (their base need not be 16-byte aligned).
template <typename IO>
__device__ __forceinline__ void gdn_stage(GdnStage<IO>& st, const float* kw, const float* kr,
                                          int64_t ks, const IO* v, const float* alpha,
                                          const float* beta, int64_t tok0, int t0, int n, int d,
                                          int row0)
{
    const int tid = threadIdx.x;
    // weights: n tokens x 2 kinds x 16 pieces of 16 bytes
    for (int e = tid; e < n * 2 * (kGdnCols / 4); e += kGdnThreads) {
        const int t = e / (2 * (kGdnCols / 4));
        const int kind = (e / (kGdnCols / 4)) & 1;
        const int q = e % (kGdnCols / 4);
        const float* src = (kind ? kr : kw) + (tok0 + t0 + t) * ks + q * 4;
        cp_async16(smem_u32(&st.kr[t][kind][q * 4]), src);
    }
    // v: n tokens x this block's rows, in 16-byte pieces
    constexpr int VP = kGdnRows * (int)sizeof(IO) / 16;   // pieces a token
    for (int e = tid; e < n * VP; e += kGdnThreads) {
        const int t = e / VP, q = e % VP;
        const int r = row0 + q * (16 / (int)sizeof(IO));
        if (r >= d)   // d is a multiple of 16 rows: a piece is all in or all out
            continue;
        cp_async16(smem_u32(&st.v[t][q * (16 / (int)sizeof(IO))]), v + (tok0 + t0 + t) * d + r);
    }
    for (int t = tid; t < n; t += kGdnThreads) {
        st.ab[t][0] = __ldg(alpha + tok0 + t0 + t);
        st.ab[t][1] = __ldg(beta + tok0 + t0 + t);
    }
}

// grid (d / 32, B); thread (row = blockIdx.x * 32 + tid / 4, column group tid % 4)
template <typename IO>
__global__ void __launch_bounds__(kGdnThreads) gdn_dense_kernel(const float* __restrict__ S0,
                                                                 const float* __restrict__ kw,
                                                                 const float* __restrict__ kr,
                                                                 int64_t ks, const IO* __restrict__ v,
                                                                 const float* __restrict__ alpha,
                                                                 const float* __restrict__ beta,
                                                                 float* __restrict__ S_out,
                                                                 float* __restrict__ y, int T, int d)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    GdnStage<IO>* stage = reinterpret_cast<GdnStage<IO>*>(smem_raw);   // [2]
    const int b = blockIdx.y;
    const int row0 = blockIdx.x * kGdnRows;
    const int lr = (int)threadIdx.x / kGdnTpr, row = row0 + lr;
    const int cg = threadIdx.x % kGdnTpr;
    // d is a multiple of 16 and a warp holds 8 rows: a warp is all in or all out, and
    // every thread still takes part in the staging and the block barriers
    const bool act = row < d;
    float2 s[kGdnPer / 2];
    const int64_t so = ((int64_t)b * d + row) * kGdnCols + cg * kGdnPer;
#pragma unroll
    for (int q = 0; q < kGdnPer / 4; ++q) {
        const float4 x = act && S0 != nullptr ? __ldg(reinterpret_cast<const float4*>(S0 + so) + q)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
        s[2 * q] = make_float2(x.x, x.y);
        s[2 * q + 1] = make_float2(x.z, x.w);
    }
    const int64_t tok0 = (int64_t)b * T;
    const int nchunks = (T + kGdnChunk - 1) / kGdnChunk;
    if (nchunks > 0)
        gdn_stage(stage[0], kw, kr, ks, v, alpha, beta, tok0, 0, min(kGdnChunk, T), d, row0);
    cp_async_commit();
    for (int c = 0; c < nchunks; ++c) {
        const int n = min(kGdnChunk, T - c * kGdnChunk);
        if (c + 1 < nchunks)
            gdn_stage(stage[(c + 1) & 1], kw, kr, ks, v, alpha, beta, tok0, (c + 1) * kGdnChunk,
                      min(kGdnChunk, T - (c + 1) * kGdnChunk), d, row0);
        cp_async_commit();
        cp_async_wait_one();   // chunk c has landed (chunk c + 1 may be in flight)
        __syncthreads();
        const GdnStage<IO>& st = stage[c & 1];
        if (act) {
            // unrolled so that a token's read (y) overlaps the next token's u
#pragma unroll 4
            for (int t = 0; t < n; ++t) {
                const float4* kk = reinterpret_cast<const float4*>(&st.kr[t][0][cg * kGdnPer]);
                const float4* rr = reinterpret_cast<const float4*>(&st.kr[t][1][cg * kGdnPer]);
                float4 k4[kGdnPer / 4];
#pragma unroll
                for (int q = 0; q < kGdnPer / 4; ++q)
                    k4[q] = kk[q];
                // u = S k over this thread's columns, two accumulators, then over the row's threads
                float2 ua = make_float2(0.f, 0.f), ub = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < kGdnPer / 4; ++q) {
                    ua = __ffma2_rn(s[2 * q], make_float2(k4[q].x, k4[q].y), ua);
                    ub = __ffma2_rn(s[2 * q + 1], make_float2(k4[q].z, k4[q].w), ub);
                }
                const float u = row_sum(ua.x + ua.y + ub.x + ub.y);
                const float al = st.ab[t][0], be = st.ab[t][1];
                const float cc = be * (to_f(st.v[t][lr]) - al * u);
                const float2 al2 = make_float2(al, al), c2 = make_float2(cc, cc);
                // S <- alpha S + c k^T, then y = S r
                float2 ya = make_float2(0.f, 0.f), yb = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < kGdnPer / 4; ++q) {
                    const float4 r4 = rr[q];
                    s[2 * q] = __ffma2_rn(c2, make_float2(k4[q].x, k4[q].y), __fmul2_rn(al2, s[2 * q]));
                    s[2 * q + 1] =
                        __ffma2_rn(c2, make_float2(k4[q].z, k4[q].w), __fmul2_rn(al2, s[2 * q + 1]));
                    ya = __ffma2_rn(s[2 * q], make_float2(r4.x, r4.y), ya);
                    yb = __ffma2_rn(s[2 * q + 1], make_float2(r4.z, r4.w), yb);
                }
                const float yv = row_sum(ya.x + ya.y + yb.x + yb.y);
                if (cg == 0)
                    __stcs(y + (tok0 + c * kGdnChunk + t) * d + row, yv);
            }
        }
        __syncthreads();   // the buffer is refilled by the next iteration's staging
    }
    cp_async_wait_all();
    if (act && S_out != nullptr) {
#pragma unroll
        for (int q = 0; q < kGdnPer / 4; ++q)
            reinterpret_cast<float4*>(S_out + so)[q] =
                make_float4(s[2 * q].x, s[2 * q].y, s[2 * q + 1].x, s[2 * q + 1].y);
    }
}

}  // namespace

cudaError_t launch_gdn_dense(bool bf_io, const float* S0, const float* kw, const float* kr,
                             int64_t ks, const void* v, const float* alpha, const float* beta,
                             float* S_out, float* y, int B, int T, int d, cudaStream_t s)
{
    if (B <= 0 || d <= 0)
        return cudaSuccess;
    const dim3 grid((unsigned)((d + kGdnRows - 1) / kGdnRows), (unsigned)B);
    if (bf_io)
        gdn_dense_kernel<bf16><<<grid, kGdnThreads, 2 * sizeof(GdnStage<bf16>), s>>>(
            S0, kw, kr, ks, (const bf16*)v, alpha, beta, S_out, y, T, d);
    else
        gdn_dense_kernel<float><<<grid, kGdnThreads, 2 * sizeof(GdnStage<float>), s>>>(
            S0, kw, kr, ks, (const float*)v, alpha, beta, S_out, y, T, d);
    return cudaGetLastError();
}

}  // namespace sdm
