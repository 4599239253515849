// addr_bwd.cu -- backward of the product-key addressing and of the projections
// ("Sparse Delta Memory" blog, "Write & Read": two sub-keys -> outer sum -> top-k,
// softmax weights; the addressing is learned end to end, paper Abstract).
//
// The top-W selection is piecewise constant, so the gradient flows through the kept
// pairs only. Per token and kind (write / read) with kept weights w_j = softmax(c)_j,
// c_j = s1[i_j] + s2[l_j] (slot i_j * n + l_j) and incoming gradients dw_j:
//   dc_j = w_j (dw_j - sum_m w_m dw_m),   ds1[i_j] += dc_j,   ds2[l_j] += dc_j.
// The score gradients go into dense rows DS_h [kind * ntok + tok][n]; then, with
// s_h = K_h q_h (q_h the half of q), two plain GEMMs per half:
//   dq_h = DS_h K_h        ([ntok, n] x [n, dk/2], per kind)
//   dK_h = DS_h^T Q_h      ([n, 2 ntok] x [2 ntok, dk/2], both kinds)
// run by cuBLAS in strict fp32 on fp32 copies of q and the sub-keys.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(float x) { return x; }

// dst [total] fp32 <- src [total] (both contiguous). vec: both 16-byte aligned, and a
// thread converts eight elements a step with 16- and 32-byte accesses; the tail (and
// every element without vec) one by one.
template <typename IO>
__global__ void __launch_bounds__(256) widen_kernel(const IO* __restrict__ src, int64_t total,
                                                    float* __restrict__ dst, bool vec)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nv = vec ? total / 8 : 0;
    for (int64_t v = i0; v < nv; v += stride) {
        float f[8];
        if constexpr (sizeof(IO) == 2) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(src) + v);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);           // bf16 -> fp32: exact
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
            const float4 a = __ldg(reinterpret_cast<const float4*>(src) + 2 * v);
            const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 2 * v + 1);
            f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
            f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        }
        float4* d = reinterpret_cast<float4*>(dst) + 2 * v;
        d[0] = make_float4(f[0], f[1], f[2], f[3]);
        d[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    for (int64_t e = nv * 8 + i0; e < total; e += stride)
        dst[e] = to_f32(src[e]);
}

// one warp per (kind, token): softmax backward over the W kept pairs, scattered into the
// dense score-gradient rows of both halves
__global__ void __launch_bounds__(256) select_bwd_kernel(const int32_t* __restrict__ idx,
                                                         const float* __restrict__ wsel,
                                                         const float* __restrict__ dwsel,
                                                         int64_t ntok, int W, int n,
                                                         float* __restrict__ ds1,
                                                         float* __restrict__ ds2)
{
    const int lane = threadIdx.x & 31;
    const int64_t q = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // kind * ntok + tok
    if (q >= 2 * ntok)
        return;   // whole warps
    const int kind = q >= ntok ? 1 : 0;                 // (q < 2 ntok)
    const int64_t tok = kind ? q - ntok : q;
    const size_t base = ((size_t)tok * 2 + kind) * W;
    float sum = 0.f;
    for (int j = lane; j < W; j += 32)
        sum = fmaf(__ldg(wsel + base + j), __ldg(dwsel + base + j), sum);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    float* r1 = ds1 + (size_t)q * n;
    float* r2 = ds2 + (size_t)q * n;
    for (int j = lane; j < W; j += 32) {
        const int32_t s = __ldg(idx + base + j);
        if (s < 0 || s >= n * n)
            continue;
        const float dc = __ldg(wsel + base + j) * (__ldg(dwsel + base + j) - sum);
        atomicAdd(r1 + s / n, dc);   // pairs of one token may share a row or a column
        atomicAdd(r2 + s % n, dc);
    }
}

unsigned grid_for(int64_t work)
{
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)num_sms_current_device() * 8;
    if (blocks > cap)
        blocks = cap;
    return (unsigned)(blocks < 1 ? 1 : blocks);
}

struct AddrBwdWs {
    size_t ds, qf, kf, total;
};

AddrBwdWs addr_bwd_layout(const sdm_cfg& c, int64_t ntok)
{
    AddrBwdWs L;
    const size_t n = (size_t)c.n_sub, h = (size_t)c.dk / 2;
    size_t o = 0;
    L.ds = o; o += ((2 * 2 * (size_t)ntok * n * 4) + 255) / 256 * 256;   // [2 halves][2 ntok][n]
    L.qf = o; o += ((2 * (size_t)ntok * c.dk * 4) + 255) / 256 * 256;    // [2 ntok][dk]
    L.kf = o; o += ((2 * n * h * 4) + 255) / 256 * 256;                  // [2 halves][n][h]
    L.total = o;
    return L;
}

template <typename IO>
cudaError_t widen(const void* src, int64_t rows, int cols, float* dst, cudaStream_t s)
{
    const int64_t total = rows * cols;
    const bool vec = (((uintptr_t)src | (uintptr_t)dst) & 15u) == 0;
    widen_kernel<IO><<<grid_for(vec ? (total + 7) / 8 : total), 256, 0, s>>>((const IO*)src, total,
                                                                              dst, vec);
    return cudaGetLastError();
}

}  // namespace

size_t address_backward_ws_bytes(const sdm_cfg& c, int64_t ntok)
{
    return addr_bwd_layout(c, ntok).total;
}

int launch_address_backward(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                            const void* q_r, int64_t ntok, const int32_t* idx, const float* wsel,
                            const float* dwsel, float* dq_w, float* dq_r, float* dK1, float* dK2,
                            void* ws, cudaStream_t s)
{
    if (ntok <= 0)
        return SDM_OK;
    if (2 * ntok > 0x7FFFFFFF)
        return SDM_EUNSUPPORTED;
    const AddrBwdWs L = addr_bwd_layout(c, ntok);
    const int n = c.n_sub, h = c.dk / 2, dk = c.dk;
    char* base = (char*)ws;
    float* ds1 = (float*)(base + L.ds);
    float* ds2 = ds1 + 2 * (size_t)ntok * n;
    float* qf = (float*)(base + L.qf);
    float* k1f = (float*)(base + L.kf);
    float* k2f = k1f + (size_t)n * h;
    const bool bf = c.dtype == SDM_BF16;
    cudaError_t e = cudaMemsetAsync(ds1, 0, 2 * 2 * (size_t)ntok * n * sizeof(float), s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(q_w, ntok, dk, qf, s) : widen<float>(q_w, ntok, dk, qf, s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(q_r, ntok, dk, qf + (size_t)ntok * dk, s)
               : widen<float>(q_r, ntok, dk, qf + (size_t)ntok * dk, s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(K1, n, h, k1f, s) : widen<float>(K1, n, h, k1f, s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(K2, n, h, k2f, s) : widen<float>(K2, n, h, k2f, s);
    if (e == cudaSuccess) {
        select_bwd_kernel<<<grid_for(2 * ntok * 32), 256, 0, s>>>(idx, wsel, dwsel, ntok, c.w, n, ds1,
                                                                  ds2);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess)
        return SDM_ECUDA;
    const int nt = (int)ntok;
    for (int half = 0; half < 2; ++half) {
        const float* ds = half ? ds2 : ds1;
        const float* kf = half ? k2f : k1f;
        // dq_h = DS_h K_h for each kind, into that kind's half of dq
        for (int kind = 0; kind < 2; ++kind) {
            const int rc = gemm_f32_rm(s, false, false, nt, h, n, ds + (size_t)kind * ntok * n, n, kf, h,
                                       (kind ? dq_r : dq_w) + half * h, dk, 0.f);
            if (rc != SDM_OK)
                return rc;
        }
        // dK_h = DS_h^T Q_h over both kinds
        const int rc = gemm_f32_rm(s, true, false, n, h, 2 * nt, ds, n, qf + half * h, dk,
                                   half ? dK2 : dK1, h, 0.f);
        if (rc != SDM_OK)
            return rc;
    }
    return SDM_OK;
}

}  // namespace sdm

// ---------------------------------------------------------- projection backward
// q_w = x W_qw, q_r = x W_qr, v = x W_v (the rounding of the outputs passed through):
//   dx = dq_w W_qw^T + dq_r W_qr^T + dv W_v^T,   dW_* = x^T d(out)_*
// GEMMs on fp32 copies of x and the weights: strict fp32 for an fp32 layer; for a bf16
// layer on the tensor cores in TF32, where x and the weights are exact (a bf16 value has
// fewer mantissa bits than TF32) and only the incoming fp32 gradients are rounded, to a
// relative 2^-11, finer than the layer's own bf16 rounding of its outputs (2^-9).

namespace sdm {

size_t project_backward_ws_bytes(const sdm_cfg& c, int64_t ntok)
{
    const size_t xb = ((size_t)ntok * c.d * 4 + 255) / 256 * 256;
    const size_t wb = ((size_t)c.d * (2 * c.dk + c.d) * 4 + 255) / 256 * 256;
    return xb + wb;
}

int launch_project_backward(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                            const float* dq_w, const float* dq_r, const float* dv, float* dx,
                            float* dW_qw, float* dW_qr, float* dW_v, void* ws, cudaStream_t s)
{
    if (ntok <= 0)
        return SDM_OK;
    if (ntok > 0x7FFFFFFF)
        return SDM_EUNSUPPORTED;
    const int d = c.d, dk = c.dk, nt = (int)ntok;
    float* xf = (float*)ws;
    float* wqw = (float*)((char*)ws + ((size_t)ntok * d * 4 + 255) / 256 * 256);
    float* wqr = wqw + (size_t)d * dk;
    float* wv = wqr + (size_t)d * dk;
    const bool bf = c.dtype == SDM_BF16;
    const bool tc = bf;   // TF32 tensor cores for a bf16 layer
    cudaError_t e = bf ? widen<bf16>(x, ntok, d, xf, s) : widen<float>(x, ntok, d, xf, s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(w.W_qw, d, dk, wqw, s) : widen<float>(w.W_qw, d, dk, wqw, s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(w.W_qr, d, dk, wqr, s) : widen<float>(w.W_qr, d, dk, wqr, s);
    if (e == cudaSuccess)
        e = bf ? widen<bf16>(w.W_v, d, d, wv, s) : widen<float>(w.W_v, d, d, wv, s);
    if (e != cudaSuccess)
        return SDM_ECUDA;
    int rc = gemm_f32_rm(s, false, true, nt, d, dk, dq_w, dk, wqw, dk, dx, d, 0.f, tc);
    if (rc == SDM_OK)
        rc = gemm_f32_rm(s, false, true, nt, d, dk, dq_r, dk, wqr, dk, dx, d, 1.f, tc);
    if (rc == SDM_OK)
        rc = gemm_f32_rm(s, false, true, nt, d, d, dv, d, wv, d, dx, d, 1.f, tc);
    if (rc == SDM_OK)
        rc = gemm_f32_rm(s, true, false, d, dk, nt, xf, d, dq_w, dk, dW_qw, dk, 0.f, tc);
    if (rc == SDM_OK)
        rc = gemm_f32_rm(s, true, false, d, dk, nt, xf, d, dq_r, dk, dW_qr, dk, 0.f, tc);
    if (rc == SDM_OK)
        rc = gemm_f32_rm(s, true, false, d, d, nt, xf, d, dv, d, dW_v, d, 0.f, tc);
    return rc;
}

}  // namespace sdm
