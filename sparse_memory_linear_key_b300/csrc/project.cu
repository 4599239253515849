// project.cu -- step P: q_w = x W_qw, q_r = x W_qr, v = x W_v ("Sparse Delta Memory"
// blog, "Write & Read": the token embedding is projected to write keys; a separate
// query projection selects the read slots).
//
// These are plain dense GEMMs with no fused epilogue (fp32 accumulation, one rounding
// to the I/O type), so they go to cuBLAS: bf16 x bf16 -> bf16 with an fp32 compute
// type, or strict fp32 (no TF32) in fp32 mode. Two handles per device, created on first
// use and bound to the caller's stream for each call: one with cuBLAS's own workspace
// (sdm_project), one that works in a region of the caller's workspace (sdm_prefill,
// sdm_decode_step), so that those calls allocate nothing and can be captured in a CUDA
// graph once a first call has set the handle up.
#include <cublas_v2.h>

#include <mutex>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

static std::mutex g_blas_mu;
static cublasHandle_t g_blas[2][64];

static cublasHandle_t blas_handle(int which)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    if (g_blas[which][dev] == nullptr) {
        cublasHandle_t h = nullptr;
        if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS)
            return nullptr;
        g_blas[which][dev] = h;
    }
    return g_blas[which][dev];
}

// out [rows, n] = x [rows, k] * Wm [k, n], all row-major. In column-major terms this
// is out^T = Wm^T x^T with Wm^T of shape [n, k] (ld n) and x^T of shape [k, rows].
static cublasStatus_t gemm(cublasHandle_t h, bool bf, const void* x, const void* Wm, void* out,
                           int64_t rows, int k, int n)
{
    const float one = 1.0f, zero = 0.0f;
    const cudaDataType_t t = bf ? CUDA_R_16BF : CUDA_R_32F;
    const cublasComputeType_t ct = bf ? CUBLAS_COMPUTE_32F : CUBLAS_COMPUTE_32F_PEDANTIC;
    return cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, n, (int)rows, k, &one, Wm, t, n, x, t, k,
                        &zero, out, t, n, ct, CUBLAS_GEMM_DEFAULT);
}

int launch_project(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                   void* q_w, void* q_r, void* v, cudaStream_t s, void* blas_ws, size_t blas_ws_bytes)
{
    if (ntok <= 0)
        return SDM_OK;
    if (ntok > 0x7FFFFFFF)
        return SDM_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_blas_mu);
    cublasHandle_t h = blas_handle(blas_ws != nullptr ? 1 : 0);
    if (h == nullptr)
        return SDM_ECUDA;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS)
        return SDM_ECUDA;
    if (blas_ws != nullptr && cublasSetWorkspace(h, blas_ws, blas_ws_bytes) != CUBLAS_STATUS_SUCCESS)
        return SDM_ECUDA;
    const bool bf = c.dtype == SDM_BF16;
    if (gemm(h, bf, x, w.W_qw, q_w, ntok, c.d, c.dk) != CUBLAS_STATUS_SUCCESS ||
        gemm(h, bf, x, w.W_qr, q_r, ntok, c.d, c.dk) != CUBLAS_STATUS_SUCCESS ||
        gemm(h, bf, x, w.W_v, v, ntok, c.d, c.d) != CUBLAS_STATUS_SUCCESS)
        return SDM_ECUDA;
    return SDM_OK;
}

}  // namespace sdm
