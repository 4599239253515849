// project.cu -- the library GEMMs of the backward pass: plain fp32 products of gradients
// with activations and weights (the forward projections run in proj_tc.cu's own kernels).
// One cuBLAS handle per device, created on first use and bound to the caller's stream
// for each call.
#include <cublas_v2.h>

#include <mutex>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

static std::mutex g_blas_mu;
static cublasHandle_t g_blas[64];

static cublasHandle_t blas_handle()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    if (g_blas[dev] == nullptr) {
        cublasHandle_t h = nullptr;
        if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS)
            return nullptr;
        g_blas[dev] = h;
    }
    return g_blas[dev];
}

// Row-major fp32 GEMM on the library's own handle (strict fp32; with tf32 the inputs are
// rounded to TF32 and the products summed in fp32 on the tensor cores):
//   C [M, N] = op(A) [M, K] op(B) [K, N] (+ beta C), op = transpose when ta / tb.
// In column-major terms C^T = op(B)^T op(A)^T, which is the call below.
int gemm_f32_rm(cudaStream_t s, bool ta, bool tb, int M, int N, int K, const float* A, int lda,
                const float* B, int ldb, float* C, int ldc, float beta, bool tf32)
{
    std::lock_guard<std::mutex> lock(g_blas_mu);
    cublasHandle_t h = blas_handle();
    if (h == nullptr || cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS)
        return SDM_ECUDA;
    const float one = 1.0f;
    return cublasGemmEx(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N, N, M, K,
                        &one, B, CUDA_R_32F, ldb, A, CUDA_R_32F, lda, &beta, C, CUDA_R_32F, ldc,
                        tf32 ? CUBLAS_COMPUTE_32F_FAST_TF32 : CUBLAS_COMPUTE_32F_PEDANTIC,
                        CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS
               ? SDM_OK
               : SDM_ECUDA;
}

}  // namespace sdm
