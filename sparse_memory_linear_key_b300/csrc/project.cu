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

// ---------------------------------------------------------- forked projections

// Per device: two side streams with a cuBLAS handle each, and the events that fork them
// off the caller's stream and join them back. q_w runs on the caller's stream, q_r and v
// on the side streams; the caller's stream waits for q_r before the addressing, and only
// the scan waits for v. Everything is recorded with events, so the three GEMMs overlap
// in eager use and become parallel branches when the caller captures a graph.
struct Fork {
    bool ready = false;
    cudaStream_t side[2] = {nullptr, nullptr};
    cublasHandle_t h[2] = {nullptr, nullptr};
    cudaEvent_t ev_fork = nullptr, ev_q = nullptr, ev_v = nullptr;
};
static Fork g_fork[64];

static Fork* fork_state()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    Fork& f = g_fork[dev];
    if (f.ready)
        return &f;
    for (int i = 0; i < 2; ++i) {
        if (f.side[i] == nullptr &&
            cudaStreamCreateWithFlags(&f.side[i], cudaStreamNonBlocking) != cudaSuccess)
            return nullptr;
        if (f.h[i] == nullptr && cublasCreate(&f.h[i]) != CUBLAS_STATUS_SUCCESS)
            return nullptr;
        if (cublasSetStream(f.h[i], f.side[i]) != CUBLAS_STATUS_SUCCESS)
            return nullptr;
    }
    cudaEvent_t* evs[3] = {&f.ev_fork, &f.ev_q, &f.ev_v};
    for (cudaEvent_t* e : evs)
        if (*e == nullptr && cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
    f.ready = true;
    return &f;
}

int launch_project_forked(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                          void* q_w, void* q_r, void* v, cudaStream_t s, void* blas_ws,
                          size_t blas_ws_bytes, std::unique_lock<std::mutex>& lock,
                          cudaEvent_t* v_ready)
{
    *v_ready = nullptr;
    if (ntok <= 0)
        return SDM_OK;
    if (ntok > 0x7FFFFFFF)
        return SDM_EUNSUPPORTED;
    lock = std::unique_lock<std::mutex>(g_blas_mu);
    cublasHandle_t h = blas_handle(1);
    Fork* f = fork_state();
    if (h == nullptr || f == nullptr)
        return SDM_ECUDA;
    // the workspace region in three parts, one per concurrent GEMM
    const size_t part = (blas_ws_bytes / 3) & ~(size_t)255;
    char* wsb = (char*)blas_ws;
    const bool bf = c.dtype == SDM_BF16;
    if (cudaEventRecord(f->ev_fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(f->side[0], f->ev_fork, 0) != cudaSuccess ||
        cudaStreamWaitEvent(f->side[1], f->ev_fork, 0) != cudaSuccess)
        return SDM_ECUDA;
    const bool ok =
        cublasSetStream(h, s) == CUBLAS_STATUS_SUCCESS &&
        cublasSetWorkspace(h, wsb, part) == CUBLAS_STATUS_SUCCESS &&
        cublasSetWorkspace(f->h[0], wsb + part, part) == CUBLAS_STATUS_SUCCESS &&
        cublasSetWorkspace(f->h[1], wsb + 2 * part, part) == CUBLAS_STATUS_SUCCESS &&
        gemm(f->h[1], bf, x, w.W_v, v, ntok, c.d, c.d) == CUBLAS_STATUS_SUCCESS &&
        gemm(f->h[0], bf, x, w.W_qr, q_r, ntok, c.d, c.dk) == CUBLAS_STATUS_SUCCESS &&
        gemm(h, bf, x, w.W_qw, q_w, ntok, c.d, c.dk) == CUBLAS_STATUS_SUCCESS;
    // both side streams join back whatever happened (a forked capture must rejoin)
    const bool joined = cudaEventRecord(f->ev_q, f->side[0]) == cudaSuccess &&
                        cudaStreamWaitEvent(s, f->ev_q, 0) == cudaSuccess &&
                        cudaEventRecord(f->ev_v, f->side[1]) == cudaSuccess;
    if (!joined)
        return SDM_ECUDA;
    *v_ready = f->ev_v;
    return ok ? SDM_OK : SDM_ECUDA;
}

}  // namespace sdm

namespace sdm {

// Row-major fp32 GEMM on the library's own handle (strict fp32; with tf32 the inputs are
// rounded to TF32 and the products summed in fp32 on the tensor cores):
//   C [M, N] = op(A) [M, K] op(B) [K, N] (+ beta C), op = transpose when ta / tb.
// In column-major terms C^T = op(B)^T op(A)^T, which is the call below.
int gemm_f32_rm(cudaStream_t s, bool ta, bool tb, int M, int N, int K, const float* A, int lda,
                const float* B, int ldb, float* C, int ldc, float beta, bool tf32)
{
    std::lock_guard<std::mutex> lock(g_blas_mu);
    cublasHandle_t h = blas_handle(0);
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
