// bank_init.cu -- a0: each sequence's bank starts as the learned initial state M0
// ("Sparse Delta Memory: Scaling the State of Linear RNNs through Sparsity",
// Abstract: the initial state of the memory is learned and used as parametric memory).
//
// HBM-bound copy: M0 is read once and written B times. Every thread moves 16-byte
// chunks, four per iteration, with streaming stores; the grid is a multiple of the
// SM count.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

__global__ void __launch_bounds__(256) bank_init_kernel(const uint4* __restrict__ M0,
                                                        uint4* __restrict__ banks,
                                                        int64_t n16, int B)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 a = __ldcs(M0 + i);
        uint4 b = __ldcs(M0 + i + stride);
        uint4 c = __ldcs(M0 + i + 2 * stride);
        uint4 d = __ldcs(M0 + i + 3 * stride);
        for (int s = 0; s < B; ++s) {
            uint4* o = banks + (int64_t)s * n16;
            __stcs(o + i, a);
            __stcs(o + i + stride, b);
            __stcs(o + i + 2 * stride, c);
            __stcs(o + i + 3 * stride, d);
        }
    }
    for (; i < n16; i += stride) {
        uint4 a = __ldcs(M0 + i);
        for (int s = 0; s < B; ++s)
            __stcs(banks + (int64_t)s * n16 + i, a);
    }
}

cudaError_t launch_bank_init(const void* M0, void* banks, size_t bank_bytes, int B,
                             cudaStream_t s)
{
    if (B <= 0 || bank_bytes == 0)
        return cudaSuccess;
    const int64_t n16 = (int64_t)(bank_bytes / 16);
    const int sms = num_sms_current_device();
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap)
        blocks = cap;
    bank_init_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint4*)M0, (uint4*)banks, n16, B);
    return cudaGetLastError();
}

}  // namespace sdm
