// bank_init.cu -- a0: each sequence's bank starts as the learned initial state M0
// ("Sparse Delta Memory: Scaling the State of Linear RNNs through Sparsity",
// Abstract: the initial state of the memory is learned and used as parametric memory).
//
// HBM-bound copy: M0 is read once and written B times. Every thread moves 16-byte
// chunks, four per iteration, with streaming stores; the grid is a multiple of the
// SM count. The first-touch kernels below give the same initial state without the
// copy of slots the sequence writes.
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

// ---------------------------------------------------------------- first touch
//
// The same initial state without the copy. Before token t a slot holds M0 unless an
// earlier token of its sequence wrote it, so the scan reads M0 for those references
// (scan.cu) and only the slots a sequence never writes need M0 in its bank afterwards.
// first_write[b][s] is the first token of sequence b whose write set holds s.

// W is a power of two and B * T < 2^31 (the host checks): the token of write reference e
// is e >> lw, its position e & (W - 1), and the sequence a 32-bit division of the token
__global__ void __launch_bounds__(256) first_touch_kernel(const int32_t* __restrict__ idx,
                                                          int64_t nref, int T, int W, int N,
                                                          int32_t* __restrict__ first_write)
{
    const int lw = __ffs(W) - 1;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nref; e += stride) {
        const uint32_t tok = (uint32_t)(e >> lw);  // b * T + t
        const int32_t s = __ldg(idx + ((int64_t)tok << (lw + 1)) + (e & (W - 1)));
        if (s >= 0 && s < N) {
            const uint32_t b = tok / (uint32_t)T;
            atomicMin(first_write + (int64_t)b * N + s, (int32_t)(tok - b * (uint32_t)T));
        }
    }
}

// One warp per slot: the sequences that never wrote it (first_write >= T) get M0's row,
// read once. Up to 32 sequences: a lane per sequence reads the first-writer table, one
// slot ahead, and each lane has eight 16-byte loads in flight (a 4 KB row at once); more
// sequences take them 32 at a time.
__global__ void __launch_bounds__(256) fill_untouched_kernel(const uint4* __restrict__ M0,
                                                             const int32_t* __restrict__ first_write,
                                                             uint4* __restrict__ banks, int B, int T,
                                                             int N, int row16)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t sl = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (B > 32) {
        for (; sl < N; sl += warps) {
            for (int b0 = 0; b0 < B; b0 += 32) {
                const int b = b0 + lane;
                const bool fresh = b < B && __ldg(first_write + (int64_t)b * N + sl) >= T;
                unsigned mask = __ballot_sync(0xFFFFFFFFu, fresh);
                if (mask == 0)
                    continue;
                const uint4* src = M0 + sl * row16;
                for (int c0 = lane; c0 < row16; c0 += 32) {
                    const uint4 v = __ldg(src + c0);
                    for (unsigned m = mask; m != 0; m &= m - 1)
                        __stcs(banks + ((int64_t)(b0 + __ffs(m) - 1) * N + sl) * row16 + c0, v);
                }
            }
        }
        return;
    }
    bool fresh = sl < N && lane < B && __ldg(first_write + (int64_t)lane * N + sl) >= T;
    while (sl < N) {
        const int64_t nx = sl + warps;
        const bool fresh_n = nx < N && lane < B && __ldg(first_write + (int64_t)lane * N + nx) >= T;
        const unsigned mask = __ballot_sync(0xFFFFFFFFu, fresh);
        if (mask != 0) {
            const uint4* src = M0 + sl * row16;
            for (int c0 = lane; c0 < row16; c0 += 8 * 32) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c0 + u * 32 < row16)
                        v[u] = __ldg(src + c0 + u * 32);
                for (unsigned m = mask; m != 0; m &= m - 1) {
                    uint4* dst = banks + ((int64_t)(__ffs(m) - 1) * N + sl) * row16;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (c0 + u * 32 < row16)
                            __stcs(dst + c0 + u * 32, v[u]);
                }
            }
        }
        sl = nx;
        fresh = fresh_n;
    }
}

cudaError_t launch_first_touch(const sdm_cfg& c, const int32_t* idx, int B, int T,
                               int32_t* first_write, cudaStream_t s)
{
    if (B <= 0)
        return cudaSuccess;
    const int N = c.n_sub * c.n_sub;
    // 0x7F7F7F7F: above every token index
    cudaError_t e = cudaMemsetAsync(first_write, 0x7F, (size_t)B * N * sizeof(int32_t), s);
    if (e != cudaSuccess || T <= 0)
        return e;
    if ((int64_t)B * T > 0x7FFFFFFF || c.w <= 0 || (c.w & (c.w - 1)) != 0)
        return cudaErrorInvalidValue;   // (the kernel's index arithmetic)
    const int64_t nref = (int64_t)B * T * c.w;
    int64_t blocks = (nref + 255) / 256;
    const int64_t cap = (int64_t)num_sms_current_device() * 8;
    if (blocks > cap)
        blocks = cap;
    first_touch_kernel<<<(unsigned)blocks, 256, 0, s>>>(idx, nref, T, c.w, N, first_write);
    return cudaGetLastError();
}

cudaError_t launch_fill_untouched(const sdm_cfg& c, const void* M0, const int32_t* first_write,
                                  void* banks, int B, int T, cudaStream_t s)
{
    if (B <= 0)
        return cudaSuccess;
    const int N = c.n_sub * c.n_sub;
    const int row16 = c.d * (c.dtype == SDM_BF16 ? 2 : 4) / 16;
    const int64_t blocks = (int64_t)num_sms_current_device() * 8;
    fill_untouched_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint4*)M0, first_write,
                                                            (uint4*)banks, B, T, N, row16);
    return cudaGetLastError();
}

}  // namespace sdm
