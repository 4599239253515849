// slot_stats.cu -- which slots the tokens write and read ("Sparse Delta Memory" blog,
// "Memory Access Patterns on a Needle-in-a-Haystack Task": the slots accessed at each
// token position -- cumulative writes, current reads -- and the write-read bucket
// overlap, whether the slots written at the needle are the slots read at the query).
//
// Both statistics are integer work over the addressing output idx [B*T][2][w]:
//   slot_counts   counts[b][s] = number of tokens t in [t0, t1) of sequence b whose
//                 write (kind 0) or read (kind 1) set holds s; one atomic per reference.
//   slot_overlap  per sequence: distinct slots written in [w0, w1), distinct slots read
//                 in [r0, r1), and distinct slots in both -- two N-bit maps per sequence
//                 (atomicOr per reference), then population counts.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

__global__ void __launch_bounds__(256) slot_counts_kernel(const int32_t* __restrict__ idx, int B,
                                                          int T, int W, int N, int kind, int t0,
                                                          int t1, uint32_t* __restrict__ counts)
{
    const int64_t span = (int64_t)(t1 - t0) * W;
    const int64_t total = (int64_t)B * span;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        const int b = (int)(e / span);
        const int64_t r = e % span;
        const int64_t tok = (int64_t)b * T + t0 + r / W;
        const int32_t s = __ldg(idx + (tok * 2 + kind) * W + r % W);
        if (s >= 0 && s < N)
            atomicAdd(counts + (int64_t)b * N + s, 1u);
    }
}

// maps: [B][2][words] (write window map, read window map)
__global__ void __launch_bounds__(256) slot_bitmap_kernel(const int32_t* __restrict__ idx, int B,
                                                          int T, int W, int N, int w0, int w1,
                                                          int r0, int r1, int words,
                                                          uint32_t* __restrict__ maps)
{
    const int64_t nw = (int64_t)(w1 - w0) * W, nr = (int64_t)(r1 - r0) * W;
    const int64_t per = nw + nr;
    const int64_t total = (int64_t)B * per;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        const int b = (int)(e / per);
        int64_t r = e % per;
        const int kind = r < nw ? 0 : 1;
        if (kind)
            r -= nw;
        const int64_t tok = (int64_t)b * T + (kind ? r0 : w0) + r / W;
        const int32_t s = __ldg(idx + (tok * 2 + kind) * W + r % W);
        if (s >= 0 && s < N)
            atomicOr(maps + ((int64_t)b * 2 + kind) * words + (s >> 5), 1u << (s & 31));
    }
}

// One block per sequence: out[b] = {popc(write map), popc(read map), popc(both)}.
__global__ void __launch_bounds__(256) slot_overlap_kernel(const uint32_t* __restrict__ maps,
                                                           int words, uint32_t* __restrict__ out)
{
    const int b = blockIdx.x;
    const uint32_t* wm = maps + (int64_t)b * 2 * words;
    const uint32_t* rm = wm + words;
    uint32_t cw = 0, cr = 0, cb = 0;
    for (int i = threadIdx.x; i < words; i += blockDim.x) {
        const uint32_t x = wm[i], y = rm[i];
        cw += __popc(x);
        cr += __popc(y);
        cb += __popc(x & y);
    }
    __shared__ uint32_t red[3][8];
    cw = __reduce_add_sync(0xFFFFFFFFu, cw);
    cr = __reduce_add_sync(0xFFFFFFFFu, cr);
    cb = __reduce_add_sync(0xFFFFFFFFu, cb);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[0][warp] = cw;
        red[1][warp] = cr;
        red[2][warp] = cb;
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        uint32_t t = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            t += red[threadIdx.x][w];
        out[(int64_t)b * 3 + threadIdx.x] = t;
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

}  // namespace

size_t slot_overlap_ws_bytes(const sdm_cfg& c, int B)
{
    const int64_t N = (int64_t)c.n_sub * c.n_sub;
    return (size_t)B * 2 * ((N + 31) / 32) * sizeof(uint32_t);
}

cudaError_t launch_slot_counts(const sdm_cfg& c, const int32_t* idx, int B, int T, int kind,
                               int t0, int t1, uint32_t* counts, cudaStream_t s)
{
    const int N = c.n_sub * c.n_sub;
    cudaError_t e = cudaMemsetAsync(counts, 0, (size_t)B * N * sizeof(uint32_t), s);
    if (e != cudaSuccess || t1 <= t0)
        return e;
    slot_counts_kernel<<<grid_for((int64_t)B * (t1 - t0) * c.w), 256, 0, s>>>(idx, B, T, c.w, N, kind,
                                                                           t0, t1, counts);
    return cudaGetLastError();
}

cudaError_t launch_slot_overlap(const sdm_cfg& c, const int32_t* idx, int B, int T, int w0, int w1,
                                int r0, int r1, uint32_t* out, void* ws, cudaStream_t s)
{
    const int N = c.n_sub * c.n_sub;
    const int words = (N + 31) / 32;
    uint32_t* maps = (uint32_t*)ws;
    cudaError_t e = cudaMemsetAsync(maps, 0, slot_overlap_ws_bytes(c, B), s);
    if (e != cudaSuccess)
        return e;
    const int64_t work = (int64_t)B * ((int64_t)(w1 - w0) + (r1 - r0)) * c.w;
    if (work > 0) {
        slot_bitmap_kernel<<<grid_for(work), 256, 0, s>>>(idx, B, T, c.w, N, w0, w1, r0, r1, words,
                                                          maps);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    slot_overlap_kernel<<<B, 256, 0, s>>>(maps, words, out);
    return cudaGetLastError();
}

}  // namespace sdm
