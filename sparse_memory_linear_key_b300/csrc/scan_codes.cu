// scan_codes.cu -- collision codes for the scan, computed for all tokens before it.
//
// The recurrence ("Sparse Delta Memory" blog, "Write & Read") is sequential in t only
// through slots that two tokens share. For every slot reference (token t, write or read
// set, position j) this kernel records the latest earlier writer of the same slot if
// it lies within the last `win` tokens of the sequence:
//   code = dt << 8 | pos   (writer t - dt wrote the slot at position pos of its write
//                           set; dt = 0 only for a read of a slot t writes itself)
//   code = kNoFwd          (no writer within the window)
// and, for the writer, sets bit pos of fwdmask[t - dt] (dt >= 1): that write is read by
// a later token while the writer may still be in flight, so the scan hands it over
// through its forwarding ring.
//
// Block: one sequence, a run of kCodeTB tokens [t0, t1). Two bitmaps over all N slots
// are built from the write lists of the window [t0 - win, t1): `once` marks slots
// written by at least one of those tokens, `twice` by at least two. A read reference
// whose `once` bit is clear, or a write reference whose `twice` bit is clear (its own
// token accounts for one write), has no earlier writer within the window: the common
// case, settled at once. The rest are queued and searched in the sorted write lists of
// the preceding tokens, newest first.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kCodeTB = 32;

__global__ void __launch_bounds__(256) codes_kernel(const int32_t* __restrict__ idx, int T, int W,
                                                    int N, int win,
                                                    uint16_t* __restrict__ codes,
                                                    unsigned long long* __restrict__ fwdmask,
                                                    int* status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int nwords = (N + 31) / 32;
    uint32_t* once = reinterpret_cast<uint32_t*>(smem_raw);
    uint32_t* twice = once + nwords;
    int32_t* lists = reinterpret_cast<int32_t*>(twice + nwords);   // [(kCodeTB + win) * W]
    int* queue = lists + (kCodeTB + win) * W;                       // [kCodeTB * 2 * W]
    __shared__ int qn;
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * kCodeTB;
    const int t1 = min(T, t0 + kCodeTB);
    const int base = max(0, t0 - win);
    const int nlist = t1 - base;
    for (int i = threadIdx.x; i < 2 * nwords; i += blockDim.x)
        once[i] = 0u;
    if (threadIdx.x == 0)
        qn = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < nlist * W; e += blockDim.x) {
        const int lt = e / W, j = e % W;
        const int32_t s = idx[(((size_t)b * T + base + lt) * 2 + 0) * W + j];
        lists[e] = s;
        if (s >= 0 && s < N) {
            const uint32_t m = 1u << (s & 31);
            if (atomicOr(&once[s >> 5], m) & m)
                atomicOr(&twice[s >> 5], m);
        } else {
            report(status, SDM_ERANGE);
        }
    }
    __syncthreads();
    const int nref = (t1 - t0) * 2 * W;
    for (int e = threadIdx.x; e < nref; e += blockDim.x) {
        const int kind = (e / W) & 1;
        const size_t o = ((size_t)b * T + t0) * 2 * W + e;
        const int32_t s = idx[o];
        bool hit = false;
        if (s >= 0 && s < N)
            hit = ((kind ? once : twice)[s >> 5] >> (s & 31)) & 1u;
        if (hit)
            queue[atomicAdd(&qn, 1)] = e;
        else
            codes[o] = kNoFwd;
    }
    __syncthreads();
    const int nq = qn;
    for (int qi = threadIdx.x; qi < nq; qi += blockDim.x) {
        const int e = queue[qi];
        const int t = t0 + e / (2 * W);
        const int kind = (e / W) & 1;
        const size_t o = ((size_t)b * T + t0) * 2 * W + e;
        const int32_t s = idx[o];
        uint16_t code = kNoFwd;
        for (int dt = kind ? 0 : 1; dt <= win; ++dt) {
            const int tp = t - dt;
            if (tp < base)
                break;
            const int32_t* L = lists + (tp - base) * W;
            int lo = 0, hi = W - 1, found = -1;
            while (lo <= hi) {
                const int mid = (lo + hi) >> 1;
                const int32_t v = L[mid];
                if (v == s) { found = mid; break; }
                if (v < s) lo = mid + 1; else hi = mid - 1;
            }
            if (found >= 0) {
                code = (uint16_t)((dt << 8) | found);
                if (dt > 0)
                    atomicOr(fwdmask + (size_t)b * T + tp, 1ull << found);
                break;
            }
        }
        codes[o] = code;
    }
}

}  // namespace

cudaError_t launch_scan_codes(const sdm_cfg& c, const int32_t* idx, int B, int T, int win,
                              uint16_t* codes, unsigned long long* fwdmask, int* status,
                              cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(fwdmask, 0, (size_t)B * T * sizeof(unsigned long long), s);
    if (e != cudaSuccess)
        return e;
    const int N = c.n_sub * c.n_sub;
    const size_t smem = (size_t)2 * ((N + 31) / 32) * 4 + (size_t)(kCodeTB + win) * c.w * 4 +
                        (size_t)kCodeTB * 2 * c.w * 4;
    e = cudaFuncSetAttribute(codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((T + kCodeTB - 1) / kCodeTB, B);
    codes_kernel<<<grid, 256, smem, s>>>(idx, T, c.w, N, win, codes, fwdmask, status);
    return cudaGetLastError();
}

}  // namespace sdm
