// scan_codes.cu -- collision codes for the scan, computed for all tokens before it.
//
// The recurrence ("Sparse Delta Memory" blog, "Write & Read") is sequential in t only
// through slots that two tokens share. For every slot reference (token t, write or read
// set, position j) this kernel records the latest earlier writer of the same slot if
// it lies within the last `win` tokens of the sequence:
//   code = dt << 8 | pos   (writer t - dt wrote the slot at position pos of its write
//                           set; dt = 0 only for a read of a slot t writes itself)
//   code = kNoFwd          (no writer within the window)
// and three per-token masks that the scan's ordering rules use:
//   fwdmask[t]   bit pos: t's write at pos is referenced by a later token within the
//                window (the scan hands it over through its forwarding ring);
//   deadmask[t]  bit pos: t's write at pos is written again by a later token within the
//                window, so its bank store is dead (every reader in between takes the
//                value from the ring, every later one the newer value);
//   warmask[t]   bit dt-1 (dt = 1..win, two words): token t-dt references (reads or
//                writes) a slot that t writes; t's bank stores wait for those tokens'
//                bank loads.
//
// Block: one sequence, a run of kCodeTB tokens [t0, t1). Bitmaps over all N slots are
// built from the lists of the window [t0 - win, t1): `once` / `twice` mark slots
// written by at least one / two of those tokens, `rref` slots read by any of them. A
// read reference whose `once` bit is clear, or a write reference whose `twice` and
// `rref` bits are clear (its own token accounts for one write), has nothing to find:
// the common case. The rest are queued and searched in the sorted lists of the
// preceding tokens, newest first.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kCodeTB = 32;

__device__ __forceinline__ int find_sorted(const int32_t* L, int W, int32_t s)
{
    int lo = 0, hi = W - 1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int32_t v = L[mid];
        if (v == s)
            return mid;
        if (v < s)
            lo = mid + 1;
        else
            hi = mid - 1;
    }
    return -1;
}

__global__ void __launch_bounds__(256) codes_kernel(const int32_t* __restrict__ idx, int T, int W,
                                                    int N, int win,
                                                    uint16_t* __restrict__ codes,
                                                    unsigned long long* __restrict__ fwdmask,
                                                    unsigned long long* __restrict__ deadmask,
                                                    unsigned long long* __restrict__ warmask,
                                                    int* status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int nwords = (N + 31) / 32;
    uint32_t* once = reinterpret_cast<uint32_t*>(smem_raw);
    uint32_t* twice = once + nwords;
    uint32_t* rref = twice + nwords;
    int32_t* wl = reinterpret_cast<int32_t*>(rref + nwords);       // [(kCodeTB + win) * W]
    int32_t* rl = wl + (kCodeTB + win) * W;                         // [(kCodeTB + win) * W]
    int* queue = rl + (kCodeTB + win) * W;                          // [kCodeTB * 2 * W]
    __shared__ int qn;
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * kCodeTB;
    const int t1 = min(T, t0 + kCodeTB);
    const int base = max(0, t0 - win);
    const int nlist = t1 - base;
    for (int i = threadIdx.x; i < 3 * nwords; i += blockDim.x)
        once[i] = 0u;
    if (threadIdx.x == 0)
        qn = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < nlist * 2 * W; e += blockDim.x) {
        const int lt = e / (2 * W), kind = (e / W) & 1, j = e % W;
        const int32_t s = idx[(((size_t)b * T + base + lt) * 2 + kind) * W + j];
        (kind ? rl : wl)[lt * W + j] = s;
        if (s >= 0 && s < N) {
            const uint32_t m = 1u << (s & 31);
            if (kind)
                atomicOr(&rref[s >> 5], m);
            else if (atomicOr(&once[s >> 5], m) & m)
                atomicOr(&twice[s >> 5], m);
        } else if (kind == 0) {
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
        if (s >= 0 && s < N) {
            const uint32_t m = 1u << (s & 31);
            // a write is searched if another write of the slot or a read of it lies in
            // the window
            hit = kind ? (once[s >> 5] & m) != 0
                       : ((twice[s >> 5] & m) != 0 || (rref[s >> 5] & m) != 0);
        }
        if (hit)
            queue[atomicAdd(&qn, 1)] = e;
        else
            codes[o] = kNoFwd;
    }
    __syncthreads();
    const int nq = qn;
    for (int qi = threadIdx.x; qi < nq; qi += blockDim.x) {
        const int e = queue[qi];
        const int lt = e / (2 * W);
        const int t = t0 + lt;
        const int kind = (e / W) & 1;
        const size_t o = ((size_t)b * T + t0) * 2 * W + e;
        const int32_t s = idx[o];
        uint16_t code = kNoFwd;
        if (kind) {
            // read: the latest writer, this token's own write included
            for (int dt = 0; dt <= win && t - dt >= base; ++dt) {
                const int pos = find_sorted(wl + (t - dt - base) * W, W, s);
                if (pos >= 0) {
                    code = (uint16_t)((dt << 8) | pos);
                    if (dt > 0)
                        atomicOr(fwdmask + (size_t)b * T + t - dt, 1ull << pos);
                    break;
                }
            }
        } else {
            // write: the latest earlier writer, and every earlier referencing token; only
            // the lists the bitmaps say can hold the slot are searched
            const uint32_t mb = 1u << (s & 31);
            const bool other_w = (twice[s >> 5] & mb) != 0, any_r = (rref[s >> 5] & mb) != 0;
            unsigned long long war0 = 0, war1 = 0;
            for (int dt = 1; dt <= win && t - dt >= base; ++dt) {
                const int tp = t - dt - base;
                const int pw = other_w ? find_sorted(wl + tp * W, W, s) : -1;
                const bool ref = pw >= 0 || (any_r && find_sorted(rl + tp * W, W, s) >= 0);
                if (pw >= 0 && code == kNoFwd) {
                    code = (uint16_t)((dt << 8) | pw);
                    atomicOr(fwdmask + (size_t)b * T + t - dt, 1ull << pw);
                    atomicOr(deadmask + (size_t)b * T + t - dt, 1ull << pw);
                }
                if (ref) {
                    if (dt <= 64)
                        war0 |= 1ull << (dt - 1);
                    else
                        war1 |= 1ull << (dt - 65);
                }
            }
            if (war0)
                atomicOr(warmask + ((size_t)b * T + t) * 2, war0);
            if (war1)
                atomicOr(warmask + ((size_t)b * T + t) * 2 + 1, war1);
        }
        codes[o] = code;
    }
}

}  // namespace

cudaError_t launch_scan_codes(const sdm_cfg& c, const int32_t* idx, int B, int T, int win,
                              uint16_t* codes, unsigned long long* masks, int* status,
                              cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    // masks: fwdmask [B*T], deadmask [B*T], warmask [B*T][2], all cleared first
    cudaError_t e = cudaMemsetAsync(masks, 0, (size_t)B * T * 4 * sizeof(unsigned long long), s);
    if (e != cudaSuccess)
        return e;
    unsigned long long* fwdmask = masks;
    unsigned long long* deadmask = masks + (size_t)B * T;
    unsigned long long* warmask = masks + (size_t)B * T * 2;
    const int N = c.n_sub * c.n_sub;
    const size_t smem = (size_t)3 * ((N + 31) / 32) * 4 + (size_t)2 * (kCodeTB + win) * c.w * 4 +
                        (size_t)kCodeTB * 2 * c.w * 4;
    e = cudaFuncSetAttribute(codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((T + kCodeTB - 1) / kCodeTB, B);
    codes_kernel<<<grid, 256, smem, s>>>(idx, T, c.w, N, win, codes, fwdmask, deadmask, warmask,
                                         status);
    return cudaGetLastError();
}

}  // namespace sdm
