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
// Block: one sequence, a run of `tb` tokens [t0, t1). The references of the window
// [t0 - win, t1) (slot ids are one contiguous run of idx) are indexed by slot: a counting
// sort places them in kBuckets hash buckets of (slot, token, kind, position) entries,
// 6 bytes each; bucket counts and offsets are 16-bit (two buckets a 32-bit word for the
// atomics; a block indexes fewer than 65,536 references). Each reference of the block then scans only its slot's bucket -- a handful
// of entries, more for popular slots -- for the latest earlier writer and the earlier
// referencing tokens. The window is indexed again by every block; the run length is the
// one whose waves of blocks cost least (below). In each phase a thread loads its slot ids
// kBatch at a time before it uses any of them, so that their L2 round trips overlap
// (one dependent load a reference made the kernel wait on L2 latency throughout).
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kBuckets = 4096;
constexpr int kCodeThreads = 512;
constexpr size_t kCodeSmemMax = 225 * 1024;
// slot ids a thread loads before it uses any of them: the loads of a batch are in flight
// together instead of one L2 round trip per reference
constexpr int kBatch = 8;

__device__ __forceinline__ uint32_t bucket_of(int32_t s)
{
    return ((uint32_t)s * 0x9E3779B1u) >> 20;   // top 12 bits
}

__global__ void __launch_bounds__(kCodeThreads) codes_kernel(const int32_t* __restrict__ idx, int T,
                                                             int W, int N, int win, int tb,
                                                             uint16_t* __restrict__ codes,
                                                             unsigned long long* __restrict__ fwdmask,
                                                             unsigned long long* __restrict__ deadmask,
                                                             unsigned long long* __restrict__ warmask,
                                                             int* status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t* off = reinterpret_cast<uint16_t*>(smem_raw);           // [kBuckets + 1]
    uint32_t* cur = reinterpret_cast<uint32_t*>(off + kBuckets + 8); // [kBuckets / 2] counts, cursors
    int32_t* slot = reinterpret_cast<int32_t*>(cur + kBuckets / 2);   // [nref window]
    uint16_t* info = reinterpret_cast<uint16_t*>(slot + (tb + win) * 2 * W);  // tloc<<7|kind<<6|pos
    __shared__ uint32_t wsum[kCodeThreads / 32];
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * tb;
    const int t1 = min(T, t0 + tb);
    const int base = max(0, t0 - win);
    const int nwin = (t1 - base) * 2 * W;
    const int32_t* wsrc = idx + ((size_t)b * T + base) * 2 * W;     // [token][write, read][W]
    // W is a power of two (the host checks): reference e of a run is token e >> (lw + 1),
    // set (e >> lw) & 1, position e & (W - 1) -- shifts, not divisions
    const int lw = __ffs(W) - 1;
    for (int i = threadIdx.x; i < kBuckets / 2; i += blockDim.x)
        cur[i] = 0u;
    __syncthreads();
    for (int e0 = threadIdx.x; e0 < nwin; e0 += kCodeThreads * kBatch) {
        int32_t sv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kCodeThreads;
            sv[u] = e < nwin ? __ldg(wsrc + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kCodeThreads;
            const int32_t s = sv[u];
            if (e >= nwin)
                break;
            if (s >= 0 && s < N) {
                const uint32_t bk = bucket_of(s);
                atomicAdd(&cur[bk >> 1], 1u << (16 * (bk & 1)));
            } else if (((e >> lw) & 1) == 0) {
                report(status, SDM_ERANGE);
            }
        }
    }
    __syncthreads();
    // exclusive prefix sum of the bucket sizes (8 buckets a thread)
    {
        constexpr int PER = kBuckets / kCodeThreads;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        uint32_t v[PER], tot = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int bk = threadIdx.x * PER + i;
            v[i] = (cur[bk >> 1] >> (16 * (bk & 1))) & 0xFFFFu;
            tot += v[i];
        }
        uint32_t inc = tot;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d)
                inc += o;
        }
        if (lane == 31)
            wsum[warp] = inc;
        __syncthreads();
        uint32_t pre = 0;
        for (int w = 0; w < warp; ++w)
            pre += wsum[w];
        uint32_t run = pre + inc - tot;
        __syncthreads();   // every count is read before the cursors replace them
#pragma unroll
        for (int i = 0; i < PER; i += 2) {
            off[threadIdx.x * PER + i] = (uint16_t)run;
            off[threadIdx.x * PER + i + 1] = (uint16_t)(run + v[i]);
            cur[(threadIdx.x * PER + i) >> 1] = run | ((run + v[i]) << 16);
            run += v[i] + v[i + 1];
        }
        if (threadIdx.x == blockDim.x - 1)
            off[kBuckets] = (uint16_t)run;
    }
    __syncthreads();
    for (int e0 = threadIdx.x; e0 < nwin; e0 += kCodeThreads * kBatch) {
        int32_t sv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kCodeThreads;
            sv[u] = e < nwin ? __ldg(wsrc + e) : -1;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kCodeThreads;
            const int32_t s = sv[u];
            if (s >= 0 && s < N) {
                const uint32_t bk = bucket_of(s);
                const uint32_t at = (atomicAdd(&cur[bk >> 1], 1u << (16 * (bk & 1))) >> (16 * (bk & 1))) & 0xFFFFu;
                slot[at] = s;
                info[at] = (uint16_t)(((e >> (lw + 1)) << 7) | (((e >> lw) & 1) << 6) | (e & (W - 1)));
            }
        }
    }
    __syncthreads();
    const int nref = (t1 - t0) * 2 * W;
    const int32_t* rsrc = idx + ((size_t)b * T + t0) * 2 * W;
    for (int e0 = threadIdx.x; e0 < nref; e0 += kCodeThreads * kBatch) {
        int32_t sv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kCodeThreads;
            sv[u] = e < nref ? __ldg(rsrc + e) : -1;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kCodeThreads;
            if (e >= nref)
                break;
            const int kind = (e >> lw) & 1;
            const int t = t0 + (e >> (lw + 1));
            const size_t o = ((size_t)b * T + t0) * 2 * W + e;
            const int32_t s = sv[u];
            uint16_t code = kNoFwd;
            if (s >= 0 && s < N) {
                const uint32_t bk = bucket_of(s);
                int best_dt = 1 << 30, best_pos = 0;
                unsigned long long war0 = 0, war1 = 0;
                for (uint32_t q = off[bk]; q < off[bk + 1]; ++q) {
                    if (slot[q] != s)
                        continue;
                    const uint32_t in = info[q];
                    const int dt = t - (base + (int)(in >> 7));
                    if (dt < 0 || dt > win)
                        continue;
                    const bool is_w = ((in >> 6) & 1) == 0;
                    // writers: the latest one at or before t (a read sees its own token's
                    // write), strictly before t for a write
                    if (is_w && dt < best_dt && (kind ? dt >= 0 : dt >= 1)) {
                        best_dt = dt;
                        best_pos = (int)(in & 0x3F);
                    }
                    // a write waits for the bank loads of every earlier referencing token
                    if (!kind && dt >= 1) {
                        if (dt <= 64)
                            war0 |= 1ull << (dt - 1);
                        else
                            war1 |= 1ull << (dt - 65);
                    }
                }
                if (best_dt <= win) {
                    code = (uint16_t)((best_dt << 8) | best_pos);
                    if (best_dt > 0) {
                        atomicOr(fwdmask + (size_t)b * T + t - best_dt, 1ull << best_pos);
                        if (!kind)
                            atomicOr(deadmask + (size_t)b * T + t - best_dt, 1ull << best_pos);
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
}

}  // namespace

cudaError_t launch_scan_codes(const sdm_cfg& c, const int32_t* idx, int B, int T, int win,
                              uint16_t* codes, unsigned long long* masks, int* status,
                              cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    if (T == 1)   // one token a sequence: the scan matches reads to own writes itself
        return cudaSuccess;
    if (c.w <= 0 || (c.w & (c.w - 1)) != 0 || c.w > 64)   // (the kernel's index arithmetic)
        return cudaErrorInvalidValue;
    // masks: fwdmask [B*T], deadmask [B*T], warmask [B*T][2], all cleared first
    cudaError_t e = cudaMemsetAsync(masks, 0, (size_t)B * T * 4 * sizeof(unsigned long long), s);
    if (e != cudaSuccess)
        return e;
    unsigned long long* fwdmask = masks;
    unsigned long long* deadmask = masks + (size_t)B * T;
    unsigned long long* warmask = masks + (size_t)B * T * 2;
    const int N = c.n_sub * c.n_sub;
    // Tokens a block: every block indexes its run and the window before it (6 bytes a
    // reference; at most 512 tokens indexed, the reach of the 9-bit token field). The
    // kernel is bound by the latency of its index, so blocks resident together on an SM
    // take about as long as one: a run of tb tokens costs its waves of blocks (as many
    // blocks an SM as shared memory and threads allow) times the references a block
    // handles, (tb + win) inserted and tb looked up. The cheapest run wins (the longer
    // one on a tie). At 4 x 4,096 tokens with a window of 35 that is runs of 56, one
    // wave, where the earlier rule (the longest run still giving two blocks an SM) took
    // runs of 48, 344 blocks for 296 places.
    const int sms = num_sms_current_device();
    auto smem_for = [&](int tb_) {
        return (size_t)(kBuckets + 8) * 2 + (size_t)kBuckets * 2 + (size_t)(tb_ + win) * 2 * c.w * 6;
    };
    int tb = 8;
    long long best = -1;
    for (int tb_ = 256; tb_ >= 8; tb_ -= 8) {
        const size_t sm = smem_for(tb_);
        if (sm > kCodeSmemMax || tb_ + win > 512 || (long long)(tb_ + win) * 2 * c.w > 65535)
            continue;
        // at most two blocks an SM: in a prefill from M0 the codes run beside the
        // first-touch table and the fill, which need room on the SMs as well
        long long per_sm = (long long)(228 * 1024) / (long long)(sm + 1024);
        per_sm = per_sm < 1 ? 1 : per_sm > 2 ? 2 : per_sm;
        const long long blocks = (long long)B * ((T + tb_ - 1) / tb_);
        const long long waves = (blocks + per_sm * sms - 1) / (per_sm * sms);
        const long long cost = waves * (2LL * tb_ + win);
        if (best < 0 || cost < best) {
            best = cost;
            tb = tb_;
        }
    }
    const size_t smem = smem_for(tb);
    e = cudaFuncSetAttribute(codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((T + tb - 1) / tb, B);
    codes_kernel<<<grid, kCodeThreads, smem, s>>>(idx, T, c.w, N, win, tb, codes, fwdmask, deadmask,
                                                  warmask, status);
    return cudaGetLastError();
}

}  // namespace sdm
