// scan.cu -- steps W and R of the recurrence for every token, in token order per
// sequence ("Sparse Delta Memory" blog, "Write & Read": selected columns are first
// decayed, then written with the delta rule; the output is a weighted sum of the
// retrieved columns; "How does SDM work?": the read follows the write and may use
// different slots).
//
// Per token t with write set S (weights k), read set R (weights r):
//   u = sum_j k_j M[S_j]                      (pre-write slot vectors)
//   M[S_j] <- alpha M[S_j] + beta k_j (v - alpha u)      rounded once to storage
//   y = sum_j r_j M[R_j]                      (post-write)
//
// Work split. Every row of a slot vector evolves independently, so the d rows are
// split into "machines" of 16 rows; a machine owns its rows of one sequence's bank
// for the whole sequence and never synchronises with other machines. Inside a
// machine, lane (sg, rg) of a warp holds rows rg*4..rg*4+3 of the W/8 slots
// sg*W/8 .. sg*W/8 + W/8 - 1 (8-byte bf16 / 16-byte fp32 accesses; the four lanes of
// one slot read one 32-byte sector), and u, y are reduced across the 8 slot groups
// with three xor-shuffles.
//
// Token parallelism. A machine runs G warps; warp g processes tokens g, g+G, g+2G...
// so G tokens are in flight, which hides HBM latency even when one sequence is all
// there is. Ordering:
//  * a warp issues the loads of token t right after its own token t-G committed, so
//    every write of a token <= t-G is visible to them;
//  * a slot of token t last written by a token t-dt with 1 <= dt < G (or by t itself
//    for a read, dt = 0) is not loaded: its post-write value is taken from the
//    shared-memory ring of the last G tokens' written values (the collision codes
//    computed by fwd_codes_kernel give dt and the position);
//  * commits (global stores + ring entry) happen strictly in token order, through a
//    per-machine watermark in shared memory (release/acquire), so no token
//    overwrites a slot that an earlier token has not read yet.
// Every wait is bounded: on time-out the kernel records SDM_ETIMEOUT and leaves.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

struct ScanParams {
    void* banks;
    const int32_t* idx;
    const float* wsel;
    const uint16_t* codes;
    const void* v;
    const float* alpha;
    const float* beta;
    float* y;
    int* status;
    int64_t machines;
    int T, d, N, G, MPC;
};

template <int SPL>
__device__ __forceinline__ void load_ids(const int32_t* p, int32_t (&o)[SPL])
{
    if constexpr (SPL % 4 == 0) {
#pragma unroll
        for (int i = 0; i < SPL; i += 4) {
            int4 v = __ldg((const int4*)(p + i));
            o[i] = v.x; o[i + 1] = v.y; o[i + 2] = v.z; o[i + 3] = v.w;
        }
    } else if constexpr (SPL == 2) {
        int2 v = __ldg((const int2*)p);
        o[0] = v.x; o[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            o[i] = __ldg(p + i);
    }
}

template <int SPL>
__device__ __forceinline__ void load_w(const float* p, float (&o)[SPL])
{
    if constexpr (SPL % 4 == 0) {
#pragma unroll
        for (int i = 0; i < SPL; i += 4) {
            float4 v = __ldg((const float4*)(p + i));
            o[i] = v.x; o[i + 1] = v.y; o[i + 2] = v.z; o[i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            o[i] = __ldg(p + i);
    }
}

template <int SPL>
__device__ __forceinline__ void load_codes(const uint16_t* p, uint16_t (&o)[SPL])
{
    if constexpr (SPL == 8) {
        uint4 v = __ldg((const uint4*)p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = (uint16_t)(w[i] & 0xFFFF);
            o[2 * i + 1] = (uint16_t)(w[i] >> 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            o[i] = __ldg(p + i);
    }
}

__device__ __forceinline__ void xor_reduce4(float (&a)[4])
{
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1)
#pragma unroll
        for (int r = 0; r < 4; ++r)
            a[r] += __shfl_xor_sync(0xFFFFFFFFu, a[r], m);
}

// Lane 0 waits for *wm >= target; the outcome is made warp-uniform and the warp
// synchronises so that every lane's later reads are ordered after the acquire.
__device__ __forceinline__ bool warp_wait_geq(const int* wm, int target, const int* abort,
                                              int* status)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = wait_geq(wm, target, abort, status) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

template <typename S, int SPL>
__global__ void __launch_bounds__(512, 1) scan_kernel(ScanParams p)
{
    using R4 = Row4<S>;
    using V = typename R4::V;
    constexpr int W = 8 * SPL;
    constexpr int ENT = SPL * 32;  // V elements per ring entry (W slots x 16 rows)

    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, MPC = p.MPC;
    const int mloc = warp / G, g = warp % G;
    int* wm_all = reinterpret_cast<int*>(smem);       // [MPC] watermarks
    int* abort_flag = wm_all + 32;                    // one flag per block
    V* ring = reinterpret_cast<V*>(smem + 256) + (size_t)mloc * (2 * G) * ENT;
    V* scratch = ring + (size_t)(G + g) * ENT;        // this warp's own-token values
    if (threadIdx.x < 32)
        wm_all[threadIdx.x] = -1;
    if (threadIdx.x == 0)
        *abort_flag = 0;
    __syncthreads();

    const int64_t m = (int64_t)blockIdx.x * MPC + mloc;
    if (m >= p.machines)
        return;
    const int mps = p.d / kScanRows;
    const int64_t b = m / mps;
    const int rs = (int)(m % mps);
    const int sg = lane >> 2, rg = lane & 3;
    const int row0 = rs * kScanRows + rg * 4;
    const int d = p.d, N = p.N, T = p.T;
    S* bank = reinterpret_cast<S*>(p.banks) + (size_t)b * N * d;
    const S* vsrc = reinterpret_cast<const S*>(p.v);
    int* wm = wm_all + mloc;

    for (int t = g; t < T; t += G) {
        const size_t tok = (size_t)b * T + t;
        const size_t wb = tok * 2 * W + sg * SPL;
        const size_t rb = wb + W;
        int32_t widx[SPL], ridx[SPL];
        uint16_t wc[SPL], rc[SPL];
        load_ids<SPL>(p.idx + wb, widx);
        load_ids<SPL>(p.idx + rb, ridx);
        load_codes<SPL>(p.codes + wb, wc);
        load_codes<SPL>(p.codes + rb, rc);

        // Loads of slots that are not forwarded. Every token <= t-G has committed
        // (our own previous token was t-G), so global memory is current for them.
        V wd[SPL], rd[SPL];
        bool wok[SPL];
        int need = -1;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const int dt = wc[i] >> 8;
            const bool fwd = wc[i] != kNoFwd && dt < G;
            wok[i] = widx[i] >= 0 && widx[i] < N;
            wd[i] = R4::zero();
            if (fwd)
                need = max(need, t - dt);
            else if (wok[i])
                wd[i] = R4::load_cg(bank + (size_t)widx[i] * d + row0);
        }
        int rneed = -1;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const int dt = rc[i] >> 8;
            const bool fwd = rc[i] != kNoFwd && dt < G;
            const bool ok = ridx[i] >= 0 && ridx[i] < N;
            rd[i] = R4::zero();
            if (fwd) {
                if (dt > 0)
                    rneed = max(rneed, t - dt);
            } else if (ok) {
                rd[i] = R4::load_cg(bank + (size_t)ridx[i] * d + row0);
            }
            if (!ok)
                report(p.status, SDM_ERANGE);
        }
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            if (!wok[i])
                report(p.status, SDM_ERANGE);

        float wk[SPL], rk[SPL];
        load_w<SPL>(p.wsel + wb, wk);
        load_w<SPL>(p.wsel + rb, rk);
        float vv[4];
        R4::to_f32(R4::load_cg(vsrc + tok * d + row0), vv);
        const float a = __ldg(p.alpha + tok), be = __ldg(p.beta + tok);

        // write slots last written by one of the previous G-1 tokens: from the ring
        need = __reduce_max_sync(0xFFFFFFFFu, need);
        if (need >= 0) {
            if (!warp_wait_geq(wm, need, abort_flag, p.status))
                return;
#pragma unroll
            for (int i = 0; i < SPL; ++i) {
                const int dt = wc[i] >> 8;
                if (wc[i] != kNoFwd && dt < G) {
                    const int pos = wc[i] & 0xFF;
                    wd[i] = ring[(size_t)((t - dt) % G) * ENT + (pos % SPL) * 32 + (pos / SPL) * 4 + rg];
                }
            }
        }

        // u = M_S k  (pre-write), reduced over the 8 slot groups
        float up[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            float mf[4];
            R4::to_f32(wd[i], mf);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                up[r] = fmaf(wk[i], mf[r], up[r]);
        }
        xor_reduce4(up);
        float c[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            c[r] = be * (vv[r] - a * up[r]);
        // M[S_j] <- alpha M[S_j] + k_j * beta (v - alpha u), rounded once
        V nw[SPL];
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            float mf[4], f[4];
            R4::to_f32(wd[i], mf);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                f[r] = fmaf(wk[i], c[r], a * mf[r]);
            nw[i] = R4::from_f32(f);
        }
        // this token's written values, for its own read of the same slots
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            scratch[i * 32 + lane] = nw[i];
        __syncwarp();

        // read slots written by this token (dt = 0, scratch) or by one of the
        // previous G-1 tokens (ring)
        rneed = __reduce_max_sync(0xFFFFFFFFu, rneed);
        if (rneed >= 0 && !warp_wait_geq(wm, rneed, abort_flag, p.status))
            return;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const int dt = rc[i] >> 8;
            if (rc[i] != kNoFwd && dt < G) {
                const int pos = rc[i] & 0xFF;
                const int off = (pos % SPL) * 32 + (pos / SPL) * 4 + rg;
                rd[i] = dt == 0 ? scratch[off] : ring[(size_t)((t - dt) % G) * ENT + off];
            }
        }
        float yp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            float mf[4];
            R4::to_f32(rd[i], mf);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                yp[r] = fmaf(rk[i], mf[r], yp[r]);
        }
        xor_reduce4(yp);
        if (sg == 0)
            __stcs(reinterpret_cast<float4*>(p.y + tok * d + row0),
                   make_float4(yp[0], yp[1], yp[2], yp[3]));

        // commit in token order: global stores, then the ring entry, then release
        if (!warp_wait_geq(wm, t - 1, abort_flag, p.status))
            return;
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            if (wok[i])
                R4::store_cg(bank + (size_t)widx[i] * d + row0, nw[i]);
        V* ent = ring + (size_t)(t % G) * ENT;
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            ent[i * 32 + lane] = nw[i];
        __threadfence_block();
        __syncwarp();
        if (lane == 0)
            st_release_cta(wm, t);
    }
}

static int pow2_floor(long long x)
{
    int p = 1;
    while ((long long)p * 2 <= x)
        p *= 2;
    return p;
}

ScanLaunch choose_scan_launch(int B, int T, int d, int num_sms)
{
    const long long machines = (long long)B * (d / kScanRows);
    ScanLaunch L{1, 4};
    if (T <= 1)
        return L;  // decode: one token, four independent machines per block
    // about 16 warps per SM in total, at most 16 tokens in flight per machine
    long long want = 16LL * num_sms / (machines > 0 ? machines : 1);
    int G = pow2_floor(want < 1 ? 1 : want);
    if (G > 16)
        G = 16;
    while (G > 1 && G / 2 >= T)
        G /= 2;
    L.G = G;
    L.MPC = G >= 4 ? 1 : 4 / G;
    return L;
}

template <typename S, int SPL>
static cudaError_t launch_scan_t(ScanParams p, cudaStream_t s)
{
    using V = typename Row4<S>::V;
    const size_t smem = 256 + (size_t)p.MPC * 2 * p.G * SPL * 32 * sizeof(V);
    auto kern = scan_kernel<S, SPL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    const int64_t blocks = (p.machines + p.MPC - 1) / p.MPC;
    kern<<<(unsigned)blocks, 32 * p.G * p.MPC, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_scan(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                        const uint16_t* codes, const void* v, const float* alpha,
                        const float* beta, void* banks, float* y, int B, int T, ScanLaunch L,
                        int* status, cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    if (L.G < 1 || L.G > 16 || L.MPC < 1 || L.G * L.MPC > 16 || (L.G & (L.G - 1)) != 0)
        return cudaErrorInvalidValue;
    ScanParams p;
    p.banks = banks;
    p.idx = idx;
    p.wsel = wsel;
    p.codes = codes;
    p.v = v;
    p.alpha = alpha;
    p.beta = beta;
    p.y = y;
    p.status = status;
    p.machines = (int64_t)B * (c.d / kScanRows);
    p.T = T;
    p.d = c.d;
    p.N = c.n_sub * c.n_sub;
    p.G = L.G;
    p.MPC = L.MPC;
    const bool bf = c.dtype == SDM_BF16;
    switch (c.w) {
    case 8: return bf ? launch_scan_t<bf16, 1>(p, s) : launch_scan_t<float, 1>(p, s);
    case 16: return bf ? launch_scan_t<bf16, 2>(p, s) : launch_scan_t<float, 2>(p, s);
    case 32: return bf ? launch_scan_t<bf16, 4>(p, s) : launch_scan_t<float, 4>(p, s);
    case 64: return bf ? launch_scan_t<bf16, 8>(p, s) : launch_scan_t<float, 8>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
