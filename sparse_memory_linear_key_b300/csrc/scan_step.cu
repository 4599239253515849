// scan_step.cu -- the recurrence for one token a sequence (a decode step), every item in
// one wave ("Sparse Delta Memory" blog, "Write & Read": selected columns are decayed, then
// written with the delta rule; the output is the weighted sum of the read columns after
// the write). The arithmetic is scan.cu's (scan_math.cuh), in the same order, so both
// give the same bits.
//
// With one token a sequence the items -- (sequence, row block of 1 KB) -- are
// independent: no token reads what another writes, and none of the persistent scan's
// ordering (progress flags, forwarding ring, window) applies. One CTA per item, 16 warps
// in scan.cu's consumer layout (a thread: 16 bytes of rows of the slots i*8 + its slot
// group):
//  1. the token's slot ids and weights into shared memory (v is loaded first);
//  2. each read of a slot the token also writes is matched to its write position (binary
//     search over the ascending write set); every other read chunk is gathered from the
//     bank into the read buffer by bulk copies, at once (rows of out-of-range ids are
//     zeroed: their weight is 0);
//  3. each thread loads its write chunks from the bank into registers, forms u, the new
//     values (rounded once) and their bank stores, and puts the new values of the token's
//     own reads into their rows of the read buffer;
//  4. y on the tensor cores (mma.sync over the read buffer, the read weights in two bf16
//     parts), as scan.cu computes it.
// A CTA holds the read buffer alone (about 69 KB) at 64 registers a thread, so two CTAs
// share an SM: 64 sequences x 4 row blocks at d = 2048 run in one wave of 256 CTAs, where
// the persistent kernel takes two items on most SMs one after the other. bf16 state with
// W >= 16 only (the tensor-core read); the persistent kernel takes every other case.
#include "scan_math.cuh"
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kStepThreads = 512;    // 16 warps x 4 row groups of 16 bytes = 1 KB
constexpr int kStepRS = 1040;        // read-buffer row stride (ldmatrix phases spread)

struct StepArgs {
    unsigned char* banks;
    const int32_t* idx;      // [B][2][W]
    const float* wsel;       // [B][2][W]
    const unsigned char* v;  // [B][d]
    const float* alpha;
    const float* beta;
    float* y;                // [B][d]
    int* status;
    int d, N, nrb, rb_rows;
};

__device__ __forceinline__ uint4 ld_u4(const unsigned char* p)
{
    return *reinterpret_cast<const uint4*>(p);
}

template <int W>
__global__ void __launch_bounds__(kStepThreads, 2) scan_step_kernel(StepArgs a)
{
    using S = bf16;
    using P = Pack16<S>;
    constexpr int SPL = W / kSG;       // slots of each set per thread: i*8 + sg
    constexpr int HPL = P::H;          // fp32 pairs per thread
    constexpr int NB = (W / 16) * 64;  // B-fragment words
    extern __shared__ __align__(16) unsigned char sm[];
    unsigned char* rbuf = sm;                                          // [W][kStepRS]
    int* sid = reinterpret_cast<int*>(sm + W * kStepRS);               // [2W] ids, -1 out of range
    float* sw = reinterpret_cast<float*>(sid + 2 * W);                 // [2W] weights
    uint32_t* bfr = reinterpret_cast<uint32_t*>(sw + 2 * W);           // [W/16][32][2]
    int* wpub = reinterpret_cast<int*>(bfr + NB);                      // [W] read pos of write i
    uint64_t* bar = reinterpret_cast<uint64_t*>(wpub + W);             // read chunks landed
    __shared__ float ab[2];

    const int item = (int)blockIdx.x;
    const int b = item / a.nrb, rb = item % a.nrb;
    const int rows = min(a.rb_rows, a.d - rb * a.rb_rows);
    const uint32_t cb = (uint32_t)rows * (uint32_t)sizeof(S);
    const int ct = threadIdx.x, w = ct >> 5, lane = ct & 31;
    const int sg = lane >> 2;
    const int rg = w * 4 + (lane & 3);
    const bool act = rg * 16 < rows * (int)sizeof(S);
    if (ct == 0) {
        mbar_init(smem_u32(bar), W);      // one arrival per read position
        fence_mbarrier_init();
    }
    // everything below reads what the kernels before wrote (a programmatic launch starts
    // before they end)
    griddep_wait();
    griddep_launch();

    // v (independent of the slot sets) first
    const uint4 vraw = act ? ld_u4(a.v + ((size_t)b * a.d + (size_t)rb * a.rb_rows) * sizeof(S) + rg * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
    // 1. slot ids and weights of the token (b: one token a sequence)
    const size_t tb = (size_t)b * 2 * W;
    if (ct < 2 * W) {
        const int id = __ldg(a.idx + tb + ct);
        const bool ok = id >= 0 && id < a.N;
        if (!ok)
            report(a.status, SDM_ERANGE);
        sid[ct] = ok ? id : -1;
        sw[ct] = __ldg(a.wsel + tb + ct);
    }
    if (ct < W)
        wpub[ct] = -1;
    if (ct == 0) {
        ab[0] = __ldg(a.alpha + b);
        ab[1] = __ldg(a.beta + b);
    }
    __syncthreads();
    // 2. reads of slots the token writes: the write position of the same slot (their rows
    // take the new values later); every other read chunk in range from the bank, at once
    // (rows of out-of-range ids zeroed)
    unsigned char* wrow = a.banks + ((size_t)b * a.N * a.d + (size_t)rb * a.rb_rows) * sizeof(S) + rg * 16;
    if (ct < W) {
        const int r = sid[W + ct];
        int src = -1;
        if (r >= 0) {
            int lo = 0, hi = W;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (sid[mid] < r)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            if (lo < W && sid[lo] == r)
                src = lo;
        }
        if (src >= 0)
            wpub[src] = ct;
        unsigned char* dst = rbuf + (size_t)ct * kStepRS;
        if (r >= 0 && src < 0) {
            mbar_arrive_expect_tx(smem_u32(bar), cb);
            bulk_g2s(smem_u32(dst), wrow - rg * 16 + (size_t)r * a.d * sizeof(S), cb, smem_u32(bar));
        } else {
            if (r < 0) {
                for (uint32_t o = 0; o < cb; o += 16)
                    *reinterpret_cast<uint4*>(dst + o) = make_uint4(0u, 0u, 0u, 0u);
            }
            mbar_arrive(smem_u32(bar));
        }
    }
    // 3. the write chunks of this thread (read twice -- for u, then again from L1 or L2 for
    // the new values -- so that no thread holds all of them while it forms the new ones;
    // nothing writes a chunk before its thread's second read, as each thread stores only its
    // own pieces, after reading them)
    uint4 q[SPL];
#pragma unroll
    for (int i = 0; i < SPL; ++i) {
        const int id = sid[i * kSG + sg];
        q[i] = act && id >= 0 ? ld_u4(wrow + (size_t)id * a.d * sizeof(S)) : make_uint4(0u, 0u, 0u, 0u);
    }
    // while they load: the read's B fragments, [k-step][lane][2] flat, as scan.cu builds them
    for (int e = ct; e < NB; e += kStepThreads) {
        const int reg = e & 1, ln = (e >> 1) & 31, ks = e >> 6;
        const int g = ln >> 2, j = 16 * ks + 2 * (ln & 3) + 8 * reg;
        const float w0 = sid[W + j] >= 0 ? sw[W + j] : 0.f;
        const float w1 = sid[W + j + 1] >= 0 ? sw[W + j + 1] : 0.f;
        bfr[e] = weight_part_bits(w0, g) | (weight_part_bits(w1, g) << 16);
    }
    float2 u[HPL];
#pragma unroll
    for (int h = 0; h < HPL; ++h)
        u[h] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < SPL; ++i) {
        const float kw = sw[i * kSG + sg];
        float2 f[HPL];
        P::unpack(q[i], f);
#pragma unroll
        for (int h = 0; h < HPL; ++h)
            u[h] = __ffma2_rn(make_float2(kw, kw), f[h], u[h]);
    }
    float2 vv[HPL];
    P::unpack(vraw, vv);
    const float al = ab[0], be = ab[1];
    const float2 al2 = make_float2(al, al), be2 = make_float2(be, be);
    float2 c[HPL];   // beta (v - alpha u)
#pragma unroll
    for (int h = 0; h < HPL; ++h)
        c[h] = __fmul2_rn(be2, __ffma2_rn(make_float2(-al, -al), slot_group_sum(u[h]), vv[h]));
    // M[S_j] <- alpha M[S_j] + k_j beta (v - alpha u), rounded once, to the bank
#pragma unroll
    for (int i = 0; i < SPL; ++i) {
        const int id = sid[i * kSG + sg];
        const float kw = sw[i * kSG + sg];
        float2 f[HPL];
        P::unpack(act && id >= 0 ? ld_u4(wrow + (size_t)id * a.d * sizeof(S)) : make_uint4(0u, 0u, 0u, 0u), f);
#pragma unroll
        for (int h = 0; h < HPL; ++h)
            f[h] = __ffma2_rn(make_float2(kw, kw), c[h], __fmul2_rn(al2, f[h]));
        q[i] = P::pack(f);
        if (act && id >= 0)
            __stcg(reinterpret_cast<uint4*>(wrow + (size_t)id * a.d * sizeof(S)), q[i]);
    }
    __syncthreads();   // (wpub complete)
    // the reads of this token's own writes take the new values
#pragma unroll
    for (int i = 0; i < SPL; ++i) {
        const int jr = wpub[i * kSG + sg];
        if (act && jr >= 0)
            *reinterpret_cast<uint4*>(rbuf + (size_t)jr * kStepRS + rg * 16) = q[i];
    }
    __syncthreads();   // (the own reads are in the read buffer)
    const bool landed = mbar_wait(smem_u32(bar), 0, nullptr, a.status);

    // 4. y = sum_j r_j M[R_j] (post-write): warp w takes rows 32w .. 32w+31 in two 16-row
    // tiles, W / 16 steps of 16 slots, fp32 accumulation
    if (landed) {
        const int gid = lane >> 2, tig = lane & 3;
        const uint32_t rbase = smem_u32(rbuf) + (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * kStepRS) +
                               (uint32_t)(16 * ((lane >> 3) & 1));
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
            const int m0 = w * 32 + 16 * t2;
            if (m0 >= rows)
                break;                                   // (warp-uniform)
            float cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < W / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                             : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                             : "r"(rbase + (uint32_t)(ks * 16 * kStepRS) + (uint32_t)(m0 * 2)));
                const uint2 bb = reinterpret_cast<const uint2*>(bfr)[ks * 32 + lane];
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                    "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                    : "+f"(cc[0]), "+f"(cc[1]), "+f"(cc[2]), "+f"(cc[3])
                    : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(bb.x), "r"(bb.y));
            }
            // columns 0 and 1 (the two parts of the weights) are in lanes tig = 0
            if (tig == 0) {
                float* yp = a.y + (size_t)b * a.d + (size_t)rb * a.rb_rows + m0 + gid;
                __stcs(yp, cc[0] + cc[1]);
                __stcs(yp + 8, cc[2] + cc[3]);
            }
        }
    } else if (ct == 0) {
        mbar_drain(smem_u32(bar), 0, kSpinLimitCycles);   // (copies land before the CTA ends)
    }
}

template <int W>
size_t step_smem()
{
    return (size_t)W * kStepRS + 2 * W * 4 * 2 + (size_t)(W / 16) * 64 * 4 + W * 4 + 16;
}

template <int W>
cudaError_t launch_step_t(const StepArgs& a, int items, cudaStream_t s, bool early)
{
    auto kern = scan_step_kernel<W>;
    const size_t smem = step_smem<W>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)items, 1, 1);
    cfg.blockDim = dim3(kStepThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool scan_step_supported(const sdm_cfg& c)
{
    return c.dtype == SDM_BF16 && (c.w == 16 || c.w == 32 || c.w == 64);
}

cudaError_t launch_scan_step(const sdm_cfg& c, const int32_t* idx, const float* wsel, const void* v,
                             const float* alpha, const float* beta, void* banks, float* y, int B,
                             int* status, cudaStream_t s, bool early)
{
    if (B <= 0)
        return cudaSuccess;
    const ScanWs L = scan_ws_layout(c, B, 1);
    StepArgs a;
    a.banks = (unsigned char*)banks;
    a.idx = idx;
    a.wsel = wsel;
    a.v = (const unsigned char*)v;
    a.alpha = alpha;
    a.beta = beta;
    a.y = y;
    a.status = status;
    a.d = c.d;
    a.N = c.n_sub * c.n_sub;
    a.nrb = L.nrb;
    a.rb_rows = L.rb_rows;
    const long long items = (long long)B * L.nrb;
    if (items > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    switch (c.w) {
    case 16: return launch_step_t<16>(a, (int)items, s, early);
    case 32: return launch_step_t<32>(a, (int)items, s, early);
    case 64: return launch_step_t<64>(a, (int)items, s, early);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
