// scan_bwd.cu -- backward of the recurrence: the gradients of the gated-delta write and
// the weighted read ("Sparse Delta Memory" blog, "Write & Read"; the method is trained
// end to end, paper Abstract) with respect to v, alpha, beta, the write and read
// weights and the bank before the tokens.
//
// Forward, per token t: old_j = M[S_j], u = sum_j k_j old_j,
//   M[S_j] <- alpha old_j + beta k_j (v - alpha u),   y = sum_j r_j M[R_j].
// Backward, for t = T-1 .. 0, with G the gradient of the loss with respect to the bank
// state after token t (G starts as the gradient with respect to the final bank):
//   read:   dr_j = <M[R_j], dy>,  G[R_j] += r_j dy              (M: the post-write state)
//   write:  g = sum_j k_j G[S_j],  c = v - alpha u,
//           dv = beta g,  dbeta = <g, c>,  dalpha = sum_j <G[S_j], old_j - beta k_j u>,
//           dk_j = beta <G[S_j], c> - alpha beta <g, old_j>,
//           G[S_j] <- alpha (G[S_j] - beta k_j g),  M[S_j] <- old_j   (from the tape)
// At the end G is the gradient with respect to the bank before the first token, and M
// is that bank again. The stored state is rounded on each write in the forward; the
// backward takes the rounding's derivative as 1 and uses the stored values.
//
// Rows are independent, so a block owns 64 rows of one sequence and walks its tokens in
// reverse; its warps share the W slots of a token (slot j in warp j % 16, or one slot a
// warp for W < 16), each lane two adjacent rows.
// Sums over rows (dk, dr, dalpha, dbeta) are per-block partials, summed over the blocks
// of a sequence by a second kernel.
//
// Latency: a token's gathers (G and M at its read slots, G at its write slots, its tape
// rows, dy and v) are 16-byte cp.async copies into a shared-memory stage, issued one
// token ahead while the token before it in the walk is processed; barriers do not wait
// for them, so the gathers of one token overlap the arithmetic of the other. A slot that
// token then writes is gathered stale. A pre-pass kernel builds per-token slot
// descriptors: for each slot of token t, the position in token t+1 that touched it last;
// token t takes that position's final G value from shared memory instead (token t+1
// leaves there the values token t takes), and gathers M from token t+1's tape row, which
// is the value the restore puts back. The same descriptors name, for a write slot that
// is also read by its own token, the read position, so the read's addition r_j dy is
// applied in registers and no barrier separates the read from the write.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kBRows = 64;
constexpr int kMetaRing = 4;   // token t, t-1 (gathers) and t-2 (being published)

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

// Sums each of the V values of every lane over the warp with V - 1 + log2(32 / V)
// exchanges: each step halves the values a lane keeps, trading the other half with the
// lane `o` away. Lane L ends with the sum of value L / (32 / V).
template <int V>
__device__ __forceinline__ float warp_sum_many(float (&x)[V], int lane)
{
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "a power of two up to 32");
#pragma unroll
    for (int h = V / 2; h >= 1; h >>= 1) {
        const int o = 32 * h / V;
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < h; ++k) {
            const float send = hi ? x[k] : x[k + h];
            const float keep = hi ? x[k + h] : x[k];
            x[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
    }
    float s = x[0];
#pragma unroll
    for (int o = 16 / V; o >= 1; o >>= 1)
        s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    return s;
}

// The pre-pass: one 16-byte descriptor per token t and slot index j < W (positions: write
// j = j, read j = W + j; "next" below is the position of the same slot in token t+1, its
// write position if it has both, or -1: no such slot, an invalid slot, or t the last
// token):
//   offw, offr: the write / read slot's row offset s d within its sequence's bank, or
//               ~0 for an invalid slot;
//   mw byte 0:  next of write position j;   byte 1: next of read position j;
//      byte 2:  the read position of token t with write j's slot, or -1;
//      byte 3:  1 if token t also writes read j's slot, else 0;
//   need byte 0 (1): 1 if token t-1 takes write (read) position j's final G value from
//               token t, else 0 -- the positions that token t must leave in shared memory.
// Slots within one kind of one token are distinct (a top-W selection).
struct BwdDesc {
    uint32_t offw, offr;
    int mw, need;
};

template <int W>
__global__ void __launch_bounds__(2 * W) bwd_prep_kernel(const int32_t* __restrict__ idx, int T,
                                                         int N, int d, BwdDesc* __restrict__ desc)
{
    __shared__ int ps[2 * W], cs[2 * W], ns[2 * W];   // tokens t-1, t, t+1
    const int64_t tok = blockIdx.x;
    const int t = (int)(tok % T);
    const int p = threadIdx.x;
    auto slot = [&](int64_t tk) {
        const int s = __ldg(idx + tk * 2 * W + p);
        return (s < 0 || s >= N) ? -1 : s;
    };
    const int s = slot(tok);
    cs[p] = s;
    ns[p] = t + 1 < T ? slot(tok + 1) : -1;
    ps[p] = t >= 1 ? slot(tok - 1) : -1;
    __syncthreads();
    int src = -1, other = -1, need = 0;
    if (s >= 0) {
        for (int k = 0; k < 2 * W; ++k)
            if (ns[k] == s) {
                src = k;
                break;
            }
        const int base = p < W ? W : 0;   // a write position looks among the reads, and back
        for (int k = 0; k < W; ++k)
            if (cs[base + k] == s) {
                other = k;
                break;
            }
        // token t-1 takes this position's value when it holds the slot, unless this is a
        // read position whose slot token t also writes (the write position serves it)
        if (p < W || other < 0)
            for (int k = 0; k < 2 * W; ++k)
                if (ps[k] == s) {
                    need = 1;
                    break;
                }
    }
    BwdDesc& o = desc[tok * W + p % W];
    int8_t* mw = reinterpret_cast<int8_t*>(&o.mw);
    int8_t* nd = reinterpret_cast<int8_t*>(&o.need);
    const uint32_t off = s >= 0 ? (uint32_t)s * (uint32_t)d : 0xFFFFFFFFu;
    if (p < W) {
        o.offw = off;
        mw[0] = (int8_t)src;
        mw[2] = (int8_t)other;
        nd[0] = (int8_t)need;
        nd[2] = 0;
    } else {
        o.offr = off;
        mw[1] = (int8_t)src;
        mw[3] = (int8_t)(other >= 0 ? 1 : 0);
        nd[1] = (int8_t)need;
        nd[3] = 0;
    }
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }


// Shape of the walk: a block owns 64 rows of one sequence; each warp is a group that
// owns slots j = group + NG i of every token, each lane rows 2 lane and 2 lane + 1 of
// them (so the per-slot index work is shared by two rows and rows move as pairs).
template <int W>
struct BwdShape {
    static constexpr int NG = W < 16 ? W : 16;   // groups (warps)
    static constexpr int threads = NG * 32;
    static constexpr int SPG = W / NG;           // slots a thread
};

// Shared memory of the walk. A token's gathers land in stage t & 1; its metadata in
// ring entry t % 4 (in flight two tokens ahead, read by the gathers issued one token
// ahead and by the token itself).
template <typename S, int W>
struct BwdStage {
    float g[2 * W][kBRows];     // G at the write positions, then at the read positions
    S st[2 * W][kBRows];        // tape rows (write positions), then bank rows (read positions)
    float dy[kBRows];
    S v[kBRows];
};
template <int W>
struct BwdMeta {
    BwdDesc desc[W];            // the token's slot descriptors
    float sw[2 * W];            // the weights: write positions, then read positions
    float gate[4];              // alpha, beta
};
template <typename S, int W>
struct BwdSmem {
    BwdStage<S, W> stage[2];
    BwdMeta<W> meta[kMetaRing];
    float2 xg[2 * W][kBRows / 2];   // the final G values of the previous token, by its position
    float2 red[2][BwdShape<W>::NG][kBRows / 2 + 1];   // per-warp sums g, u (padded rows)
    float2 red2[2][kBRows / 2];                       // their sums over the warps
    float acc[2][2 * W + 2];        // partial sums of token t in entry t & 1
};

__device__ __forceinline__ float2 ld_pair(const bf16* p)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 ld_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ void st_pair(bf16* p, float2 x)
{
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x.x, x.y);
}
__device__ __forceinline__ void st_pair(float* p, float2 x) { *reinterpret_cast<float2*>(p) = x; }
__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }
__device__ __forceinline__ float dot2(float2 a, float2 b) { return fmaf(a.x, b.x, a.y * b.y); }

// partials: [nblk][B*T][2W + 2] = dk[W], dr[W], dalpha, dbeta of this block's rows
template <typename S, int W>
__global__ void __launch_bounds__(BwdShape<W>::threads, 1) scan_bwd_kernel(
    const BwdDesc* __restrict__ desc, const float* __restrict__ wsel,
    const S* __restrict__ v, const float* __restrict__ alpha,
    const float* __restrict__ beta, const S* __restrict__ tape, S* __restrict__ banks,
    const float* __restrict__ dy, float* __restrict__ dbank, float* __restrict__ dv,
    float* __restrict__ part, int B, int T, int d, int N)
{
    constexpr int NG = BwdShape<W>::NG, NT = BwdShape<W>::threads, SPG = BwdShape<W>::SPG;
    constexpr int P = 2 * W + 2;
    constexpr int GCH = kBRows * 4 / 16;      // 16-byte chunks of a G row segment
    constexpr int SCH = kBRows * (int)sizeof(S) / 16;
    static_assert(P <= NT, "one partial sum a thread");
    static_assert(NT >= 194, "the metadata copies' thread ranges");
    static_assert(SPG >= 1 && 32 % SPG == 0, "whole lanes per reduced value");
    static_assert(W <= 64, "metadata copies fit their thread ranges");
    static_assert(NT % 64 == 0 && 2 * (NT / 64) == NG, "two warps' partials a lane in the sum of g, u");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<S, W>& sm = *reinterpret_cast<BwdSmem<S, W>*>(smem_raw);
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int grp = tid >> 5, lane = tid & 31;
    const int rr = 2 * lane;                  // the lane's first row within the block
    const int row0 = blockIdx.x * kBRows;
    const int row = row0 + rr;
    const int nrows = min(kBRows, d - row0);  // a multiple of 16: d is
    const bool act = rr < nrows;              // both rows, nrows being even
    S* bank = banks + (size_t)b * N * d;
    float* G = dbank + (size_t)b * N * d;
    if (T <= 0)
        return;
    const int64_t tok0 = (int64_t)b * T;

    // token tk's slot descriptors, weights and gates into ring entry mb
    auto issue_meta = [&](int64_t tk, int mb) {
        BwdMeta<W>& m = sm.meta[mb];
        if (tid < W)
            cp_async16(smem_u32(&m.desc[tid]), desc + tk * W + tid);
        else if (tid >= 64 && tid < 64 + W / 2)
            cp_async16(smem_u32(&m.sw[(tid - 64) * 4]), wsel + tk * 2 * W + (tid - 64) * 4);
        else if (tid == 192)
            cp_async4(smem_u32(&m.gate[0]), alpha + tk);
        else if (tid == 193)
            cp_async4(smem_u32(&m.gate[1]), beta + tk);
    };
    // token tk's gathers into stage gb, its metadata in ring entry mb (landed). Issued
    // before the token after it (tk + 1) stores anything: the slots that token writes
    // are loaded stale here and replaced from xg when token tk runs.
    auto issue_gathers = [&](int64_t tk, int mb, int gb) {
        const BwdMeta<W>& m = sm.meta[mb];
        BwdStage<S, W>& g = sm.stage[gb];
        const int gch = nrows * 4 / 16, sch = nrows * (int)sizeof(S) / 16;
        // a thread's chunks are the same every token: fixed trip counts
        constexpr int GIT = (2 * W * GCH + NT - 1) / NT, SIT = (2 * W * SCH + NT - 1) / NT;
#pragma unroll
        for (int it = 0; it < GIT; ++it) {
            const int k = tid + it * NT;
            const int p = k / GCH, c = k % GCH;
            if (k >= 2 * W * GCH || c >= gch)
                continue;
            const uint32_t off = (&m.desc[p % W].offw)[p / W];   // offw, then offr
            if (off != 0xFFFFFFFFu)
                cp_async16(smem_u32(&g.g[p][c * 4]), G + (off + row0 + c * 4));
        }
#pragma unroll
        for (int it = 0; it < SIT; ++it) {
            const int k = tid + it * NT;
            const int p = k / SCH, c = k % SCH;
            if (k >= 2 * W * SCH || c >= sch)
                continue;
            const uint32_t off = (&m.desc[p % W].offw)[p / W];
            if (off == 0xFFFFFFFFu)
                continue;
            const int e16 = c * (16 / (int)sizeof(S));
            const S* src;
            if (p < W) {
                src = tape + ((size_t)tk * W + p) * d;   // the pre-write row of the write
            } else {
                // the bank after token tk's write: token tk + 1's pre-write row if it
                // wrote the slot (the value its restore puts back), else the bank row
                const int q = (int8_t)(m.desc[p - W].mw >> 8);
                src = (q >= 0 && q < W) ? tape + ((size_t)(tk + 1) * W + q) * d : bank + off;
            }
            cp_async16(smem_u32(&g.st[p][e16]), src + row0 + e16);
        }
        if (tid < nrows / 4)
            cp_async16(smem_u32(&g.dy[tid * 4]), dy + tk * d + row0 + tid * 4);
        else if (tid >= 32 && tid - 32 < sch)
            cp_async16(smem_u32(&g.v[(tid - 32) * (16 / (int)sizeof(S))]),
                       v + tk * d + row0 + (tid - 32) * (16 / (int)sizeof(S)));
    };

    issue_meta(tok0 + T - 1, (T - 1) % kMetaRing);
    if (T >= 2)
        issue_meta(tok0 + T - 2, (T - 2) % kMetaRing);
    cp_async_commit();
    if (tid < P) {
        sm.acc[0][tid] = 0.f;
        sm.acc[1][tid] = 0.f;
    }
    cp_async_wait_all();
    __syncthreads();
    issue_gathers(tok0 + T - 1, (T - 1) % kMetaRing, (T - 1) & 1);
    cp_async_commit();
    const float2 zero2 = make_float2(0.f, 0.f);
    for (int t = T - 1; t >= 0; --t) {
        const int64_t tok = tok0 + t;
        const int mb = t % kMetaRing, cb = t & 1;
        // token t's gathers and token t - 1's metadata have landed (issued during token
        // t + 1); token t + 1's xg, partial sums and stores are complete
        cp_async_wait_all();
        __syncthreads();
        if (t + 1 < T && tid < P) {
            part[((size_t)blockIdx.x * B * T + tok + 1) * P + tid] = sm.acc[cb ^ 1][tid];
            sm.acc[cb ^ 1][tid] = 0.f;   // token t - 1 adds into it after the next barrier
        }
        if (t >= 1)
            issue_gathers(tok - 1, (t - 1) % kMetaRing, cb ^ 1);
        if (t >= 2)
            issue_meta(tok - 2, (t - 2) % kMetaRing);
        cp_async_commit();

        const BwdMeta<W>& m = sm.meta[mb];
        const BwdStage<S, W>& g = sm.stage[cb];
        const float2 dy2 = act ? *reinterpret_cast<const float2*>(&g.dy[rr]) : zero2;
        // ---- this token's values: G from the previous token's final values where it
        // touched the slot, else as gathered. Offsets within a sequence's bank fit 32 bits.
        // All shared-memory loads of the token first (descriptors, weights, then the
        // values they select), so that no load waits behind a store and the slots'
        // dependency chains interleave; then the arithmetic and the stores.
        int4 dd[SPG];
        float kw[SPG], rwt[SPG], rmw[SPG];
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int j = grp + NG * i;
            dd[i] = *reinterpret_cast<const int4*>(&m.desc[j]);
            kw[i] = m.sw[j];
            rwt[i] = m.sw[W + j];
        }
        float2 gw[SPG], gr[SPG], ow[SPG], mr[SPG];
        uint32_t offw[SPG], offr[SPG];   // G / bank offsets of the slots' rows, or ~0
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int j = grp + NG * i;
            const int mw = dd[i].z;
            const int qw = (int8_t)mw, qr = (int8_t)(mw >> 8), rm = (int8_t)(mw >> 16);
            const bool okw = act && (uint32_t)dd[i].x != 0xFFFFFFFFu;
            const bool okr = act && (uint32_t)dd[i].y != 0xFFFFFFFFu;
            offw[i] = okw ? (uint32_t)dd[i].x + (uint32_t)row : 0xFFFFFFFFu;
            offr[i] = okr ? (uint32_t)dd[i].y + (uint32_t)row : 0xFFFFFFFFu;
            // G: the previous token's final value where it touched the slot, else as
            // gathered
            const float2* pw = qw >= 0 ? sm.xg[qw] : reinterpret_cast<const float2*>(g.g[j]);
            const float2* pq = qr >= 0 ? sm.xg[qr] : reinterpret_cast<const float2*>(g.g[W + j]);
            gw[i] = okw ? pw[lane] : zero2;
            gr[i] = okr ? pq[lane] : zero2;
            ow[i] = okw ? ld_pair(&g.st[j][rr]) : zero2;
            mr[i] = okr ? ld_pair(&g.st[W + j][rr]) : zero2;
            rmw[i] = rm >= 0 ? m.sw[W + rm] : 0.f;
        }
        // ---- read: dr_j = <M[R_j], dy> (M after this token's write), G[R_j] += r_j dy
        float pr[SPG];
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            pr[i] = dot2(mr[i], dy2);
            if (offr[i] != 0xFFFFFFFFu && (dd[i].z >> 24) == 0)   // else the write stores it
                st_pair(G + offr[i], __ffma2_rn(dup(rwt[i]), dy2, gr[i]));
        }
        // ---- write: G at the write slots after the read's additions
        float2 gp = zero2, up = zero2;
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            if ((int8_t)(dd[i].z >> 16) >= 0)
                gw[i] = __ffma2_rn(dup(rmw[i]), dy2, gw[i]);
            const float2 k2 = dup(kw[i]);
            gp = __ffma2_rn(k2, gw[i], gp);
            up = __ffma2_rn(k2, ow[i], up);
        }
        sm.red[0][grp][lane] = gp;
        sm.red[1][grp][lane] = up;
        {
            const float sum = warp_sum_many<SPG>(pr, lane);
            if (lane % (32 / SPG) == 0)
                atomicAdd(&sm.acc[cb][W + grp + NG * (lane / (32 / SPG))], sum);
        }
        __syncthreads();   // red complete; every thread has read xg
        {
            // g, u summed over the warps: TPO adjacent lanes share one (quantity, row
            // pair), each adding two warps' partials, then exchange
            constexpr int TPO = NT / 64;
            const int o = tid / TPO, part = tid % TPO;
            float2 sum = __fadd2_rn(sm.red[o >> 5][2 * part][o & 31], sm.red[o >> 5][2 * part + 1][o & 31]);
#pragma unroll
            for (int x = 1; x < TPO; x <<= 1) {
                sum.x += __shfl_xor_sync(0xFFFFFFFFu, sum.x, x);
                sum.y += __shfl_xor_sync(0xFFFFFFFFu, sum.y, x);
            }
            if (part == 0)
                sm.red2[o >> 5][o & 31] = sum;
        }
        __syncthreads();   // red2 complete
        const float2 gs = sm.red2[0][lane], u = sm.red2[1][lane];
        const float al = m.gate[0], be = m.gate[1];
        const float2 c = __ffma2_rn(dup(-al), u, act ? ld_pair(&g.v[rr]) : zero2);
        float pa = 0.f;
        float pk[SPG];
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int j = grp + NG * i;
            const float bk = be * kw[i];
            // dalpha: <G_j, old_j - beta k_j u>;  dk_j: beta <G_j, c> - alpha beta <g, old_j>
            pa += dot2(gw[i], __ffma2_rn(dup(-bk), u, ow[i]));
            pk[i] = be * dot2(gw[i], c) - al * be * dot2(gs, ow[i]);
            const float2 gn = __fmul2_rn(dup(al), __ffma2_rn(dup(-bk), gs, gw[i]));
            if (offw[i] != 0xFFFFFFFFu) {
                st_pair(G + offw[i], gn);
                // the tape value, stored back exactly (a stored value converts to fp32
                // and back unchanged)
                st_pair(bank + offw[i], ow[i]);
            }
            if (dd[i].w & 0xFF)   // only what token t - 1 takes from this token
                sm.xg[j][lane] = gn;
            if (dd[i].w & 0xFF00)
                sm.xg[W + j][lane] = __ffma2_rn(dup(rwt[i]), dy2, gr[i]);
        }
        {
            const float sum = warp_sum_many<SPG>(pk, lane);
            if (lane % (32 / SPG) == 0)
                atomicAdd(&sm.acc[cb][grp + NG * (lane / (32 / SPG))], sum);
        }
        pa = warp_sum(pa);
        const float pb = warp_sum(grp == 0 ? dot2(gs, c) : 0.f);
        if (lane == 0) {
            atomicAdd(&sm.acc[cb][2 * W], pa);
            atomicAdd(&sm.acc[cb][2 * W + 1], pb);
        }
        if (grp == 0 && act)
            *reinterpret_cast<float2*>(dv + tok * d + row) = __fmul2_rn(dup(be), gs);
        // red, xg and the stage are rewritten only after the next token's first barrier
    }
    __syncthreads();
    if (tid < P)
        part[((size_t)blockIdx.x * B * T + tok0) * P + tid] = sm.acc[0][tid];
}

// sums of the per-block partials: dwsel [B*T][2][W] (write weights, then read weights),
// dalpha, dbeta [B*T]
__global__ void __launch_bounds__(256) scan_bwd_reduce(const float* __restrict__ part, int nblk,
                                                      int64_t ntok, int W, float* __restrict__ dwsel,
                                                      float* __restrict__ dalpha,
                                                      float* __restrict__ dbeta)
{
    const int P = 2 * W + 2;
    const int64_t total = ntok * P;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        float sum = 0.f;
        for (int k = 0; k < nblk; ++k)
            sum += part[(size_t)k * total + e];
        const int64_t tok = e / P;
        const int q = (int)(e % P);
        if (q < 2 * W)
            dwsel[tok * 2 * W + q] = sum;
        else if (q == 2 * W)
            dalpha[tok] = sum;
        else
            dbeta[tok] = sum;
    }
}

template <typename S, int W>
cudaError_t launch_bwd_t(const int32_t* idx, const float* wsel, BwdDesc* desc, const void* v,
                         const float* alpha, const float* beta, const void* tape, void* banks,
                         const float* dy, float* dbank, float* dv, float* part, int B, int T, int d,
                         int N, cudaStream_t s)
{
    bwd_prep_kernel<W><<<(unsigned)((int64_t)B * T), 2 * W, 0, s>>>(idx, T, N, d, desc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)((d + kBRows - 1) / kBRows), (unsigned)B);
    const size_t smem = sizeof(BwdSmem<S, W>);
    e = cudaFuncSetAttribute(scan_bwd_kernel<S, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess)
        return e;
    scan_bwd_kernel<S, W><<<grid, BwdShape<W>::threads, smem, s>>>(
        desc, wsel, (const S*)v, alpha, beta, (const S*)tape, (S*)banks, dy, dbank, dv, part, B, T,
        d, N);
    return cudaGetLastError();
}

// workspace: the per-block partials, then the slot descriptors
size_t part_bytes(const sdm_cfg& c, int B, int T)
{
    const size_t nblk = (size_t)(c.d + kBRows - 1) / kBRows;
    return (nblk * (size_t)B * T * (2 * c.w + 2) * sizeof(float) + 255) / 256 * 256;
}

}  // namespace

size_t scan_backward_ws_bytes(const sdm_cfg& c, int B, int T)
{
    return part_bytes(c, B, T) + (size_t)B * T * c.w * sizeof(BwdDesc);
}

cudaError_t launch_scan_backward(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                                 const void* v, const float* alpha, const float* beta,
                                 const void* tape, void* banks, const float* dy, float* dbank,
                                 float* dv, float* dalpha, float* dbeta, float* dwsel, int B,
                                 int T, void* ws, cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    if ((int64_t)B * T > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    const int N = c.n_sub * c.n_sub;
    if ((uint64_t)N * (uint64_t)c.d > 0xFFFFFFFFull)   // offsets within a bank are 32-bit
        return cudaErrorInvalidValue;
    float* part = (float*)ws;
    BwdDesc* desc = (BwdDesc*)((char*)ws + part_bytes(c, B, T));
    const bool bf = c.dtype == SDM_BF16;
    cudaError_t e;
#define SDM_BWD(WW)                                                                                \
    (bf ? launch_bwd_t<bf16, WW>(idx, wsel, desc, v, alpha, beta, tape, banks, dy, dbank, dv,      \
                                 part, B, T, c.d, N, s)                                            \
        : launch_bwd_t<float, WW>(idx, wsel, desc, v, alpha, beta, tape, banks, dy, dbank, dv,     \
                                  part, B, T, c.d, N, s))
    switch (c.w) {
    case 8: e = SDM_BWD(8); break;
    case 16: e = SDM_BWD(16); break;
    case 32: e = SDM_BWD(32); break;
    case 64: e = SDM_BWD(64); break;
    default: return cudaErrorInvalidValue;
    }
#undef SDM_BWD
    if (e != cudaSuccess)
        return e;
    const int nblk = (c.d + kBRows - 1) / kBRows;
    const int64_t work = (int64_t)B * T * (2 * c.w + 2);
    int64_t blocks = (work + 255) / 256;
    if (blocks > (int64_t)num_sms_current_device() * 8)
        blocks = (int64_t)num_sms_current_device() * 8;
    scan_bwd_reduce<<<(unsigned)blocks, 256, 0, s>>>(part, nblk, (int64_t)B * T, c.w, dwsel, dalpha,
                                                     dbeta);
    return cudaGetLastError();
}

}  // namespace sdm
