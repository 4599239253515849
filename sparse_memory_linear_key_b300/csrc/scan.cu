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
// Work unit ("item"): one token of one sequence on one row block -- 1 KB of every slot
// vector (512 rows in bf16, 256 in fp32). Rows evolve independently, so the row blocks
// of a sequence are independent streams of tokens. Each item moves 2 x W gathered 1 KB
// chunks in and W chunks out: random 1 KB chunks are what HBM serves near its copy
// bandwidth (32-byte gathers reach only about a sixth of it).
//
// Persistent kernel, one CTA per SM, items claimed in increasing order from a global
// counter (t-major, so every stream advances together). Per CTA:
//  * a producer warp claims the next item and gathers its W write chunks into the write
//    buffer and its W read chunks (plus weights and v) into one of two read buffers with
//    cp.async.bulk, while
//  * 8 consumer warps compute the current item: they copy the write chunks into
//    registers (freeing the write buffer for the next item at once), form u, wait for
//    the write-after-read clearance, store the new slot values straight to HBM, and
//    reduce the read chunks into y.
// Ordering between tokens of one stream, which may run on different SMs, goes through
// one progress flag per item in global memory (1 = its chunks are loaded, 2 = its
// writes are visible):
//  * read after write: a reference whose latest earlier writer lies within the last
//    kFwdWindow tokens (from the collision codes) waits for that writer's flag = 2
//    before its chunk is copied; a read of a slot the same token writes (distance 0) is
//    not loaded but forwarded from the new values in shared memory;
//  * write after read: the stores of token t wait until tokens t-kFwdWindow .. t-1 have
//    loaded (flag >= 1);
//  * window: token t starts only when tokens t-2*kFwdWindow+1 .. t-kFwdWindow are
//    committed, so every older writer is visible and every older reader done.
// Every wait is bounded: on time-out the kernel records SDM_ETIMEOUT, raises a global
// abort flag that all CTAs watch, waits for its own copies in flight and leaves.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kChunk = 1024;       // bytes of one slot's row block
constexpr int kCWarps = 8;         // consumer warps
constexpr int kScanThreads = 32 * (kCWarps + 1);
constexpr int kMaxW = 64;

struct ScanArgs {
    unsigned char* banks;
    const int32_t* idx;
    const float* wsel;
    const uint16_t* codes;
    const unsigned char* v;
    const float* alpha;
    const float* beta;
    float* y;
    int* status;
    int* flags;                     // [B][nrb][T] progress of each item
    unsigned long long* counter;    // next item to claim
    int* abort_flag;
    long long items;                // B * T * nrb
    int B, T, d, N, nrb, rb_rows;
};

// Everything the consumers need about one item besides the chunks.
struct __align__(16) Meta {
    float wsel[2 * kMaxW];          // write weights, then read weights (bulk copy target)
    unsigned char v[kChunk];        // v rows of this row block (bulk copy target)
    int wid[kMaxW];                 // write slot ids, -1 if out of range
    signed char fpos[kMaxW];        // read ref j: its position in the write set if the
                                    // token writes that slot itself, else -1
    unsigned long long fmask;       // bit j: read ref j is such a forwarded slot
    long long tok;                  // b * T + t
    int b, t, rb, rows;
    float alpha, beta;
    int valid;                      // 0: no more work
};

enum { kFullW = 0, kEmptyW = 1, kFullR = 2, kEmptyR = 4, kWar = 6, kCbar = 8, kNumBars = 9 };

template <typename S>
struct Pack16;

template <>
struct Pack16<bf16> {
    static constexpr int R = 8;
    static __device__ __forceinline__ void unpack(const uint4& q, float (&f)[8])
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    // round-to-nearest-even, once per value
    static __device__ __forceinline__ uint4 pack(const float (&f)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Pack16<float> {
    static constexpr int R = 4;
    static __device__ __forceinline__ void unpack(const uint4& q, float (&f)[4])
    {
        f[0] = __uint_as_float(q.x);
        f[1] = __uint_as_float(q.y);
        f[2] = __uint_as_float(q.z);
        f[3] = __uint_as_float(q.w);
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[4])
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

__device__ __forceinline__ int warp_sum(int x) { return __reduce_add_sync(0xFFFFFFFFu, x); }

// ------------------------------------------------------------------ producer warp

template <typename S, int W>
__device__ void scan_producer(const ScanArgs& a, unsigned char* wbuf, unsigned char* rbuf,
                              Meta* meta, uint64_t* bars)
{
    constexpr int JW = (W + 31) / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t fullW = smem_u32(bars + kFullW), emptyW = smem_u32(bars + kEmptyW);
    int armedW = -1, armedR[2] = {-1, -1};  // item sequence numbers whose phases were armed
    uint32_t missW = 0, missR = 0;          // this lane's counted-but-unissued bytes
    bool ok = true;
    int k = 0;
    for (;; ++k) {
        const int p = k & 1;
        const uint32_t fullR = smem_u32(bars + kFullR + p), emptyR = smem_u32(bars + kEmptyR + p);
        Meta& m = meta[p];
        unsigned char* rb_buf = rbuf + (size_t)p * W * kChunk;
        unsigned long long item = 0;
        int aborted = 0;
        if (lane == 0) {
            item = atomicAdd(a.counter, 1ull);
            aborted = ld_relaxed_gpu(a.abort_flag);
        }
        item = __shfl_sync(0xFFFFFFFFu, item, 0);
        aborted = __shfl_sync(0xFFFFFFFFu, aborted, 0);
        if (item >= (unsigned long long)a.items || aborted != 0) {
            // end of work: hand the consumers an empty item
            ok = mbar_wait(emptyW, (k & 1) ^ 1, a.abort_flag, a.status) &&
                 mbar_wait(emptyR, ((k >> 1) & 1) ^ 1, a.abort_flag, a.status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (ok && lane == 0) {
                m.valid = 0;
                mbar_arrive(fullW);
                mbar_arrive(fullR);
            }
            break;
        }
        const long long S_ = (long long)a.B * a.nrb;
        const int t = (int)(item / S_);
        const int rem = (int)(item % S_);
        const int b = rem / a.nrb, rb = rem % a.nrb;
        const long long tok = (long long)b * a.T + t;
        const int rows = min(a.rb_rows, a.d - rb * a.rb_rows);
        const uint32_t cb = (uint32_t)rows * (uint32_t)sizeof(S);
        const int* fl = a.flags + ((long long)b * a.nrb + rb) * a.T;
        const unsigned char* bank =
            a.banks + ((size_t)b * a.N * a.d + (size_t)rb * a.rb_rows) * sizeof(S);
        const size_t slot_bytes = (size_t)a.d * sizeof(S);

        // slot ids and collision codes of this token
        int wid[JW], rid[JW];
        uint16_t wc[JW], rc[JW];
        bool has[JW];
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) {
            const int j = lane + 32 * jj;
            has[jj] = j < W;
            if (has[jj]) {
                wid[jj] = __ldg(a.idx + tok * 2 * W + j);
                rid[jj] = __ldg(a.idx + tok * 2 * W + W + j);
                wc[jj] = __ldg(a.codes + tok * 2 * W + j);
                rc[jj] = __ldg(a.codes + tok * 2 * W + W + j);
            } else {
                wid[jj] = rid[jj] = -1;
                wc[jj] = rc[jj] = kNoFwd;
            }
        }
        // window: tokens t-2*win+1 .. t-win of this stream committed
        {
            int got[kFwdWindow / 32];
#pragma unroll
            for (int q = 0; q < kFwdWindow / 32; ++q) {
                const int tt = t - kFwdWindow - lane - 32 * q;
                got[q] = (tt >= 0 && tt > t - 2 * kFwdWindow) ? ld_relaxed_gpu(fl + tt) : 2;
            }
#pragma unroll
            for (int q = 0; q < kFwdWindow / 32; ++q) {
                const int tt = t - kFwdWindow - lane - 32 * q;
                if (got[q] < 2 && !spin_geq_gpu(fl + tt, 2, a.abort_flag, a.status))
                    ok = false;
            }
            fence_acq_rel_gpu();
            fence_proxy_async_global();
        }
        if (__any_sync(0xFFFFFFFFu, !ok))
            break;

        // ---- write chunks
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(emptyW, (k & 1) ^ 1, a.abort_flag, a.status))) {
            ok = false;
            break;
        }
        bool wval[JW], wdep[JW];
        int nW = 0;
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) {
            wval[jj] = has[jj] && wid[jj] >= 0 && wid[jj] < a.N;
            if (has[jj] && !wval[jj])
                report(a.status, SDM_ERANGE);
            wdep[jj] = wval[jj] && wc[jj] != kNoFwd;  // an earlier writer within the window
            nW += wval[jj] ? 1 : 0;
        }
        missW = (uint32_t)nW * cb;
        const int totW = warp_sum(nW);
        if (lane == 0)
            mbar_arrive_expect_tx(fullW, (uint32_t)totW * cb);
        armedW = k;
        __syncwarp();
#pragma unroll
        for (int jj = 0; jj < JW; ++jj)
            if (wval[jj] && !wdep[jj]) {
                bulk_g2s(smem_u32(wbuf + (size_t)(lane + 32 * jj) * kChunk),
                         bank + (size_t)wid[jj] * slot_bytes, cb, fullW);
                missW -= cb;
            }

        // ---- read chunks, weights and v
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(emptyR, ((k >> 1) & 1) ^ 1, a.abort_flag, a.status))) {
            ok = false;
            break;
        }
        bool rval[JW], rdep[JW], rown[JW];
        int nR = 0;
        unsigned long long fmask = 0;
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) {
            const int j = lane + 32 * jj;
            rval[jj] = has[jj] && rid[jj] >= 0 && rid[jj] < a.N;
            if (has[jj] && !rval[jj])
                report(a.status, SDM_ERANGE);
            const int dt = rc[jj] >> 8;
            rown[jj] = rval[jj] && rc[jj] != kNoFwd && dt == 0;
            rdep[jj] = rval[jj] && rc[jj] != kNoFwd && dt > 0;
            nR += (rval[jj] && !rown[jj]) ? 1 : 0;
            if (has[jj]) {
                m.wid[j] = wval[jj] ? wid[jj] : -1;
                m.fpos[j] = rown[jj] ? (signed char)(rc[jj] & 0xFF) : (signed char)-1;
            }
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, rown[jj]);
            fmask |= (unsigned long long)bal << (32 * jj);
        }
        missR = (uint32_t)nR * cb;
        const int totR = warp_sum(nR);
        if (lane == 0) {
            m.fmask = fmask;
            m.tok = tok;
            m.b = b;
            m.t = t;
            m.rb = rb;
            m.rows = rows;
            m.alpha = __ldg(a.alpha + tok);
            m.beta = __ldg(a.beta + tok);
            m.valid = 1;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive_expect_tx(fullR, (uint32_t)totR * cb + 2 * W * 4 + cb);
        armedR[p] = k;
        __syncwarp();
        if (lane == 0)
            bulk_g2s(smem_u32(m.wsel), a.wsel + tok * 2 * W, 2 * W * 4, fullR);
        if (lane == 1)
            bulk_g2s(smem_u32(m.v), a.v + ((size_t)tok * a.d + (size_t)rb * a.rb_rows) * sizeof(S),
                     cb, fullR);
#pragma unroll
        for (int jj = 0; jj < JW; ++jj)
            if (rval[jj] && !rown[jj] && !rdep[jj]) {
                bulk_g2s(smem_u32(rb_buf + (size_t)(lane + 32 * jj) * kChunk),
                         bank + (size_t)rid[jj] * slot_bytes, cb, fullR);
                missR -= cb;
            }

        // ---- chunks whose latest writer is still in the window: wait for its commit
#pragma unroll
        for (int jj = 0; jj < JW; ++jj)
            if (ok && wdep[jj]) {
                const int tw = t - (wc[jj] >> 8);
                if (spin_geq_gpu(fl + tw, 2, a.abort_flag, a.status)) {
                    fence_acq_rel_gpu();
                    fence_proxy_async_global();
                    bulk_g2s(smem_u32(wbuf + (size_t)(lane + 32 * jj) * kChunk),
                             bank + (size_t)wid[jj] * slot_bytes, cb, fullW);
                    missW -= cb;
                } else {
                    ok = false;
                }
            }
#pragma unroll
        for (int jj = 0; jj < JW; ++jj)
            if (ok && rdep[jj]) {
                const int tw = t - (rc[jj] >> 8);
                if (spin_geq_gpu(fl + tw, 2, a.abort_flag, a.status)) {
                    fence_acq_rel_gpu();
                    fence_proxy_async_global();
                    bulk_g2s(smem_u32(rb_buf + (size_t)(lane + 32 * jj) * kChunk),
                             bank + (size_t)rid[jj] * slot_bytes, cb, fullR);
                    missR -= cb;
                } else {
                    ok = false;
                }
            }
        if (__any_sync(0xFFFFFFFFu, !ok))
            break;

        // ---- write after read: tokens t-win .. t-1 of this stream have loaded
        {
            int got[kFwdWindow / 32];
#pragma unroll
            for (int q = 0; q < kFwdWindow / 32; ++q) {
                const int tt = t - 1 - lane - 32 * q;
                got[q] = tt >= 0 ? ld_relaxed_gpu(fl + tt) : 1;
            }
#pragma unroll
            for (int q = 0; q < kFwdWindow / 32; ++q) {
                const int tt = t - 1 - lane - 32 * q;
                if (got[q] < 1 && !spin_geq_gpu(fl + tt, 1, a.abort_flag, a.status))
                    ok = false;
            }
            fence_acq_rel_gpu();
        }
        if (__any_sync(0xFFFFFFFFu, !ok))
            break;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(bars + kWar + p));
        missW = missR = 0;
    }
    if (__all_sync(0xFFFFFFFFu, ok))
        return;
    // Failure (time-out or abort): declare the bytes that were counted but never
    // copied, then wait, boundedly, for the copies that are in flight into this CTA's
    // shared memory before the CTA may end.
    if (ld_relaxed_gpu(a.abort_flag) == 0)
        st_relaxed_gpu(a.abort_flag, 1);
    const int mw = warp_sum((int)missW), mr = warp_sum((int)missR);
    const int p = k & 1;
    if (lane == 0) {
        if (armedW == k && mw > 0)
            mbar_complete_tx(fullW, (uint32_t)mw);
        if (armedR[p] == k && mr > 0)
            mbar_complete_tx(smem_u32(bars + kFullR + p), (uint32_t)mr);
        if (armedW >= 0)
            mbar_wait(fullW, armedW & 1, nullptr, a.status);
        for (int q = 0; q < 2; ++q)
            if (armedR[q] >= 0)
                mbar_wait(smem_u32(bars + kFullR + q), (armedR[q] >> 1) & 1, nullptr, a.status);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- consumer warps

template <typename S, int W>
__device__ void scan_consumer(const ScanArgs& a, const unsigned char* wbuf, unsigned char* rbuf,
                              const Meta* meta, uint64_t* bars)
{
    constexpr int SPL = W / 4;         // slots of each set per thread
    using P = Pack16<S>;
    constexpr int RPL = P::R;          // rows per thread (16 bytes)
    const int ct = threadIdx.x, w = ct >> 5, lane = ct & 31;
    const int sg = lane >> 3;          // slot group: slots sg*SPL .. sg*SPL + SPL - 1
    const int rg = w * 8 + (lane & 7); // row group: rows rg*RPL .. rg*RPL + RPL - 1
    const uint32_t fullW = smem_u32(bars + kFullW), emptyW = smem_u32(bars + kEmptyW);
    const uint32_t cbar = smem_u32(bars + kCbar);
    // Barrier of the consumer warps (one arrival per warp). Every exit below is taken
    // by whole warps (the wait outcomes are made warp-uniform), and a warp that is
    // left waiting here gives up after the bounded wait, so no warp can hang.
    int cuses = 0;
    auto consumer_barrier = [&]() -> bool {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(cbar);
        const bool okb = mbar_wait(cbar, cuses & 1, a.abort_flag, a.status);
        ++cuses;
        return __all_sync(0xFFFFFFFFu, okb);
    };
    for (int k = 0;; ++k) {
        const int p = k & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(fullW, k & 1, a.abort_flag, a.status)))
            return;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(bars + kFullR + p), (k >> 1) & 1,
                                               a.abort_flag, a.status)))
            return;
        const Meta& m = meta[p];
        if (!m.valid)
            return;
        const unsigned char* rb_buf = rbuf + (size_t)p * W * kChunk;
        const bool act = rg * 16 < m.rows * (int)sizeof(S);
        uint4 Mv[SPL];
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            Mv[i] = act ? *reinterpret_cast<const uint4*>(wbuf + (size_t)(sg * SPL + i) * kChunk +
                                                          rg * 16)
                        : make_uint4(0, 0, 0, 0);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(emptyW);
        int* flag = a.flags + ((long long)m.b * a.nrb + m.rb) * a.T + m.t;
        if (ct == 0)
            st_release_gpu(flag, 1);  // this token's chunks are loaded

        // u = M_S k (pre-write), reduced over the four slot groups
        float u[RPL];
#pragma unroll
        for (int r = 0; r < RPL; ++r)
            u[r] = 0.f;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const float kw = m.wsel[sg * SPL + i];
            float f[RPL];
            P::unpack(Mv[i], f);
#pragma unroll
            for (int r = 0; r < RPL; ++r)
                u[r] = fmaf(kw, f[r], u[r]);
        }
#pragma unroll
        for (int r = 0; r < RPL; ++r) {
            u[r] += __shfl_xor_sync(0xFFFFFFFFu, u[r], 8);
            u[r] += __shfl_xor_sync(0xFFFFFFFFu, u[r], 16);
        }
        float vv[RPL];
        P::unpack(act ? *reinterpret_cast<const uint4*>(m.v + rg * 16) : make_uint4(0, 0, 0, 0), vv);
        const float al = m.alpha, be = m.beta;
        float c[RPL];
#pragma unroll
        for (int r = 0; r < RPL; ++r)
            c[r] = be * (vv[r] - al * u[r]);

        // M[S_j] <- alpha M[S_j] + k_j beta (v - alpha u), rounded once, stored
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(smem_u32(bars + kWar + p), (k >> 1) & 1, a.abort_flag, a.status)))
            return;
        S* bank = reinterpret_cast<S*>(a.banks) + (size_t)m.b * a.N * a.d +
                  (size_t)m.rb * a.rb_rows + rg * RPL;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const float kw = m.wsel[sg * SPL + i];
            float f[RPL];
            P::unpack(Mv[i], f);
#pragma unroll
            for (int r = 0; r < RPL; ++r)
                f[r] = fmaf(kw, c[r], al * f[r]);
            Mv[i] = P::pack(f);
            const int id = m.wid[sg * SPL + i];
            if (act && id >= 0)
                __stcg(reinterpret_cast<uint4*>(bank + (size_t)id * a.d), Mv[i]);
        }
        // read slots this token writes itself: their new values, from registers
        const unsigned long long fm0 = m.fmask;
        if (fm0 != 0) {
            unsigned long long fm = fm0;
            while (fm != 0) {
                const int j = __ffsll((long long)fm) - 1;
                fm &= fm - 1;
                const int q = m.fpos[j];
#pragma unroll
                for (int i = 0; i < SPL; ++i)
                    if (act && q == sg * SPL + i)
                        *reinterpret_cast<uint4*>(rbuf + (size_t)p * W * kChunk +
                                                  (size_t)j * kChunk + rg * 16) = Mv[i];
            }
            if (!consumer_barrier())
                return;
        }

        // y = sum_j r_j M[R_j] (post-write)
        float yv[RPL];
#pragma unroll
        for (int r = 0; r < RPL; ++r)
            yv[r] = 0.f;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const float rw = m.wsel[W + sg * SPL + i];
            float f[RPL];
            P::unpack(act ? *reinterpret_cast<const uint4*>(rb_buf + (size_t)(sg * SPL + i) * kChunk +
                                                            rg * 16)
                          : make_uint4(0, 0, 0, 0),
                      f);
#pragma unroll
            for (int r = 0; r < RPL; ++r)
                yv[r] = fmaf(rw, f[r], yv[r]);
        }
#pragma unroll
        for (int r = 0; r < RPL; ++r) {
            yv[r] += __shfl_xor_sync(0xFFFFFFFFu, yv[r], 8);
            yv[r] += __shfl_xor_sync(0xFFFFFFFFu, yv[r], 16);
        }
        if (sg == 0 && act) {
            float* yp = a.y + (size_t)m.tok * a.d + (size_t)m.rb * a.rb_rows + rg * RPL;
#pragma unroll
            for (int r = 0; r < RPL; r += 4)
                __stcs(reinterpret_cast<float4*>(yp + r),
                       make_float4(yv[r], yv[r + 1], yv[r + 2], yv[r + 3]));
        }

        // commit: every consumer's stores visible, then the flag
        __threadfence();
        if (!consumer_barrier())
            return;
        if (ct == 0)
            st_release_gpu(flag, 2);
        if (fm0 != 0)
            fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(bars + kEmptyR + p));
    }
}

template <typename S, int W>
__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(ScanArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* wbuf = smem;
    unsigned char* rbuf = smem + (size_t)W * kChunk;
    Meta* meta = reinterpret_cast<Meta*>(smem + (size_t)3 * W * kChunk);
    uint64_t* bars = reinterpret_cast<uint64_t*>(meta + 2);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bars + kFullW), 1);
        mbar_init(smem_u32(bars + kEmptyW), kCWarps);
        for (int p = 0; p < 2; ++p) {
            mbar_init(smem_u32(bars + kFullR + p), 1);
            mbar_init(smem_u32(bars + kEmptyR + p), kCWarps);
            mbar_init(smem_u32(bars + kWar + p), 1);
        }
        mbar_init(smem_u32(bars + kCbar), kCWarps);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x >= 32 * kCWarps)
        scan_producer<S, W>(a, wbuf, rbuf, meta, bars);
    else
        scan_consumer<S, W>(a, wbuf, rbuf, meta, bars);
}

template <typename S, int W>
cudaError_t launch_scan_t(const ScanArgs& a, cudaStream_t s)
{
    const size_t smem = (size_t)3 * W * kChunk + 2 * sizeof(Meta) + kNumBars * sizeof(uint64_t);
    auto kern = scan_kernel<S, W>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    long long grid = num_sms_current_device();
    if (grid > a.items)
        grid = a.items;
    kern<<<(unsigned)grid, kScanThreads, smem, s>>>(a);
    return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int scan_block_rows(const sdm_cfg& c)
{
    const int es = c.dtype == SDM_BF16 ? 2 : 4;
    return kChunk / es;
}

int scan_row_blocks(const sdm_cfg& c)
{
    const int r = scan_block_rows(c);
    return (c.d + r - 1) / r;
}

size_t scan_flags_bytes(const sdm_cfg& c, int B, int T)
{
    return align256((size_t)B * scan_row_blocks(c) * T * sizeof(int)) + 256;
}

cudaError_t launch_scan(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                        const uint16_t* codes, const void* v, const float* alpha,
                        const float* beta, void* banks, float* y, int B, int T, void* flags,
                        int* status, cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    const size_t fb = scan_flags_bytes(c, B, T);
    cudaError_t e = cudaMemsetAsync(flags, 0, fb, s);
    if (e != cudaSuccess)
        return e;
    ScanArgs a;
    a.banks = (unsigned char*)banks;
    a.idx = idx;
    a.wsel = wsel;
    a.codes = codes;
    a.v = (const unsigned char*)v;
    a.alpha = alpha;
    a.beta = beta;
    a.y = y;
    a.status = status;
    a.flags = (int*)flags;
    a.counter = (unsigned long long*)((char*)flags + fb - 256);
    a.abort_flag = (int*)((char*)flags + fb - 128);
    a.B = B;
    a.T = T;
    a.d = c.d;
    a.N = c.n_sub * c.n_sub;
    a.nrb = scan_row_blocks(c);
    a.rb_rows = scan_block_rows(c);
    a.items = (long long)B * T * a.nrb;
    const bool bf = c.dtype == SDM_BF16;
    switch (c.w) {
    case 8: return bf ? launch_scan_t<bf16, 8>(a, s) : launch_scan_t<float, 8>(a, s);
    case 16: return bf ? launch_scan_t<bf16, 16>(a, s) : launch_scan_t<float, 16>(a, s);
    case 32: return bf ? launch_scan_t<bf16, 32>(a, s) : launch_scan_t<float, 32>(a, s);
    case 64: return bf ? launch_scan_t<bf16, 64>(a, s) : launch_scan_t<float, 64>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
