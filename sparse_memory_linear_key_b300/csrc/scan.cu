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
// of a sequence are independent streams of tokens. An item gathers W write chunks and
// W read chunks of 1 KB and scatters W chunks back: random 1 KB chunks are served by
// HBM near its copy bandwidth, unlike the 32-byte pieces a finer split would give.
//
// Persistent kernel, one CTA per SM, items claimed in increasing order from a global
// counter (t-major, so all streams advance together). Warp roles in a CTA:
//  P   claims the next item, reads its slot ids and codes, checks its window and writes
//      its description (which chunks come from the bank);
//  C   16 warps: take the write chunks into registers, which frees the write buffer,
//      then gather the next item's chunks from the bank with cp.async.bulk into it and
//      into one of two read buffers (alternating items), each warp issuing 1/16 of the
//      copies (one warp alone issues them too slowly); then form u and the new values,
//      publish the slots later tokens need into the ring, reduce the read chunks into
//      y, and store the new values to the bank;
//  D   copies the chunks whose latest writer is still in flight, from that writer's
//      forwarding-ring entry, once the writer has published it;
//  F1  clears the item's bank stores (write after read);
//  M   marks the item's progress: bank loads done, ring entries and bank stores
//      published.
// Ordering between tokens of one stream, which may run on different SMs, goes through
// one progress flag per item in global memory: 1 = its bank loads are done, 2 = its
// ring entries are visible, 3 = its bank stores are visible (raised with atomic max, so
// it never goes down whichever mark lands first).
//  * read after write: a reference whose latest writer lies within the last `win`
//    tokens (collision codes) is copied from that writer's ring entry once its flag is
//    >= 2; a read of a slot the same token writes is forwarded in shared memory; older
//    writers are visible in the bank (window rule below);
//  * write after read: the bank stores of token t wait until each token within the
//    window that references a slot t writes has flag >= 1 (the codes mark them; bank
//    loads happen first, so this never waits on a dependency);
//  * write after write: a write that a later token within the window overwrites is
//    not stored at all (dead store: readers in between take the ring entry, readers
//    after it the newer value), so two stores of one slot are always a window apart;
//  * window: token t starts only when tokens t-2*win+1 .. t-win have flag 3; the ring
//    has 2*win entries per stream, so an entry is reused only when all its readers are
//    done.
// Without ring space (a workspace of only min_total bytes) dependent references wait
// for flag 3 and read the bank.
// Every wait is bounded: on time-out the kernel records SDM_ETIMEOUT and raises a
// global abort flag that every warp watches. Each warp leaves as a whole, and no warp
// waits on another without a bound, so none can hang.
#include <cstddef>

#include "scan_math.cuh"
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kChunk = 1024;       // bytes of a full row block of one slot
constexpr int kStride = 1088;      // shared-memory stride between chunks (bank spread)
constexpr int kCWarps = 16;        // consumer warps
constexpr int kWarpP = kCWarps, kWarpD = kCWarps + 1, kWarpF1 = kCWarps + 2;
// 20 warps: five per SM sub-partition, which leaves each thread up to 96 registers
constexpr int kScanThreads = 32 * (kCWarps + 4);
constexpr int kLaunchRegs = 96;    // registers a thread at launch (__launch_bounds__)
constexpr int kConsumerRegs = 104, kRoleRegs = 64;
static_assert(kCWarps * 32 * kConsumerRegs + 4 * 32 * kRoleRegs <= kScanThreads * kLaunchRegs,
              "register split exceeds the block's launch allocation");
static_assert(kCWarps % 4 == 0, "consumer warps must form whole warpgroups");
constexpr int kMaxW = 64;

// With bf16 state and W >= 16 the read y = sum_j r_j M[R_j] runs on the tensor cores
// (mma.sync m16n8k16 per 16 rows, the read chunks as A through ldmatrix.trans). The eight
// slots that one ldmatrix phase reads at one row offset must then fall in different banks:
// read chunks are 1040 bytes apart (260 words, 4 mod 32). Write chunks keep 1088 (16 mod
// 32), right for the lanes of the consumers' SIMT pattern.
template <typename S, int W>
struct ScanShape {
    static constexpr bool kMmaY = sizeof(S) == 2 && W >= 16;
    static constexpr int kRStride = kMmaY ? 1040 : kStride;
};

struct ScanArgs {
    unsigned char* banks;
    const int32_t* idx;
    const float* wsel;
    const uint16_t* codes;
    const unsigned long long* masks;  // per token: fwdmask [B*T], deadmask [B*T], warmask [B*T][2]
    const unsigned char* v;
    const float* alpha;
    const float* beta;
    float* y;
    int* status;
    int* flags;                     // [B][nrb][T]
    unsigned long long* counter;    // next item to claim
    int* abort_flag;
    unsigned char* ring;            // null: no forwarding ring
    const unsigned char* m0;        // non-null: banks start as M0 without a copy; the
                                    // first write of a slot in a sequence, and every
                                    // read before it, loads the slot from M0
    const int* first_write;         // [B][N] first token writing each slot (>= T: none)
    unsigned char* tape;            // non-null: [B*T][W][d] pre-write values of the write
                                    // slots, for the backward pass
    long long items;                // B * T * nrb
    long long spin_limit;           // bound of every wait, SM clock cycles
    long long skip_item;            // diagnostics: an item never processed (-1: none)
    int B, T, d, N, nrb, rb_rows, win, ring_entries, chunk_bytes;
};

// How long a warp leaving an aborted kernel waits for the copies it started (cycles, about
// two milliseconds): far longer than any copy takes to land.
constexpr long long kDrainCycles = 4000000LL;

// Everything about one item besides the chunks.
struct __align__(16) Meta {
    float wsel[2 * kMaxW];          // write weights, then read weights (bulk copy target)
    unsigned char v[kChunk];        // v rows of this row block (bulk copy target)
    int wid[kMaxW];                 // write slot ids, -1 if out of range
    int rid[kMaxW];                 // read slot ids, -1 if out of range
    uint16_t code[2 * kMaxW];       // collision codes, write refs then read refs
    signed char fpos[kMaxW];        // read ref j: position in the write set if own write
    unsigned long long fmask;       // bit j: read ref j is such a slot
    unsigned long long fwdmask;     // bit j: write slot j goes to the ring
    unsigned long long deadmask;    // bit j: write slot j is rewritten within the window
    unsigned long long war[2];      // bit dt-1: token t-dt must have loaded before our stores
    unsigned long long wload;       // bit j: write chunk j is gathered from the bank
    unsigned long long rload;       // bit j: read chunk j is gathered from the bank
    unsigned long long rdmask;      // bit j: read chunk j is copied by D (writer in flight)
    unsigned long long m0w, m0r;    // bit j: write / read chunk j is gathered from M0
    long long tok;                  // b * T + t
    int b, t, rb, rows;
    float alpha, beta;
    int valid;                      // 0: no more work
    // y on the tensor cores: bit j set when read slot j is in range (its weight counts),
    // and for each write position the read position of the same slot (-1: not read by
    // this token)
    unsigned long long rvalid;
    signed char rpos[kMaxW];
};
static_assert(offsetof(Meta, wsel) % 16 == 0 && offsetof(Meta, v) % 16 == 0,
              "bulk copy targets must be 16-byte aligned");

// mbarriers: full* = an item's chunks landed (armed by the consumer warps issuing them),
// Wfree = the consumers took the write chunks, EmptyR = item description and read
// buffer free again (F1 and M done), DepB / DepR = D's write / read chunk copies landed
// (read chunks are needed only after u and the new values), Posted = item described,
// War = bank stores cleared, Fwdw / Stored = consumers wrote the ring / the bank,
// Cbar = barrier of the consumer warps, Lmark = M marked the item loaded (the consumers
// arm the next item's FullW only then, so that FullW is never two phases ahead of M).
// The [2] ones alternate with the items.
enum {
    kFullW = 0, kWfree = 1, kFullR = 2, kEmptyR = 4, kDepB = 6, kPosted = 8, kWar = 10,
    kFwdw = 12, kStored = 14, kCbar = 16, kLmark = 17, kDepR = 18, kNumBars = 20
};

__device__ __forceinline__ bool uniform_wait(uint32_t bar, uint32_t parity, const ScanArgs& a)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, a.abort_flag, a.status, a.spin_limit));
}

// warp-uniform non-blocking test of an mbarrier phase
__device__ __forceinline__ bool uniform_test(uint32_t bar, uint32_t parity)
{
    int r = 0;
    if ((threadIdx.x & 31) == 0)
        r = mbar_test(bar, parity) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, r, 0) != 0;
}

__device__ __forceinline__ int* item_flag(const ScanArgs& a, int b, int rb, int t)
{
    return a.flags + ((long long)b * a.nrb + rb) * a.T + t;
}

__device__ __forceinline__ unsigned char* ring_entry(const ScanArgs& a, int b, int rb, int t, int pos)
{
    const long long e = ((long long)b * a.nrb + rb) * a.ring_entries + t % a.ring_entries;
    return a.ring + ((size_t)e * kMaxW + pos) * a.chunk_bytes;
}

// Wait (bounded) until every flag of tokens [lo, hi) of one stream is >= target, reading
// them all first; the caller follows with fence_acq_rel_gpu().
__device__ __forceinline__ bool window_geq(const ScanArgs& a, const int* fl, int lo, int hi,
                                           int target)
{
    const int lane = threadIdx.x & 31;
    lo = max(lo, 0);
    int got[kMaxWindow / 32];
#pragma unroll
    for (int q = 0; q < kMaxWindow / 32; ++q) {
        const int tt = lo + lane + 32 * q;
        got[q] = tt < hi ? ld_relaxed_gpu(fl + tt) : target;
    }
    bool ok = true;
#pragma unroll
    for (int q = 0; q < kMaxWindow / 32; ++q) {
        const int tt = lo + lane + 32 * q;
        if (ok && got[q] < target &&
            !spin_geq_gpu(fl + tt, target, a.abort_flag, a.status, a.spin_limit))
            ok = false;
    }
    return __all_sync(0xFFFFFFFFu, ok);
}

// ------------------------------------------------------------- P: item descriptions

// A claimed item and what the producer needs of it, read one item ahead.
template <int JW>
struct Ahead {
    unsigned long long item;
    int t, b, rb;
    int wid[JW], rid[JW];
    int ftw[JW], ftr[JW];            // first writer of the slot in the sequence (M0 mode)
    uint16_t wc[JW], rc[JW];
    float alpha, beta;               // lane 0
    unsigned long long fwdmask, deadmask, war0, war1;  // lane 0
};

template <int W, int JW>
__device__ __forceinline__ void fetch_ahead(const ScanArgs& a, unsigned long long item, Ahead<JW>& n)
{
    const int lane = threadIdx.x & 31;
    n.item = item;
    if (item >= (unsigned long long)a.items)
        return;
    const long long S_ = (long long)a.B * a.nrb;
    n.t = (int)(item / S_);
    const int rem = (int)(item % S_);
    n.b = rem / a.nrb;
    n.rb = rem % a.nrb;
    const long long tok = (long long)n.b * a.T + n.t;
#pragma unroll
    for (int jj = 0; jj < JW; ++jj) {
        const int j = lane + 32 * jj;
        if (j < W) {
            n.wid[jj] = __ldg(a.idx + tok * 2 * W + j);
            n.rid[jj] = __ldg(a.idx + tok * 2 * W + W + j);
            n.wc[jj] = a.T > 1 ? __ldg(a.codes + tok * 2 * W + j) : kNoFwd;
            n.rc[jj] = a.T > 1 ? __ldg(a.codes + tok * 2 * W + W + j) : kNoFwd;
        } else {
            n.wid[jj] = n.rid[jj] = -1;
            n.wc[jj] = n.rc[jj] = kNoFwd;
        }
    }
    if (a.T == 1) {
        // one token a sequence (a decode step): no earlier writer exists, and a read's only
        // possible writer is its own token -- matched here instead of by the codes kernel:
        // the write set is in ascending order, so each read id is looked up by a binary
        // search over it (element i of the set is in lane i % 32, register i / 32)
        auto wid_at = [&](int i) -> int {
            int v = __shfl_sync(0xFFFFFFFFu, n.wid[0], i & 31);
#pragma unroll
            for (int jj = 1; jj < JW; ++jj) {
                const int u = __shfl_sync(0xFFFFFFFFu, n.wid[jj], i & 31);
                if ((i >> 5) == jj)
                    v = u;
            }
            return v;
        };
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) {
            const int r = n.rid[jj];
            int at = -1;                       // the last position holding an id below r
#pragma unroll
            for (int step = W / 2; step > 0; step >>= 1) {
                const int cand = at + step;
                if (wid_at(cand) < r)
                    at = cand;
            }
            const int pos = at + 1;
            const int found = wid_at(pos < W ? pos : W - 1);
            if (pos < W && found == r && r >= 0 && r < a.N)
                n.rc[jj] = (uint16_t)pos;       // dt = 0, position pos
        }
    }
    // M0 mode: the first writer of each referenced slot in this sequence
#pragma unroll
    for (int jj = 0; jj < JW; ++jj) {
        n.ftw[jj] = n.ftr[jj] = 0;
        if (a.m0 != nullptr) {
            const int* fw = a.first_write + (size_t)n.b * a.N;
            if (n.wid[jj] >= 0 && n.wid[jj] < a.N)
                n.ftw[jj] = __ldg(fw + n.wid[jj]);
            if (n.rid[jj] >= 0 && n.rid[jj] < a.N)
                n.ftr[jj] = __ldg(fw + n.rid[jj]);
        }
    }
    if (lane == 0) {
        n.alpha = __ldg(a.alpha + tok);
        n.beta = __ldg(a.beta + tok);
        const size_t BT = (size_t)a.B * a.T;
        // without the ring, nothing is handed over and every store is needed; with one
        // token a sequence nothing else references this token's slots
        const bool many = a.T > 1;
        n.fwdmask = many && a.ring != nullptr ? __ldg(a.masks + tok) : 0ull;
        n.deadmask = many && a.ring != nullptr ? __ldg(a.masks + BT + tok) : 0ull;
        n.war0 = many ? __ldg(a.masks + 2 * BT + 2 * tok) : 0ull;
        n.war1 = many ? __ldg(a.masks + 2 * BT + 2 * tok + 1) : 0ull;
    }
}

template <typename S, int W>
__device__ void role_producer(const ScanArgs& a, Meta* meta, uint64_t* bars)
{
    constexpr int JW = (W + 31) / 32;
    constexpr bool kMmaY = ScanShape<S, W>::kMmaY;
    const int lane = threadIdx.x & 31;
    // the next item in claim order (a withheld item, for diagnostics, is claimed and
    // dropped: the tokens that depend on it then wait for it until their bound runs out)
    // With one token a sequence the items are independent: block b takes items b, b +
    // grid, ... without a shared counter.
    unsigned long long next_static = blockIdx.x;
    auto claim = [&]() -> unsigned long long {
        unsigned long long item = 0;
        if (a.T == 1 && a.skip_item < 0) {
            item = next_static;
            next_static += gridDim.x;
            return item;
        }
        if (lane == 0) {
            item = atomicAdd(a.counter, 1ull);
            if (item == (unsigned long long)a.skip_item)
                item = atomicAdd(a.counter, 1ull);
        }
        return __shfl_sync(0xFFFFFFFFu, item, 0);
    };
    Ahead<JW> nx;
    fetch_ahead<W, JW>(a, claim(), nx);
    // the abort flag, read one item ahead so that its load overlaps the fetch (the flags
    // are clear at launch)
    int ab = 0;
    for (int k = 0;; ++k) {
        const int p = k & 1;
        Meta& m = meta[p];
        const int aborted = __shfl_sync(0xFFFFFFFFu, ab, 0);
        // the description slot (and read buffer) is free once item k-2 is done
        if (!uniform_wait(smem_u32(bars + kEmptyR + p), ((k >> 1) & 1) ^ 1, a))
            return;
        if (nx.item >= (unsigned long long)a.items || aborted != 0) {
            // end of work: an empty item tells every role to finish
            if (lane == 0) {
                m.valid = 0;
                mbar_arrive(smem_u32(bars + kPosted + p));
            }
            return;
        }
        const int t = nx.t, b = nx.b, rb = nx.rb;
        const int* fl = item_flag(a, b, rb, 0);
        // window: tokens t-2*win+1 .. t-win of this stream are committed (acquired, when
        // there are any)
        if (!window_geq(a, fl, t - 2 * a.win + 1, t - a.win + 1, 3))
            return;
        if (t - a.win + 1 > 0)
            fence_acq_rel_gpu();

        unsigned long long wload = 0, rload = 0, fmask = 0, rdmask = 0, m0w = 0, m0r = 0;
        unsigned long long rvalid = 0;
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) {
            const int j = lane + 32 * jj;
            const bool has = j < W;
            const bool wval = has && nx.wid[jj] >= 0 && nx.wid[jj] < a.N;
            const bool rval = has && nx.rid[jj] >= 0 && nx.rid[jj] < a.N;
            if ((has && !wval) || (has && !rval))
                report(a.status, SDM_ERANGE);
            const int dt = nx.rc[jj] >> 8;
            const bool rown = rval && nx.rc[jj] != kNoFwd && dt == 0;
            const bool rdep = rval && nx.rc[jj] != kNoFwd && dt > 0;
            // bank loads: references with no writer within the window (D copies the rest)
            wload |= (unsigned long long)__ballot_sync(0xFFFFFFFFu, wval && nx.wc[jj] == kNoFwd)
                     << (32 * jj);
            rload |= (unsigned long long)__ballot_sync(0xFFFFFFFFu, rval && !rown && !rdep)
                     << (32 * jj);
            fmask |= (unsigned long long)__ballot_sync(0xFFFFFFFFu, rown) << (32 * jj);
            rdmask |= (unsigned long long)__ballot_sync(0xFFFFFFFFu, rdep) << (32 * jj);
            // M0 mode: a bank load of a slot no earlier token of the sequence wrote reads
            // M0 (a write is the first when its token is the first writer)
            m0w |= (unsigned long long)__ballot_sync(
                       0xFFFFFFFFu, a.m0 != nullptr && wval && nx.wc[jj] == kNoFwd && nx.ftw[jj] >= t)
                   << (32 * jj);
            m0r |= (unsigned long long)__ballot_sync(
                       0xFFFFFFFFu, a.m0 != nullptr && rval && !rown && !rdep && nx.ftr[jj] > t)
                   << (32 * jj);
            rvalid |= (unsigned long long)__ballot_sync(0xFFFFFFFFu, rval) << (32 * jj);
            if (has) {
                m.wid[j] = wval ? nx.wid[jj] : -1;
                m.rid[j] = rval ? nx.rid[jj] : -1;
                m.code[j] = nx.wc[jj];
                m.code[W + j] = nx.rc[jj];
                m.fpos[j] = rown ? (signed char)(nx.rc[jj] & 0xFF) : (signed char)-1;
            }
        }
        if (lane == 0) {
            m.fmask = fmask;
            m.fwdmask = nx.fwdmask;
            m.deadmask = nx.deadmask;
            m.war[0] = nx.war0;
            m.war[1] = nx.war1;
            m.wload = wload;
            m.rload = rload;
            m.rdmask = rdmask;
            m.m0w = m0w;
            m.m0r = m0r;
            m.rvalid = rvalid;
            m.tok = (long long)b * a.T + t;
            m.b = b;
            m.t = t;
            m.rb = rb;
            m.rows = min(a.rb_rows, a.d - rb * a.rb_rows);
            m.alpha = nx.alpha;
            m.beta = nx.beta;
            m.valid = 1;
        }
        if (kMmaY) {
            // for each write position, the read position of the same slot
#pragma unroll
            for (int jj = 0; jj < JW; ++jj)
                if (lane + 32 * jj < kMaxW)
                    m.rpos[lane + 32 * jj] = -1;
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < JW; ++jj) {
                const int j = lane + 32 * jj;
                if (j < W && m.fpos[j] >= 0)
                    m.rpos[m.fpos[j]] = (signed char)j;
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(bars + kPosted + p));  // consumers and D may start on it

        // ---- the next item
        ab = lane == 0 ? ld_relaxed_gpu(a.abort_flag) : 0;
        fetch_ahead<W, JW>(a, claim(), nx);
    }
}

// ------------------------------------------------------- D: in-flight dependencies

template <typename S, int W>
__device__ void role_deps(const ScanArgs& a, unsigned char* wbuf, unsigned char* rbuf,
                          const Meta* meta, uint64_t* bars)
{
    constexpr int JR = (2 * W + 31) / 32;   // references per lane
    const int lane = threadIdx.x & 31;
    const int need = a.ring != nullptr ? 2 : 3;
    for (int k = 0;; ++k) {
        const int p = k & 1;
        if (!uniform_wait(smem_u32(bars + kPosted + p), (k >> 1) & 1, a)) {
            // aborted: the previous item's copies land before the CTA may end
            if (k > 0 && lane == 0) {
                mbar_drain(smem_u32(bars + kDepB + (p ^ 1)), ((k - 1) >> 1) & 1, kDrainCycles);
                mbar_drain(smem_u32(bars + kDepR + (p ^ 1)), ((k - 1) >> 1) & 1, kDrainCycles);
            }
            __syncwarp();
            return;
        }
        const Meta& m = meta[p];
        if (!m.valid)
            return;
        const uint32_t depB = smem_u32(bars + kDepB + p), depR = smem_u32(bars + kDepR + p);
        const uint32_t cb = (uint32_t)m.rows * (uint32_t)sizeof(S);
        const int t = m.t, b = m.b, rb = m.rb;
        const int* fl = item_flag(a, b, rb, 0);
        // references whose latest writer lies within the window: write chunks first
        // (q < JW), then read chunks
        bool dep[JR];
        int nw = 0, nr = 0;
#pragma unroll
        for (int q = 0; q < JR; ++q) {
            const int r = lane + 32 * q;
            dep[q] = false;
            if (r < 2 * W) {
                const uint16_t c = m.code[r];
                const int id = r < W ? m.wid[r] : m.rid[r - W];
                dep[q] = id >= 0 && c != kNoFwd && (c >> 8) > 0;
            }
            nw += (dep[q] && r < W) ? 1 : 0;
            nr += (dep[q] && r >= W) ? 1 : 0;
        }
        const int totw = __reduce_add_sync(0xFFFFFFFFu, nw);
        const int totr = __reduce_add_sync(0xFFFFFFFFu, nr);
        if (lane == 0) {
            mbar_arrive_expect_tx(depB, (uint32_t)totw * cb);
            mbar_arrive_expect_tx(depR, (uint32_t)totr * cb);
        }
        // write chunks go to the write buffer, free once item k-1 has taken its own
        bool ok = totw == 0 || k == 0 || uniform_wait(smem_u32(bars + kWfree), (k - 1) & 1, a);
        uint32_t missw = (uint32_t)nw * cb, missr = (uint32_t)nr * cb;
        // read the writers' flags together, then wait for the ones not yet published
        int got[JR];
#pragma unroll
        for (int q = 0; q < JR; ++q)
            got[q] = dep[q] ? ld_relaxed_gpu(fl + t - (m.code[lane + 32 * q] >> 8)) : need;
#pragma unroll
        for (int q = 0; q < JR; ++q) {
            if (!dep[q] || !ok)
                continue;
            const int r = lane + 32 * q;
            const uint16_t c = m.code[r];
            const int tw = t - (c >> 8);
            if (got[q] < need && !spin_geq_gpu(fl + tw, need, a.abort_flag, a.status, a.spin_limit)) {
                ok = false;
                continue;
            }
            fence_acq_rel_gpu();
            fence_proxy_async_global();
            const bool is_w = r < W;
            const int j = is_w ? r : r - W;
            const unsigned char* src;
            if (a.ring != nullptr) {
                src = ring_entry(a, b, rb, tw, c & 0xFF);
            } else {
                const int id = is_w ? m.wid[j] : m.rid[j];
                src = a.banks + (((size_t)b * a.N + id) * a.d + (size_t)rb * a.rb_rows) * sizeof(S);
            }
            constexpr int RS = ScanShape<S, W>::kRStride;
            unsigned char* dst = is_w ? wbuf + (size_t)j * kStride
                                      : rbuf + ((size_t)p * W + j) * RS;
            bulk_g2s(smem_u32(dst), src, cb, is_w ? depB : depR);
            (is_w ? missw : missr) -= cb;
        }
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            // declare what was not copied, wait (bounded) for what was, and leave
            if (lane == 0)
                st_relaxed_gpu(a.abort_flag, 1);
            const int mw = __reduce_add_sync(0xFFFFFFFFu, (int)missw);
            const int mr = __reduce_add_sync(0xFFFFFFFFu, (int)missr);
            if (lane == 0) {
                if (mw > 0)
                    mbar_complete_tx(depB, (uint32_t)mw);
                if (mr > 0)
                    mbar_complete_tx(depR, (uint32_t)mr);
                mbar_drain(depB, (k >> 1) & 1, kDrainCycles);
                mbar_drain(depR, (k >> 1) & 1, kDrainCycles);
                if (k > 0) {   // and the previous item's, if the consumers never took them
                    mbar_drain(smem_u32(bars + kDepB + (p ^ 1)), ((k - 1) >> 1) & 1, kDrainCycles);
                    mbar_drain(smem_u32(bars + kDepR + (p ^ 1)), ((k - 1) >> 1) & 1, kDrainCycles);
                }
            }
            __syncwarp();
            return;
        }
    }
}

// ------------------------------------------------------------------ F1: clearance

template <int W>
__device__ void role_clear(const ScanArgs& a, const Meta* meta, uint64_t* bars)
{
    const int lane = threadIdx.x & 31;
    for (int k = 0;; ++k) {
        const int p = k & 1;
        if (!uniform_wait(smem_u32(bars + kPosted + p), (k >> 1) & 1, a))
            return;
        const Meta& m = meta[p];
        if (!m.valid)
            return;
        const int t = m.t;
        const int* fl = item_flag(a, m.b, m.rb, 0);
        const unsigned long long war[2] = {m.war[0], m.war[1]};
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(bars + kEmptyR + p));  // done with the item description
        // write after read: the tokens that reference a slot this token writes have done
        // their bank loads (lane q watches dt = q+1, q+33, q+65, q+97). A token's
        // in-window earlier writer of a slot never stores it (dead store), so there is
        // no write-after-write wait.
        bool ok = true;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int dt = lane + 32 * q + 1;
            const bool need = (war[q >> 1] >> ((dt - 1) & 63)) & 1;
            if (ok && need && !spin_geq_gpu(fl + t - dt, 1, a.abort_flag, a.status, a.spin_limit))
                ok = false;
        }
        if (!__all_sync(0xFFFFFFFFu, ok))
            return;
        if ((war[0] | war[1]) != 0)   // (acquire what the flags published)
            fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(bars + kWar + p));
    }
}

// ------------------------------------------------------------ M: progress marks

// Raises each item's flag: to 1 as soon as its bank chunks have landed and to 3 once the
// consumers have stored its new slot values (the consumers' arrival, release at CTA
// scope, followed by this release at GPU scope publishes their global writes); the
// consumers raise it to 2 themselves once they have written its ring entries. The three marks advance independently: the
// warp polls whichever is next for each and never blocks one behind another (a later
// item's bank loads may wait on other tokens' commits, this item's among them). With one
// token a sequence no item waits on another's flag, and the marks are only the CTA's own
// barrier arrivals.
__device__ void role_marks(const ScanArgs& a, const Meta* meta, uint64_t* bars)
{
    const int lane = threadIdx.x & 31;
    int kl = 0, kp = 0, kc = 0;   // next item to mark loaded, ring-published, committed
    int end = -1;                 // item number of the empty end item, once seen
    long long idle = clock64();
    long long next_poll = idle + kAbortPollCycles;
    while (true) {
        bool progress = false;
        if (end < 0) {
            const int p = kl & 1;
            if (uniform_test(smem_u32(bars + kFullW), kl & 1) &&
                uniform_test(smem_u32(bars + kFullR + p), (kl >> 1) & 1)) {
                const Meta& m = meta[p];
                if (!m.valid) {
                    end = kl;
                    progress = true;
                } else if (a.ring != nullptr ||
                           (uniform_test(smem_u32(bars + kDepB + p), (kl >> 1) & 1) &&
                            uniform_test(smem_u32(bars + kDepR + p), (kl >> 1) & 1))) {
                    // (without the ring, dependent references are bank loads too)
                    if (lane == 0) {
                        if (a.T > 1)
                            red_max_release_gpu(item_flag(a, m.b, m.rb, m.t), 1);
                        mbar_arrive(smem_u32(bars + kLmark));
                    }
                    ++kl;
                    progress = true;
                }
            }
        }
        if (kp < kl && uniform_test(smem_u32(bars + kFwdw + (kp & 1)), (kp >> 1) & 1)) {
            ++kp;                  // (the consumers published the ring entries: flag 2)
            progress = true;
        }
        if (kc < kp && uniform_test(smem_u32(bars + kStored + (kc & 1)), (kc >> 1) & 1)) {
            const Meta& m = meta[kc & 1];
            int* flag = item_flag(a, m.b, m.rb, m.t);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(bars + kEmptyR + (kc & 1)));
                if (a.T > 1)
                    red_max_release_gpu(flag, 3);  // bank stores visible
            }
            ++kc;
            progress = true;
        }
        if (end >= 0 && kc == end)
            return;
        if (progress) {
            idle = clock64();
            continue;
        }
        __nanosleep(20);
        const long long now = clock64();
        if (now < next_poll)
            continue;
        next_poll = now + kAbortPollCycles;
        int stop = 0;
        if (lane == 0) {
            if (ld_relaxed_gpu(a.abort_flag) != 0) {
                stop = 1;
            } else if (now - idle > a.spin_limit) {
                report(a.status, SDM_ETIMEOUT);
                st_relaxed_gpu(a.abort_flag, 1);
                stop = 1;
            }
        }
        if (__shfl_sync(0xFFFFFFFFu, stop, 0))
            return;
    }
}

// ---------------------------------------------------------------- C: consumers

template <typename S, int W>
__device__ void role_consumer(const ScanArgs& a, unsigned char* wbuf, unsigned char* rbuf,
                              const Meta* meta, uint64_t* bars, float* ybuf, uint32_t* bfr,
                              int* fwdcnt)
{
    constexpr int SPL = W / kSG;       // slots of each set per thread: i*8 + sg
    constexpr bool kMmaY = ScanShape<S, W>::kMmaY;
    constexpr int RS = ScanShape<S, W>::kRStride;
    using P = Pack16<S>;
    constexpr int RPL = P::R;          // rows per thread (16 bytes)
    constexpr int HPL = P::H;          // fp32 pairs per thread
    const int ct = threadIdx.x, w = ct >> 5, lane = ct & 31;
    const int sg = lane >> 2;          // slot group
    const int rg = w * 4 + (lane & 3); // row group: rows rg*RPL .. rg*RPL + RPL - 1
    const uint32_t cbar = smem_u32(bars + kCbar);
    // Split barrier of the consumer warps (one arrival per warp, waited for later). Exits
    // are taken by whole warps, and a warp left waiting gives up after the bounded wait.
    auto consumer_arrive = [&]() {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(cbar);
    };
    auto consumer_wait = [&](int k) -> bool {
        return __all_sync(0xFFFFFFFFu,
                          mbar_wait(cbar, k & 1, a.abort_flag, a.status, a.spin_limit));
    };
    int armed = -1;   // the last item whose bank gathers this warp has issued
    // Leaving an aborted kernel at item k: the gathers this warp issued land first (item
    // k's if its arrival was not yet seen, and item k+1's if already issued), each wait
    // bounded: a phase that another warp never armed does not complete, and its wait
    // runs to the bound, by which time every copy issued has long landed.
    auto leave = [&](int k, bool seen) {
        if (lane == 0) {
            if (!seen && armed >= k) {
                mbar_drain(smem_u32(bars + kFullW), k & 1, kDrainCycles);
                mbar_drain(smem_u32(bars + kFullR + (k & 1)), (k >> 1) & 1, kDrainCycles);
            }
            if (armed == k + 1) {
                mbar_drain(smem_u32(bars + kFullW), (k + 1) & 1, kDrainCycles);
                mbar_drain(smem_u32(bars + kFullR + ((k + 1) & 1)), ((k + 1) >> 1) & 1,
                           kDrainCycles);
            }
        }
        __syncwarp();
    };
    // Bank gathers of item kn, split over the consumer warps (8 bulk copies a warp at
    // W = 64). The full barriers count one arrival per consumer warp: each warp declares
    // the bytes of its own copies (arrive.expect_tx) before issuing them, so no copy can
    // land on a phase that does not expect it yet. For the empty end item each warp just
    // arrives.
    auto issue = [&](int kn) {
        armed = kn;
        const int pn = kn & 1;
        const Meta& mn = meta[pn];
        const uint32_t fw = smem_u32(bars + kFullW), fr = smem_u32(bars + kFullR + pn);
        if (!mn.valid) {
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(fw);
                mbar_arrive(fr);
            }
            return;
        }
        const uint32_t cb = (uint32_t)mn.rows * (uint32_t)sizeof(S);
        const bool is_r = lane >= 4;
        const int j = w + kCWarps * (lane & 3);
        const unsigned long long mask = is_r ? mn.rload : mn.wload;
        const bool chunk = lane < 8 && j < W && ((mask >> j) & 1);
        const bool wsel_copy = lane == 8 && w == 0, v_copy = lane == 8 && w == 1;
        const uint32_t wb = __reduce_add_sync(0xFFFFFFFFu, chunk && !is_r ? cb : 0u);
        const uint32_t rb = __reduce_add_sync(
            0xFFFFFFFFu, (chunk && is_r ? cb : 0u) + (wsel_copy ? 2u * W * 4 : 0u) + (v_copy ? cb : 0u));
        if (lane == 0) {
            mbar_arrive_expect_tx(fw, wb);
            mbar_arrive_expect_tx(fr, rb);
        }
        __syncwarp();
        // this thread's bank stores of earlier items before the copies read the bank (with
        // one token a sequence no item reads what another writes)
        if (a.T > 1)
            fence_proxy_async_global();
        const unsigned char* bank =
            a.banks + ((size_t)mn.b * a.N * a.d + (size_t)mn.rb * a.rb_rows) * sizeof(S);
        if (chunk) {
            const int id = is_r ? mn.rid[j] : mn.wid[j];
            unsigned char* dst = is_r ? rbuf + ((size_t)pn * W + j) * RS : wbuf + (size_t)j * kStride;
            const bool from_m0 = (((is_r ? mn.m0r : mn.m0w) >> j) & 1) != 0;
            const unsigned char* src =
                from_m0 ? a.m0 + ((size_t)id * a.d + (size_t)mn.rb * a.rb_rows) * sizeof(S)
                        : bank + (size_t)id * a.d * sizeof(S);
            bulk_g2s(smem_u32(dst), src, cb, is_r ? fr : fw);
        } else if (wsel_copy) {
            bulk_g2s(smem_u32(mn.wsel), a.wsel + mn.tok * 2 * W, 2 * W * 4, fr);
        } else if (v_copy) {
            bulk_g2s(smem_u32(mn.v), a.v + ((size_t)mn.tok * a.d + (size_t)mn.rb * a.rb_rows) * sizeof(S),
                     cb, fr);
        }
    };
    if (!uniform_wait(smem_u32(bars + kPosted), 0, a))
        return;
    issue(0);
    for (int k = 0;; ++k) {
        const int p = k & 1;
        if (!uniform_wait(smem_u32(bars + kFullW), k & 1, a) ||
            !uniform_wait(smem_u32(bars + kFullR + p), (k >> 1) & 1, a)) {
            leave(k, false);
            return;
        }
        const Meta& m = meta[p];
        if (!m.valid)
            return;
        unsigned char* rb_buf = rbuf + (size_t)p * W * RS;
        const bool act = rg * 16 < m.rows * (int)sizeof(S);
        if constexpr (kMmaY) {
            // The read's B fragments, [k-step][lane][2] flat: lane (g, q) of step ks holds
            // the weights of read slots 16 ks + 2q, + 1 (register 0) and + 8, + 9 (register
            // 1) in column g: the nearest bf16 in column 0, the nearest bf16 of what that
            // leaves in column 1 (about 16 bits of the fp32 weight together), zero elsewhere
            // and for slots out of range. The weights have landed with FullR; each warp
            // fills 16 entries, published to every warp by the consumer barrier below.
            uint32_t* bt = bfr + p * (W / 16) * 64;
            for (int e = w * 16 + lane; lane < 16 && e < (W / 16) * 64; e += kCWarps * 16) {
                const int reg = e & 1, ln = (e >> 1) & 31, ks = e >> 6;
                const int g = ln >> 2, j = 16 * ks + 2 * (ln & 3) + 8 * reg;
                const float w0 = ((m.rvalid >> j) & 1) ? m.wsel[W + j] : 0.f;
                const float w1 = ((m.rvalid >> (j + 1)) & 1) ? m.wsel[W + j + 1] : 0.f;
                bt[e] = weight_part_bits(w0, g) | (weight_part_bits(w1, g) << 16);
            }
        }
        // y = sum_j r_j M[R_j] (post-write). The chunks gathered from the bank need nothing
        // of the write: each thread reduces its read slots i*8 + sg, then the slot groups
        // are summed. Chunks D copies from the ring and this token's own writes are few;
        // the lane of slot group 0 adds them afterwards to the partial, which waits in
        // shared memory.
        float* ypart = ybuf + (w * 4 + (lane & 3)) * RPL;
        const bool y_rest = (m.rdmask | m.fmask) != 0;   // same for every thread
        auto y_bank = [&]() {
            float2 yv[HPL];
#pragma unroll
            for (int h = 0; h < HPL; ++h)
                yv[h] = make_float2(0.f, 0.f);
            const unsigned long long sel = m.rload;
#pragma unroll
            for (int i = 0; i < SPL; ++i) {
                if (!act || !((sel >> (i * kSG + sg)) & 1))
                    continue;
                const float rw = m.wsel[W + i * kSG + sg];
                float2 f[HPL];
                P::unpack(*reinterpret_cast<const uint4*>(rb_buf + (size_t)(i * kSG + sg) * RS +
                                                          rg * 16),
                          f);
#pragma unroll
                for (int h = 0; h < HPL; ++h)
                    yv[h] = __ffma2_rn(make_float2(rw, rw), f[h], yv[h]);
            }
#pragma unroll
            for (int h = 0; h < HPL; ++h)
                yv[h] = slot_group_sum(yv[h]);
            if (sg == 0 && act) {
                if (y_rest) {
#pragma unroll
                    for (int h = 0; h < HPL; h += 2)
                        *reinterpret_cast<float4*>(ypart + 2 * h) =
                            make_float4(yv[h].x, yv[h].y, yv[h + 1].x, yv[h + 1].y);
                } else {
                    float* yp = a.y + (size_t)m.tok * a.d + (size_t)m.rb * a.rb_rows + rg * RPL;
#pragma unroll
                    for (int h = 0; h < HPL; h += 2)
                        __stcs(reinterpret_cast<float4*>(yp + 2 * h),
                               make_float4(yv[h].x, yv[h].y, yv[h + 1].x, yv[h + 1].y));
                }
            }
        };
        // while a write-side dependency is still in flight, the bank chunks of the read
        // go first; otherwise the write goes first (later tokens wait for its ring entries)
        const bool bank_first = !kMmaY && !uniform_test(smem_u32(bars + kDepB + p), (k >> 1) & 1);
        if (bank_first)
            y_bank();
        if (!uniform_wait(smem_u32(bars + kDepB + p), (k >> 1) & 1, a)) {
            leave(k, true);
            return;
        }
        uint4 Mv[SPL];
#pragma unroll
        for (int i = 0; i < SPL; ++i)
            Mv[i] = act ? *reinterpret_cast<const uint4*>(wbuf + (size_t)(i * kSG + sg) * kStride +
                                                          rg * 16)
                        : make_uint4(0, 0, 0, 0);
        consumer_arrive();   // this warp has taken its write chunks
        if (a.tape != nullptr && act) {
            // the pre-write values of this token's write slots, for the backward pass
            unsigned char* tp = a.tape + ((size_t)m.tok * W * a.d + (size_t)m.rb * a.rb_rows) * sizeof(S) +
                                rg * 16;
#pragma unroll
            for (int i = 0; i < SPL; ++i)
                __stcs(reinterpret_cast<uint4*>(tp + (size_t)(i * kSG + sg) * a.d * sizeof(S)), Mv[i]);
        }

        // u = M_S k (pre-write), reduced over the slot groups; fp32 pairs throughout
        float2 u[HPL];
#pragma unroll
        for (int h = 0; h < HPL; ++h)
            u[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const float kw = m.wsel[i * kSG + sg];
            float2 f[HPL];
            P::unpack(Mv[i], f);
#pragma unroll
            for (int h = 0; h < HPL; ++h)
                u[h] = __ffma2_rn(make_float2(kw, kw), f[h], u[h]);
        }
        // every consumer has taken the write chunks: the buffer is free for item k+1
        if (!consumer_wait(k)) {
            leave(k, true);
            return;
        }
        if (ct == 0)
            mbar_arrive(smem_u32(bars + kWfree));
        const uint32_t posted_next = smem_u32(bars + kPosted + ((k + 1) & 1));
        const uint32_t lmark = smem_u32(bars + kLmark);
        bool issued = uniform_test(lmark, k & 1) && uniform_test(posted_next, ((k + 1) >> 1) & 1);
        if (issued)
            issue(k + 1);
        float2 vv[HPL];
        P::unpack(act ? *reinterpret_cast<const uint4*>(m.v + rg * 16) : make_uint4(0, 0, 0, 0), vv);
        const float al = m.alpha, be = m.beta;
        const float2 al2 = make_float2(al, al), be2 = make_float2(be, be);
        float2 c[HPL];   // beta (v - alpha u)
#pragma unroll
        for (int h = 0; h < HPL; ++h)
            c[h] = __fmul2_rn(be2, __ffma2_rn(make_float2(-al, -al), slot_group_sum(u[h]), vv[h]));
        // M[S_j] <- alpha M[S_j] + k_j beta (v - alpha u), rounded once
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const float kw = m.wsel[i * kSG + sg];
            float2 f[HPL];
            P::unpack(Mv[i], f);
#pragma unroll
            for (int h = 0; h < HPL; ++h)
                f[h] = __ffma2_rn(make_float2(kw, kw), c[h], __fmul2_rn(al2, f[h]));
            Mv[i] = P::pack(f);
        }
        // slots that later tokens read while this one may be in flight: to the ring
        // (this thread holds slots i*8 + sg: its bits of the mask are sg, sg+8, ...)
        const unsigned long long fw = (m.fwdmask >> sg) & 0x0101010101010101ull;
        if (fw != 0 && act) {
            unsigned char* re = ring_entry(a, m.b, m.rb, m.t, 0) + rg * 16;
#pragma unroll
            for (int i = 0; i < SPL; ++i)
                if ((fw >> (8 * i)) & 1)
                    __stcg(reinterpret_cast<uint4*>(re + (size_t)(i * kSG + sg) * a.chunk_bytes), Mv[i]);
        }
        __syncwarp();
        if (lane == 0) {
            // The last consumer warp done with the item's ring entries publishes them at
            // GPU scope itself (flag 2), one polling step sooner than the marks warp would:
            // each warp's arrival is a release at CTA scope, the last one's an acquire,
            // and its release at GPU scope carries the others' stores along. (With one
            // token a sequence nothing reads the flags; an item with no forwarded slot has
            // no ring entry that a later token copies, and the flag 3 its commit raises
            // answers every wait for flag 2.)
            if (a.T > 1 && m.fwdmask != 0) {
                int old;
                asm volatile("atom.acq_rel.cta.shared::cta.add.s32 %0, [%1], 1;"
                             : "=r"(old)
                             : "r"(smem_u32(fwdcnt + p))
                             : "memory");
                if (old % kCWarps == kCWarps - 1)
                    red_max_release_gpu(item_flag(a, m.b, m.rb, m.t), 2);
            }
            mbar_arrive(smem_u32(bars + kFwdw + p));
        }
        if constexpr (kMmaY) {
            // reads of slots this token writes: the new values go into the read buffer at
            // their read positions (rows of this warp's row groups only)
            if (m.fmask != 0 && act) {
#pragma unroll
                for (int i = 0; i < SPL; ++i) {
                    const int j = m.rpos[i * kSG + sg];
                    if (j >= 0)
                        *reinterpret_cast<uint4*>(rb_buf + (size_t)j * RS + rg * 16) = Mv[i];
                }
            }
            __syncwarp();
            // the read chunks D copies from writers still in flight (only items that have
            // some wait: the others stay clear of D's progress)
            if (m.rdmask != 0 && !uniform_wait(smem_u32(bars + kDepR + p), (k >> 1) & 1, a)) {
                leave(k, true);
                return;
            }
            // y of this warp's 32 rows: two 16-row tiles, W / 16 steps of 16 slots each;
            // A = the read chunks (ldmatrix.trans: slot rows of 8 consecutive state rows),
            // B = the weights in two bf16 parts (columns 0 and 1), fp32 accumulation
            const int gid = lane >> 2, tig = lane & 3;
            const uint32_t rbase = smem_u32(rb_buf) +
                                   (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * RS) +
                                   (uint32_t)(16 * ((lane >> 3) & 1));
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {
                const int m0 = w * 32 + 16 * t2;
                if (m0 >= m.rows)
                    break;                                   // (warp-uniform)
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < W / 16; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                 : "r"(rbase + (uint32_t)(ks * 16 * RS) + (uint32_t)(m0 * 2)));
                    const uint2 bb = reinterpret_cast<const uint2*>(bfr + p * (W / 16) * 64)[ks * 32 + lane];
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(bb.x), "r"(bb.y));
                }
                // columns 0 and 1 (the two parts of the weights) are in lanes tig = 0
                if (tig == 0) {
                    float* yp = a.y + (size_t)m.tok * a.d + (size_t)m.rb * a.rb_rows + m0 + gid;
                    __stcs(yp, c[0] + c[1]);
                    __stcs(yp + 8, c[2] + c[3]);
                }
            }
        }
        if (!kMmaY && !bank_first)
            y_bank();
        if (!kMmaY && y_rest) {
            // the read chunks D copies (writer still in flight when this item was described)
            if (!uniform_wait(smem_u32(bars + kDepR + p), (k >> 1) & 1, a)) {
                leave(k, true);
                return;
            }
            // own writes: the new value of write position pos is in the registers of slot
            // group pos % 8; that lane adds it, and a slot-group sum collects the terms
            float2 ye[HPL];
#pragma unroll
            for (int h = 0; h < HPL; ++h)
                ye[h] = make_float2(0.f, 0.f);
            const unsigned long long fm = m.fmask;
            if (fm != 0) {
                unsigned long long q = fm;
                while (q != 0) {
                    const int j = __ffsll((long long)q) - 1;
                    q &= q - 1;
                    const int pos = m.fpos[j];
                    if (!act || pos % kSG != sg)
                        continue;
                    const float rw = m.wsel[W + j];
                    // every register slot, weighted 0 but the one at pos (a selected
                    // register index would move Mv to local memory)
#pragma unroll
                    for (int i = 0; i < SPL; ++i) {
                        const float sc = i == pos / kSG ? rw : 0.f;
                        float2 f[HPL];
                        P::unpack(Mv[i], f);
#pragma unroll
                        for (int h = 0; h < HPL; ++h)
                            ye[h] = __ffma2_rn(make_float2(sc, sc), f[h], ye[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < HPL; ++h)
                    ye[h] = slot_group_sum(ye[h]);
            }
            if (sg == 0 && act) {
                // chunks copied by D, all of them, by this lane alone
                unsigned long long rd = m.rdmask;
                while (rd != 0) {
                    const int j = __ffsll((long long)rd) - 1;
                    rd &= rd - 1;
                    const float rw = m.wsel[W + j];
                    float2 f[HPL];
                    P::unpack(*reinterpret_cast<const uint4*>(rb_buf + (size_t)j * RS + rg * 16), f);
#pragma unroll
                    for (int h = 0; h < HPL; ++h)
                        ye[h] = __ffma2_rn(make_float2(rw, rw), f[h], ye[h]);
                }
                float* yp = a.y + (size_t)m.tok * a.d + (size_t)m.rb * a.rb_rows + rg * RPL;
#pragma unroll
                for (int h = 0; h < HPL; h += 2) {
                    const float4 pp = *reinterpret_cast<const float4*>(ypart + 2 * h);
                    __stcs(reinterpret_cast<float4*>(yp + 2 * h),
                           make_float4(pp.x + ye[h].x, pp.y + ye[h].y, pp.z + ye[h + 1].x,
                                       pp.w + ye[h + 1].y));
                }
            }
        }
        if (!issued && uniform_test(lmark, k & 1) &&
            uniform_test(posted_next, ((k + 1) >> 1) & 1)) {
            issue(k + 1);
            issued = true;
        }

        // bank stores, once cleared
        if (!uniform_wait(smem_u32(bars + kWar + p), (k >> 1) & 1, a)) {
            leave(k, true);
            return;
        }
        S* bank = reinterpret_cast<S*>(a.banks) + (size_t)m.b * a.N * a.d +
                  (size_t)m.rb * a.rb_rows + rg * RPL;
        const unsigned long long dead = m.deadmask;
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
            const int id = m.wid[i * kSG + sg];
            if (act && id >= 0 && !((dead >> (i * kSG + sg)) & 1))
                __stcg(reinterpret_cast<uint4*>(bank + (size_t)id * a.d), Mv[i]);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(bars + kStored + p));
        if (!issued) {
            if (!uniform_wait(lmark, k & 1, a) || !uniform_wait(posted_next, ((k + 1) >> 1) & 1, a)) {
                leave(k, true);
                return;
            }
            issue(k + 1);
        }
    }
}

template <typename S, int W>
__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(ScanArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ int fwdcnt[2];      // consumer warps done with an item's ring entries
    unsigned char* wbuf = smem;
    constexpr int RS = ScanShape<S, W>::kRStride;
    unsigned char* rbuf = smem + (size_t)W * kStride;
    Meta* meta = reinterpret_cast<Meta*>(smem + (size_t)W * kStride + (size_t)2 * W * RS);
    uint64_t* bars = reinterpret_cast<uint64_t*>(meta + 2);
    float* ybuf = reinterpret_cast<float*>(bars + kNumBars);   // [64 row groups][8 rows]
    uint32_t* bfr = reinterpret_cast<uint32_t*>(ybuf + (kChunk / 16) * 8);   // [2][W/16][32][2]
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bars + kFullW), kCWarps);
        mbar_init(smem_u32(bars + kWfree), 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(smem_u32(bars + kFullR + p), kCWarps);
            mbar_init(smem_u32(bars + kEmptyR + p), 2);     // F1 + M
            mbar_init(smem_u32(bars + kDepB + p), 1);
            mbar_init(smem_u32(bars + kDepR + p), 1);
            mbar_init(smem_u32(bars + kPosted + p), 1);
            mbar_init(smem_u32(bars + kWar + p), 1);
            mbar_init(smem_u32(bars + kFwdw + p), kCWarps);
            mbar_init(smem_u32(bars + kStored + p), kCWarps);
        }
        mbar_init(smem_u32(bars + kCbar), kCWarps);
        fwdcnt[0] = fwdcnt[1] = 0;
        mbar_init(smem_u32(bars + kLmark), 1);
        fence_mbarrier_init();
    }
    if (ScanShape<S, W>::kMmaY) {
        // the tensor-core read takes every slot of a read buffer (weight 0 where a slot id is
        // out of range): slots no copy ever reaches must hold finite values
        for (int e = threadIdx.x; e < 2 * W * RS / 16; e += blockDim.x)
            reinterpret_cast<uint4*>(rbuf)[e] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_shared();   // (before bulk copies write the buffers)
    }
    griddep_wait();   // (a programmatic launch: the kernel before has completed)
    griddep_launch();
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    // Register split: the block is launched with 96 registers a thread (640 x 96 =
    // 61,440). The four consumer warpgroups take 104 (4 x 128 x 104 = 53,248), the role
    // warpgroup (warps 16..19) gives back down to 64 (128 x 64 = 8,192): 61,440 in all.
    if (warp < kCWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kConsumerRegs) : "memory");
        role_consumer<S, W>(a, wbuf, rbuf, meta, bars, ybuf, bfr, fwdcnt);
        return;
    }
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRoleRegs) : "memory");
    if (warp == kWarpP)
        role_producer<S, W>(a, meta, bars);
    else if (warp == kWarpD)
        role_deps<S, W>(a, wbuf, rbuf, meta, bars);
    else if (warp == kWarpF1)
        role_clear<W>(a, meta, bars);
    else
        role_marks(a, meta, bars);
}

template <typename S, int W>
cudaError_t launch_scan_t(const ScanArgs& a, cudaStream_t s, bool early)
{
    const size_t smem = (size_t)W * kStride + (size_t)2 * W * ScanShape<S, W>::kRStride +
                        2 * sizeof(Meta) + kNumBars * sizeof(uint64_t) +
                        (size_t)(kChunk / 16) * 8 * sizeof(float) +  // partial y: 64 row groups x 8 rows
                        (size_t)2 * (W / 16 > 0 ? W / 16 : 1) * 64 * sizeof(uint32_t);  // B fragments
    auto kern = scan_kernel<S, W>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    long long grid = num_sms_current_device();
    if (grid > a.items)
        grid = a.items;
    if (!early) {
        kern<<<(unsigned)grid, kScanThreads, smem, s>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kScanThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

ScanWs scan_ws_layout(const sdm_cfg& c, int B, int T)
{
    ScanWs L{};
    const int es = c.dtype == SDM_BF16 ? 2 : 4;
    L.rb_rows = kChunk / es;
    L.nrb = (c.d + L.rb_rows - 1) / L.rb_rows;
    L.chunk_bytes = (c.d < L.rb_rows ? c.d : L.rb_rows) * es;
    // Window: the tokens of one stream the grid keeps in flight (one CTA per SM, about
    // two items each) plus 16, between 16 and kMaxWindow tokens. A wider window hands more
    // references over through the ring (a reference whose writer lies within the window
    // is copied from the writer's ring entry even when the writer is long done); a
    // narrower one holds tokens back until the window behind them has committed. Swept on
    // this GPU (d = 2048: one, two and four sequences, 74, 37 and 18.5 tokens in flight a
    // stream; d = 3840, two sequences), in flight + 16 sits at the optimum of every case.
    const long long streams = (long long)(B > 0 ? B : 1) * L.nrb;
    const double inflight = 2.0 * num_sms_current_device() / (double)streams;
    long long win = (long long)(inflight + 0.5) + 16;
    if (win < 16)
        win = 16;
    if (win > kMaxWindow)
        win = kMaxWindow;
    L.win = (int)win;
    L.ring_entries = T < 2 * L.win ? (T > 0 ? T : 1) : 2 * L.win;
    size_t o = 0;
    L.codes = o; o += align256((size_t)B * T * 2 * c.w * 2);
    L.masks = o; o += align256((size_t)B * T * 32);
    L.flags = o; L.flags_bytes = align256((size_t)B * L.nrb * T * 4) + 256; o += L.flags_bytes;
    L.min_total = o;
    L.ring = o;
    L.ring_bytes = (size_t)B * L.nrb * L.ring_entries * kMaxW * L.chunk_bytes;
    o += align256(L.ring_bytes);
    L.total = o;
    return L;
}

cudaError_t launch_scan(const sdm_cfg& c, const int32_t* idx, const float* wsel, const void* v,
                        const float* alpha, const float* beta, void* banks, float* y, int B,
                        int T, void* ws, size_t ws_bytes, int* status, cudaStream_t s,
                        const void* m0, const int32_t* first_write, void* tape,
                        long long spin_limit, long long skip_item, bool early)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    // one token a sequence: independent items, all in one wave (scan_step.cu)
    if (T == 1 && m0 == nullptr && first_write == nullptr && tape == nullptr && spin_limit <= 0 &&
        skip_item < 0 && scan_step_supported(c))
        return launch_scan_step(c, idx, wsel, v, alpha, beta, banks, y, B, status, s, early);
    const ScanWs L = scan_ws_layout(c, B, T);
    char* base = (char*)ws;
    if (!early) {
        const cudaError_t e = clear_scan_flags(c, B, T, ws, s);
        if (e != cudaSuccess)
            return e;
    }
    ScanArgs a;
    a.banks = (unsigned char*)banks;
    a.idx = idx;
    a.wsel = wsel;
    a.codes = (const uint16_t*)(base + L.codes);
    a.masks = (const unsigned long long*)(base + L.masks);
    a.v = (const unsigned char*)v;
    a.alpha = alpha;
    a.beta = beta;
    a.y = y;
    a.status = status;
    a.flags = (int*)(base + L.flags);
    a.counter = (unsigned long long*)(base + L.flags + L.flags_bytes - 256);
    a.abort_flag = (int*)(base + L.flags + L.flags_bytes - 128);
    a.ring = ws_bytes >= L.total ? (unsigned char*)(base + L.ring) : nullptr;
    a.m0 = (const unsigned char*)m0;
    a.first_write = first_write;
    a.tape = (unsigned char*)tape;
    a.B = B;
    a.T = T;
    a.d = c.d;
    a.N = c.n_sub * c.n_sub;
    a.nrb = L.nrb;
    a.rb_rows = L.rb_rows;
    a.win = L.win;
    a.ring_entries = L.ring_entries;
    a.chunk_bytes = L.chunk_bytes;
    a.items = (long long)B * T * a.nrb;
    a.spin_limit = spin_limit > 0 ? spin_limit : kSpinLimitCycles;
    a.skip_item = skip_item;
    const bool bf = c.dtype == SDM_BF16;
    switch (c.w) {
    case 8: return bf ? launch_scan_t<bf16, 8>(a, s, early) : launch_scan_t<float, 8>(a, s, early);
    case 16: return bf ? launch_scan_t<bf16, 16>(a, s, early) : launch_scan_t<float, 16>(a, s, early);
    case 32: return bf ? launch_scan_t<bf16, 32>(a, s, early) : launch_scan_t<float, 32>(a, s, early);
    case 64: return bf ? launch_scan_t<bf16, 64>(a, s, early) : launch_scan_t<float, 64>(a, s, early);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t clear_scan_flags(const sdm_cfg& c, int B, int T, void* ws, cudaStream_t s)
{
    const ScanWs L = scan_ws_layout(c, B, T);
    return cudaMemsetAsync((char*)ws + L.flags, 0, L.flags_bytes, s);
}

}  // namespace sdm
