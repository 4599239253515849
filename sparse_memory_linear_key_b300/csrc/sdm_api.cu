// sdm_api.cu -- the extern "C" entry points of libsdm.so (declared in include/sdm.h):
// argument validation, workspace layout and the launch sequence of each operation.
#include <cuda_runtime.h>

#include <mutex>

#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

int num_sms_current_device()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev] = v;
    }
    return cache[dev];
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Few tokens, several a sequence: only q_w and q_r are on the way to the addressing, so v
// is projected on a side stream forked off the caller's stream and joined back before the
// scan (event record / wait, so that a captured graph gets a parallel branch). One side
// stream and two events per device; the lock keeps another thread's call off them from
// the fork until the join is enqueued. (One token a sequence takes the early-launch chain
// in prefill_impl instead.) From M0 with several tokens a sequence, the same side stream
// takes the first-touch table and the fill of never-written slots while the caller's
// stream computes the collision codes: both need only the slot ids, the fill (bound by
// HBM) hides the codes (bound by the latency of their index), and the scan waits for both.
constexpr int64_t kForkTokens = 256;

struct ProjFork {
    bool ready = false;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_v = nullptr;
};
static ProjFork g_fork[64];
static std::mutex g_fork_mu;

static ProjFork* fork_state()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    ProjFork& f = g_fork[dev];
    if (f.ready)
        return &f;
    if (f.side == nullptr && cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking) != cudaSuccess)
        return nullptr;
    if (f.ev_fork == nullptr &&
        cudaEventCreateWithFlags(&f.ev_fork, cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    if (f.ev_v == nullptr && cudaEventCreateWithFlags(&f.ev_v, cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    f.ready = true;
    return &f;
}

// Shapes the scan alone needs (the recurrence does not care how the slots were
// chosen, so w <= n_sub is not required here): d % 16, w in {8,16,32,64}, w <= N.
static int check_scan_cfg(const sdm_cfg* cfg)
{
    if (cfg == nullptr)
        return SDM_EINVAL;
    const sdm_cfg& c = *cfg;
    if (c.d <= 0 || c.n_sub <= 0 || c.w <= 0 || (c.dtype != SDM_F32 && c.dtype != SDM_BF16))
        return SDM_EINVAL;
    if (c.d % kRowAlign != 0 || (c.w != 8 && c.w != 16 && c.w != 32 && c.w != 64))
        return SDM_EUNSUPPORTED;
    if ((long long)c.n_sub * c.n_sub < c.w || c.n_sub > 512)
        return SDM_EUNSUPPORTED;
    return SDM_OK;
}

static size_t esize(const sdm_cfg& c) { return c.dtype == SDM_BF16 ? 2 : 4; }

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? SDM_OK : SDM_ECUDA; }

// Workspace layout of a prefill / decode call over B sequences of T tokens.
struct PrefillWs {
    size_t q_w, q_r, v, idx, wsel, scan, addr, total;
};

static PrefillWs prefill_layout(const sdm_cfg& c, int B, int T)
{
    PrefillWs L;
    const int64_t ntok = (int64_t)B * T;
    size_t o = 0;
    const size_t W2 = (size_t)2 * c.w;
    L.q_w = o; o += align256((size_t)ntok * c.dk * esize(c));
    L.q_r = o; o += align256((size_t)ntok * c.dk * esize(c));
    L.v = o; o += align256((size_t)ntok * c.d * esize(c));
    L.idx = o; o += align256((size_t)ntok * W2 * 4);
    L.wsel = o; o += align256((size_t)ntok * W2 * 4);
    L.scan = o; o += scan_ws_layout(c, B, T).total;
    L.addr = o; o += align256(address_ws_bytes(c, ntok));
    L.total = o;
    return L;
}

}  // namespace sdm

using namespace sdm;

extern "C" {

const char* sdm_status_string(int status)
{
    switch (status) {
    case SDM_OK: return "SDM_OK";
    case SDM_EINVAL: return "SDM_EINVAL: invalid argument";
    case SDM_EUNSUPPORTED: return "SDM_EUNSUPPORTED: shape outside the supported set";
    case SDM_ECUDA: return "SDM_ECUDA: CUDA runtime or library error";
    case SDM_ETIMEOUT: return "SDM_ETIMEOUT: a bounded device wait ran out";
    case SDM_EWORKSPACE: return "SDM_EWORKSPACE: workspace too small";
    case SDM_ERANGE: return "SDM_ERANGE: slot id out of range on the device";
    default: return "unknown sdm status";
    }
}

const char* sdm_version(void) { return "0.1.0"; }

int sdm_check_cfg(const sdm_cfg* cfg)
{
    if (cfg == nullptr)
        return SDM_EINVAL;
    const sdm_cfg& c = *cfg;
    if (c.d <= 0 || c.n_sub <= 0 || c.dk <= 0 || c.w <= 0 ||
        (c.dtype != SDM_F32 && c.dtype != SDM_BF16))
        return SDM_EINVAL;
    if (c.d % kRowAlign != 0)
        return SDM_EUNSUPPORTED;
    if (c.w != 8 && c.w != 16 && c.w != 32 && c.w != 64)
        return SDM_EUNSUPPORTED;
    if (c.n_sub < c.w || c.n_sub > 512)
        return SDM_EUNSUPPORTED;
    if (c.dk % 2 != 0 || (c.dk / 2) % 8 != 0 || c.dk / 2 > 128)
        return SDM_EUNSUPPORTED;
    // the sub-key table of one half is staged in shared memory, padded to a power of two
    int P = 32;
    while (P < c.n_sub)
        P *= 2;
    const size_t smem = (size_t)(c.dk / 2) * P * esize(c) + 8 * (c.dk / 2) * 4;
    if (smem > 200 * 1024)
        return SDM_EUNSUPPORTED;
    return SDM_OK;
}

size_t sdm_address_workspace_bytes(const sdm_cfg* cfg, int64_t ntok)
{
    if (sdm_check_cfg(cfg) != SDM_OK || ntok < 0)
        return 0;
    return address_ws_bytes(*cfg, ntok);
}

size_t sdm_scan_workspace_bytes(const sdm_cfg* cfg, int B, int T)
{
    if (check_scan_cfg(cfg) != SDM_OK || B < 0 || T < 0)
        return 0;
    return scan_ws_layout(*cfg, B, T).total;
}

size_t sdm_scan_min_workspace_bytes(const sdm_cfg* cfg, int B, int T)
{
    if (check_scan_cfg(cfg) != SDM_OK || B < 0 || T < 0)
        return 0;
    return scan_ws_layout(*cfg, B, T).min_total;
}

size_t sdm_workspace_bytes(const sdm_cfg* cfg, int B, int T)
{
    if (sdm_check_cfg(cfg) != SDM_OK || B < 0 || T < 0)
        return 0;
    return prefill_layout(*cfg, B, T).total;
}

int sdm_init_bank(const sdm_cfg* cfg, const void* M0, void* banks, int B, void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || (B > 0 && (M0 == nullptr || banks == nullptr)) || !aligned16(M0) ||
        !aligned16(banks))
        return SDM_EINVAL;
    const size_t N = (size_t)cfg->n_sub * cfg->n_sub;
    const size_t bytes = N * cfg->d * esize(*cfg);
    const char* a = (const char*)M0;
    const char* b = (const char*)banks;
    if (B > 0 && a < b + bytes * B && b < a + bytes)
        return SDM_EINVAL;  // overlap
    return cuda_status(launch_bank_init(M0, banks, bytes, B, (cudaStream_t)stream));
}

int sdm_project(const sdm_cfg* cfg, const sdm_weights* w, const void* x, int64_t ntok,
                void* q_w, void* q_r, void* v, void* stream)
{
    int rc = sdm_check_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (w == nullptr || ntok < 0)
        return SDM_EINVAL;
    if (ntok == 0)
        return SDM_OK;
    const void* ptrs[] = {x, q_w, q_r, v, w->W_qw, w->W_qr, w->W_v};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p))
            return SDM_EINVAL;
    if (ntok > 0x7FFFFFFF)
        return SDM_EUNSUPPORTED;
    return cuda_status(launch_project_tc(*cfg, *w, x, ntok, q_w, q_r, v, (cudaStream_t)stream));
}

int sdm_address(const sdm_cfg* cfg, const void* K1, const void* K2, const void* q_w,
                const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                size_t ws_bytes, int* dev_status, void* stream)
{
    int rc = sdm_check_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (ntok < 0)
        return SDM_EINVAL;
    if (ntok == 0)
        return SDM_OK;
    const void* ptrs[] = {K1, K2, q_w, q_r, idx, wsel, ws};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p))
            return SDM_EINVAL;
    if (((uintptr_t)ws & 255u) != 0)
        return SDM_EINVAL;
    if (ws_bytes < address_ws_bytes(*cfg, ntok))
        return SDM_EWORKSPACE;
    return cuda_status(launch_address(*cfg, K1, K2, q_w, q_r, ntok, idx, wsel, ws, dev_status,
                                      (cudaStream_t)stream));
}

static int scan_impl(const sdm_cfg& c, const int32_t* idx, const float* wsel, const void* v,
                     const float* alpha, const float* beta, void* banks, float* y, int B, int T,
                     void* ws, size_t ws_bytes, int* dev_status, cudaStream_t s,
                     const void* m0 = nullptr, const int32_t* first_write = nullptr,
                     bool early = false)
{
    const ScanWs L = scan_ws_layout(c, B, T);
    char* base = (char*)ws;
    // one token a sequence: the scan matches a token's reads with its writes itself
    cudaError_t e = T > 1 ? launch_scan_codes(c, idx, B, T, L.win, (uint16_t*)(base + L.codes),
                                              (unsigned long long*)(base + L.masks), dev_status, s)
                          : cudaSuccess;
    if (e != cudaSuccess)
        return SDM_ECUDA;
    e = launch_scan(c, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes, dev_status, s, m0,
                    first_write, nullptr, 0, -1, early);
    return cuda_status(e);
}

int sdm_scan_prepare(const sdm_cfg* cfg, const int32_t* idx, int B, int T, void* ws,
                     size_t ws_bytes, int* dev_status, void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0)
        return SDM_EINVAL;
    if (B == 0 || T == 0)
        return SDM_OK;
    if (idx == nullptr || ws == nullptr || !aligned16(idx) || ((uintptr_t)ws & 255u) != 0)
        return SDM_EINVAL;
    const ScanWs L = scan_ws_layout(*cfg, B, T);
    if (ws_bytes < L.min_total)
        return SDM_EWORKSPACE;
    char* base = (char*)ws;
    return cuda_status(launch_scan_codes(*cfg, idx, B, T, L.win, (uint16_t*)(base + L.codes),
                                         (unsigned long long*)(base + L.masks), dev_status,
                                         (cudaStream_t)stream));
}

static int check_scan_args(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                           const void* v, const float* alpha, const float* beta, void* banks,
                           float* y, int B, int T, const void* ws, size_t ws_bytes,
                           int* dev_status)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0)
        return SDM_EINVAL;
    if (B == 0 || T == 0)
        return SDM_OK;
    const void* ptrs[] = {idx, wsel, v, alpha, beta, banks, y, ws, dev_status};
    for (const void* p : ptrs)
        if (p == nullptr)
            return SDM_EINVAL;
    const void* al[] = {idx, wsel, v, banks, y};
    for (const void* p : al)
        if (!aligned16(p))
            return SDM_EINVAL;
    if (((uintptr_t)ws & 255u) != 0)
        return SDM_EINVAL;
    if (ws_bytes < scan_ws_layout(*cfg, B, T).min_total)
        return SDM_EWORKSPACE;
    return SDM_OK;
}

int sdm_scan_run(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
                 const float* alpha, const float* beta, void* banks, float* y, int B, int T,
                 const void* ws, size_t ws_bytes, int* dev_status, void* stream)
{
    const int rc = check_scan_args(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes,
                                   dev_status);
    if (rc != SDM_OK || B == 0 || T == 0)
        return rc;
    return cuda_status(launch_scan(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T,
                                   const_cast<void*>(ws), ws_bytes, dev_status,
                                   (cudaStream_t)stream));
}

int sdm_scan_run_diag(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
                      const float* alpha, const float* beta, void* banks, float* y, int B, int T,
                      const void* ws, size_t ws_bytes, long long spin_limit_cycles,
                      long long skip_item, int* dev_status, void* stream)
{
    const int rc = check_scan_args(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes,
                                   dev_status);
    if (rc != SDM_OK || B == 0 || T == 0)
        return rc;
    return cuda_status(launch_scan(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T,
                                   const_cast<void*>(ws), ws_bytes, dev_status,
                                   (cudaStream_t)stream, nullptr, nullptr, nullptr,
                                   spin_limit_cycles, skip_item < 0 ? -1 : skip_item));
}

int sdm_scan(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
             const float* alpha, const float* beta, void* banks, float* y, int B, int T,
             void* ws, size_t ws_bytes, int* dev_status, void* stream)
{
    const int rc = check_scan_args(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes,
                                   dev_status);
    if (rc != SDM_OK || B == 0 || T == 0)
        return rc;
    return scan_impl(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes, dev_status,
                     (cudaStream_t)stream);
}

// ------------------------------------------------------------- first-touch init

static bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    const char* x = (const char*)a;
    const char* y = (const char*)b;
    return x < y + nb && y < x + na;
}

size_t sdm_first_touch_bytes(const sdm_cfg* cfg, int B)
{
    if (check_scan_cfg(cfg) != SDM_OK || B < 0)
        return 0;
    return (size_t)B * cfg->n_sub * cfg->n_sub * sizeof(int32_t);
}

int sdm_first_touch(const sdm_cfg* cfg, const int32_t* idx, int B, int T, int32_t* first_write,
                    void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0)
        return SDM_EINVAL;
    if (B == 0)
        return SDM_OK;
    if (first_write == nullptr || (T > 0 && idx == nullptr) || !aligned16(first_write))
        return SDM_EINVAL;
    return cuda_status(launch_first_touch(*cfg, idx, B, T, first_write, (cudaStream_t)stream));
}

int sdm_scan_run_m0(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
                    const float* alpha, const float* beta, const void* M0,
                    const int32_t* first_write, void* banks, float* y, int B, int T, const void* ws,
                    size_t ws_bytes, int* dev_status, void* stream)
{
    const int rc = check_scan_args(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes,
                                   dev_status);
    if (rc != SDM_OK || B == 0 || T == 0)
        return rc;
    const size_t bank = (size_t)cfg->n_sub * cfg->n_sub * cfg->d * esize(*cfg);
    if (M0 == nullptr || first_write == nullptr || !aligned16(M0) ||
        overlaps(M0, bank, banks, bank * B))
        return SDM_EINVAL;
    return cuda_status(launch_scan(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T,
                                   const_cast<void*>(ws), ws_bytes, dev_status,
                                   (cudaStream_t)stream, M0, first_write));
}

int sdm_fill_untouched(const sdm_cfg* cfg, const void* M0, const int32_t* first_write,
                       void* banks, int B, int T, void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0)
        return SDM_EINVAL;
    if (B == 0)
        return SDM_OK;
    const size_t bank = (size_t)cfg->n_sub * cfg->n_sub * cfg->d * esize(*cfg);
    if (M0 == nullptr || first_write == nullptr || banks == nullptr || !aligned16(M0) ||
        !aligned16(banks) || overlaps(M0, bank, banks, bank * B))
        return SDM_EINVAL;
    return cuda_status(
        launch_fill_untouched(*cfg, M0, first_write, banks, B, T, (cudaStream_t)stream));
}

static int prefill_impl(const sdm_cfg* cfg, const sdm_weights* w, const void* M0, const void* x,
                        const float* alpha, const float* beta, void* banks, float* y, int B, int T,
                        int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes,
                        int* dev_status, void* stream)
{
    int rc = sdm_check_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (w == nullptr || B < 0 || T < 0)
        return SDM_EINVAL;
    if (B > 0 && T == 0 && M0 != nullptr)   // no tokens: the banks are just M0
        return sdm_init_bank(cfg, M0, banks, B, stream);
    if (B == 0 || T == 0)
        return SDM_OK;
    const void* ptrs[] = {x, alpha, beta, banks, y, ws, dev_status, w->K1, w->K2};
    for (const void* p : ptrs)
        if (p == nullptr)
            return SDM_EINVAL;
    const void* al[] = {x, banks, y, w->K1, w->K2, idx_out, w_out};
    for (const void* p : al)
        if (!aligned16(p))
            return SDM_EINVAL;
    if (((uintptr_t)ws & 255u) != 0)
        return SDM_EINVAL;
    const int64_t ntok = (int64_t)B * T;
    const PrefillWs L = prefill_layout(*cfg, B, T);
    const size_t bank = (size_t)cfg->n_sub * cfg->n_sub * cfg->d * esize(*cfg);
    if (M0 != nullptr && (!aligned16(M0) || overlaps(M0, bank, banks, bank * B)))
        return SDM_EINVAL;
    // M0 mode: the first-touch table follows the prefill workspace
    const size_t need = L.total + (M0 != nullptr ? align256((size_t)B * cfg->n_sub * cfg->n_sub * 4) : 0);
    if (ws_bytes < need)
        return SDM_EWORKSPACE;
    int32_t* first_write = M0 != nullptr ? (int32_t*)((char*)ws + L.total) : nullptr;
    char* base = (char*)ws;
    void* q_w = base + L.q_w;
    void* q_r = base + L.q_r;
    void* v = base + L.v;
    int32_t* idx = idx_out ? idx_out : (int32_t*)(base + L.idx);
    float* wsel = w_out ? w_out : (float*)(base + L.wsel);

    cudaStream_t s = (cudaStream_t)stream;
    if (ntok > 0x7FFFFFFF)
        return SDM_EUNSUPPORTED;
    std::unique_lock<std::mutex> lock;
    ProjFork* f = nullptr;
    bool ok = true;
    // One token a sequence (a decode step): projections -> addressing -> scan is a chain
    // of three short kernels, each launched early (programmatic dependent launch): the
    // projections set up while the kernel before them (the previous step's scan) ends, the
    // addressing stages its sub-key table while the projections run, the scan sets up
    // while the addressing runs. One projection launch for q and v, and the scan's flags
    // cleared by the addressing kernel, so that each kernel has one kernel before it and
    // nothing else lies between them.
    const bool early = T == 1 && ntok <= kForkTokens;
    void* scan_ws = base + L.scan;
    const ScanWs SL = scan_ws_layout(*cfg, B, T);
    if (early) {
        ok = launch_project_tc(*cfg, *w, x, ntok, q_w, q_r, v, s, 7, true) == cudaSuccess;
    } else if (ntok <= kForkTokens) {
        lock = std::unique_lock<std::mutex>(g_fork_mu);
        f = fork_state();
        if (f == nullptr)
            return SDM_ECUDA;
        if (cudaEventRecord(f->ev_fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(f->side, f->ev_fork, 0) != cudaSuccess)
            return SDM_ECUDA;
        ok = launch_project_tc(*cfg, *w, x, ntok, q_w, q_r, v, f->side, 4) == cudaSuccess;
        // the side stream is joined back whatever happened (a forked capture must rejoin)
        if (cudaEventRecord(f->ev_v, f->side) != cudaSuccess)
            return SDM_ECUDA;
        ok = ok && launch_project_tc(*cfg, *w, x, ntok, q_w, q_r, v, s, 3) == cudaSuccess;
    } else {
        ok = launch_project_tc(*cfg, *w, x, ntok, q_w, q_r, v, s) == cudaSuccess;
    }
    // from M0 with several tokens a sequence: first touch and fill beside the codes
    const bool fill_beside = M0 != nullptr && T > 1;
    ok = ok &&
         launch_address(*cfg, w->K1, w->K2, q_w, q_r, ntok, idx, wsel, base + L.addr, dev_status,
                        s, ntok <= kForkTokens, early ? (char*)scan_ws + SL.flags : nullptr,
                        early ? SL.flags_bytes : 0) == cudaSuccess &&
         (M0 == nullptr || fill_beside ||
          launch_first_touch(*cfg, idx, B, T, first_write, s) == cudaSuccess);
    if (f != nullptr) {
        // v is ready for the scan
        const bool joined = cudaStreamWaitEvent(s, f->ev_v, 0) == cudaSuccess;
        lock.unlock();
        ok = ok && joined;
    }
    if (!ok)
        return SDM_ECUDA;
    if (fill_beside) {
        lock = std::unique_lock<std::mutex>(g_fork_mu);
        f = fork_state();
        if (f == nullptr)
            return SDM_ECUDA;
        if (cudaEventRecord(f->ev_fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(f->side, f->ev_fork, 0) != cudaSuccess)
            return SDM_ECUDA;
        ok = launch_first_touch(*cfg, idx, B, T, first_write, f->side) == cudaSuccess &&
             launch_fill_untouched(*cfg, M0, first_write, banks, B, T, f->side) == cudaSuccess;
        // the side stream is joined back whatever happened (a forked capture must rejoin)
        if (cudaEventRecord(f->ev_v, f->side) != cudaSuccess)
            return SDM_ECUDA;
        ok = ok && launch_scan_codes(*cfg, idx, B, T, SL.win, (uint16_t*)((char*)scan_ws + SL.codes),
                                     (unsigned long long*)((char*)scan_ws + SL.masks), dev_status,
                                     s) == cudaSuccess;
        const bool joined = cudaStreamWaitEvent(s, f->ev_v, 0) == cudaSuccess;
        lock.unlock();
        if (!ok || !joined)
            return SDM_ECUDA;
        return cuda_status(launch_scan(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T, scan_ws,
                                       SL.total, dev_status, s, M0, first_write));
    }
    rc = scan_impl(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T, scan_ws, SL.total, dev_status,
                   s, M0, first_write, early);
    if (rc != SDM_OK || M0 == nullptr)
        return rc;
    return cuda_status(launch_fill_untouched(*cfg, M0, first_write, banks, B, T, s));
}

int sdm_prefill(const sdm_cfg* cfg, const sdm_weights* w, const void* x, const float* alpha,
                const float* beta, void* banks, float* y, int B, int T, int32_t* idx_out,
                float* w_out, void* ws, size_t ws_bytes, int* dev_status, void* stream)
{
    return prefill_impl(cfg, w, nullptr, x, alpha, beta, banks, y, B, T, idx_out, w_out, ws,
                        ws_bytes, dev_status, stream);
}

size_t sdm_prefill_m0_workspace_bytes(const sdm_cfg* cfg, int B, int T)
{
    const size_t base = sdm_workspace_bytes(cfg, B, T);
    if (base == 0)
        return 0;
    return base + align256((size_t)B * cfg->n_sub * cfg->n_sub * 4);
}

int sdm_prefill_m0(const sdm_cfg* cfg, const sdm_weights* w, const void* M0, const void* x,
                   const float* alpha, const float* beta, void* banks, float* y, int B, int T,
                   int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes, int* dev_status,
                   void* stream)
{
    if (M0 == nullptr)
        return SDM_EINVAL;
    return prefill_impl(cfg, w, M0, x, alpha, beta, banks, y, B, T, idx_out, w_out, ws, ws_bytes,
                        dev_status, stream);
}

// ------------------------------------------------------------ backward (a5 + a6)

size_t sdm_tape_bytes(const sdm_cfg* cfg, int B, int T)
{
    if (check_scan_cfg(cfg) != SDM_OK || B < 0 || T < 0)
        return 0;
    return (size_t)B * T * cfg->w * cfg->d * esize(*cfg);
}

int sdm_scan_run_train(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
                       const float* alpha, const float* beta, const void* M0,
                       const int32_t* first_write, void* banks, float* y, int B, int T,
                       const void* ws, size_t ws_bytes, void* tape, int* dev_status, void* stream)
{
    const int rc = check_scan_args(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws, ws_bytes,
                                   dev_status);
    if (rc != SDM_OK || B == 0 || T == 0)
        return rc;
    const size_t bank = (size_t)cfg->n_sub * cfg->n_sub * cfg->d * esize(*cfg);
    if (tape == nullptr || !aligned16(tape) || (M0 != nullptr) != (first_write != nullptr) ||
        (M0 != nullptr && (!aligned16(M0) || overlaps(M0, bank, banks, bank * B))))
        return SDM_EINVAL;
    return cuda_status(launch_scan(*cfg, idx, wsel, v, alpha, beta, banks, y, B, T,
                                   const_cast<void*>(ws), ws_bytes, dev_status,
                                   (cudaStream_t)stream, M0, first_write, tape));
}

size_t sdm_scan_backward_workspace_bytes(const sdm_cfg* cfg, int B, int T)
{
    if (check_scan_cfg(cfg) != SDM_OK || B < 0 || T < 0)
        return 0;
    return scan_backward_ws_bytes(*cfg, B, T);
}

int sdm_scan_backward(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
                      const float* alpha, const float* beta, const void* tape, void* banks,
                      const float* dy, float* dbank, float* dv, float* dalpha, float* dbeta,
                      float* dwsel, int B, int T, void* ws, size_t ws_bytes, void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0)
        return SDM_EINVAL;
    if (B == 0 || T == 0)
        return SDM_OK;
    const void* ptrs[] = {idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, dalpha, dbeta,
                          dwsel, ws};
    for (const void* p : ptrs)
        if (p == nullptr)
            return SDM_EINVAL;
    for (const void* p : ptrs)   // rows are staged by 16-byte copies
        if (!aligned16(p))
            return SDM_EINVAL;
    if ((uint64_t)cfg->n_sub * cfg->n_sub * (uint64_t)cfg->d > 0xFFFFFFFFull)
        return SDM_EUNSUPPORTED;   // offsets within one bank are 32-bit
    if (ws_bytes < scan_backward_ws_bytes(*cfg, B, T))
        return SDM_EWORKSPACE;
    return cuda_status(launch_scan_backward(*cfg, idx, wsel, v, alpha, beta, tape, banks, dy, dbank,
                                            dv, dalpha, dbeta, dwsel, B, T, ws,
                                            (cudaStream_t)stream));
}

size_t sdm_address_backward_workspace_bytes(const sdm_cfg* cfg, int64_t ntok)
{
    if (sdm_check_cfg(cfg) != SDM_OK || ntok < 0)
        return 0;
    return address_backward_ws_bytes(*cfg, ntok);
}

int sdm_address_backward(const sdm_cfg* cfg, const void* K1, const void* K2, const void* q_w,
                         const void* q_r, int64_t ntok, const int32_t* idx, const float* wsel,
                         const float* dwsel, float* dq_w, float* dq_r, float* dK1, float* dK2,
                         void* ws, size_t ws_bytes, void* stream)
{
    int rc = sdm_check_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (ntok < 0)
        return SDM_EINVAL;
    if (ntok == 0)
        return SDM_OK;
    const void* ptrs[] = {K1, K2, q_w, q_r, idx, wsel, dwsel, dq_w, dq_r, dK1, dK2, ws};
    for (const void* p : ptrs)
        if (p == nullptr)
            return SDM_EINVAL;
    if (((uintptr_t)ws & 255u) != 0)
        return SDM_EINVAL;
    if (ws_bytes < address_backward_ws_bytes(*cfg, ntok))
        return SDM_EWORKSPACE;
    return launch_address_backward(*cfg, K1, K2, q_w, q_r, ntok, idx, wsel, dwsel, dq_w, dq_r, dK1,
                                   dK2, ws, (cudaStream_t)stream);
}

size_t sdm_project_backward_workspace_bytes(const sdm_cfg* cfg, int64_t ntok)
{
    if (sdm_check_cfg(cfg) != SDM_OK || ntok < 0)
        return 0;
    return project_backward_ws_bytes(*cfg, ntok);
}

int sdm_project_backward(const sdm_cfg* cfg, const sdm_weights* w, const void* x, int64_t ntok,
                         const float* dq_w, const float* dq_r, const float* dv, float* dx,
                         float* dW_qw, float* dW_qr, float* dW_v, void* ws, size_t ws_bytes,
                         void* stream)
{
    int rc = sdm_check_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (w == nullptr || ntok < 0)
        return SDM_EINVAL;
    if (ntok == 0)
        return SDM_OK;
    const void* ptrs[] = {w->W_qw, w->W_qr, w->W_v, x, dq_w, dq_r, dv, dx, dW_qw, dW_qr, dW_v, ws};
    for (const void* p : ptrs)
        if (p == nullptr)
            return SDM_EINVAL;
    if (((uintptr_t)ws & 255u) != 0)
        return SDM_EINVAL;
    if (ws_bytes < project_backward_ws_bytes(*cfg, ntok))
        return SDM_EWORKSPACE;
    return launch_project_backward(*cfg, *w, x, ntok, dq_w, dq_r, dv, dx, dW_qw, dW_qr, dW_v, ws,
                                   (cudaStream_t)stream);
}

// ------------------------------------------------------ dense-state comparator

int sdm_gdn_dense_scan(const sdm_cfg* cfg, const float* S0, const float* kw, const float* kr,
                       int64_t k_stride, const void* v, const float* alpha, const float* beta,
                       float* S_out, float* y, int B, int T, void* stream)
{
    if (cfg == nullptr)
        return SDM_EINVAL;
    const sdm_cfg& c = *cfg;
    if (c.d <= 0 || (c.dtype != SDM_F32 && c.dtype != SDM_BF16) || B < 0 || T < 0)
        return SDM_EINVAL;
    if (c.w != 64 || c.d % kRowAlign != 0)
        return SDM_EUNSUPPORTED;
    if (B == 0)
        return SDM_OK;
    if (T > 0 && (kw == nullptr || kr == nullptr || v == nullptr || alpha == nullptr ||
                  beta == nullptr || y == nullptr))
        return SDM_EINVAL;
    if (k_stride < c.w || k_stride % 4 != 0 || !aligned16(kw) || !aligned16(kr) || !aligned16(S0) ||
        !aligned16(S_out) || ((uintptr_t)v & (esize(c) - 1)) != 0 || ((uintptr_t)y & 3u) != 0)
        return SDM_EINVAL;
    return cuda_status(launch_gdn_dense(c.dtype == SDM_BF16, S0, kw, kr, k_stride, v, alpha, beta,
                                        S_out, y, B, T, c.d, (cudaStream_t)stream));
}

// ------------------------------------------------------ slot-access statistics

static bool window_ok(int lo, int hi, int T) { return 0 <= lo && lo <= hi && hi <= T; }

int sdm_slot_counts(const sdm_cfg* cfg, const int32_t* idx, int B, int T, int kind, int t0, int t1,
                    uint32_t* counts, void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0 || (kind != 0 && kind != 1) || !window_ok(t0, t1, T))
        return SDM_EINVAL;
    if (B == 0)
        return SDM_OK;
    if (counts == nullptr || (t1 > t0 && idx == nullptr) || !aligned16(counts))
        return SDM_EINVAL;
    return cuda_status(
        launch_slot_counts(*cfg, idx, B, T, kind, t0, t1, counts, (cudaStream_t)stream));
}

size_t sdm_slot_overlap_workspace_bytes(const sdm_cfg* cfg, int B)
{
    if (check_scan_cfg(cfg) != SDM_OK || B < 0)
        return 0;
    return slot_overlap_ws_bytes(*cfg, B);
}

int sdm_slot_overlap(const sdm_cfg* cfg, const int32_t* idx, int B, int T, int w0, int w1, int r0,
                     int r1, uint32_t* out, void* ws, size_t ws_bytes, void* stream)
{
    int rc = check_scan_cfg(cfg);
    if (rc != SDM_OK)
        return rc;
    if (B < 0 || T < 0 || !window_ok(w0, w1, T) || !window_ok(r0, r1, T))
        return SDM_EINVAL;
    if (B == 0)
        return SDM_OK;
    if (out == nullptr || ws == nullptr || ((w1 > w0 || r1 > r0) && idx == nullptr) ||
        ((uintptr_t)ws & 15u) != 0)
        return SDM_EINVAL;
    if (ws_bytes < slot_overlap_ws_bytes(*cfg, B))
        return SDM_EWORKSPACE;
    return cuda_status(
        launch_slot_overlap(*cfg, idx, B, T, w0, w1, r0, r1, out, ws, (cudaStream_t)stream));
}

int sdm_decode_step(const sdm_cfg* cfg, const sdm_weights* w, const void* x, const float* alpha,
                    const float* beta, void* banks, float* y, int B, int32_t* idx_out,
                    float* w_out, void* ws, size_t ws_bytes, int* dev_status, void* stream)
{
    return sdm_prefill(cfg, w, x, alpha, beta, banks, y, B, 1, idx_out, w_out, ws, ws_bytes,
                       dev_status, stream);
}

}  // extern "C"
