/*
 * sdm.h -- C ABI of the B300 (sm_103a) Sparse Delta Memory layer library, libsdm.so.
 *
 * One Sparse Delta Memory (SDM) layer keeps a memory bank M of N = n_sub^2 slot
 * vectors of width d per sequence. Per token it (A) selects W write slots and W read
 * slots by product keys, (W) writes the write slots with a gated delta rule and
 * (R) returns the softmax-weighted sum of the read slots ("Sparse Delta Memory" blog
 * post, sections "How does SDM work?" and "Write & Read: slot selection, gated update,
 * and retrieval"; "Sparse Delta Memory: Scaling the State of Linear RNNs through
 * Sparsity", Abstract: the bank starts from a learned initial state).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous, base addresses 16-byte aligned. The library allocates no device
 *    memory; scratch comes from the caller's workspace `ws` of `ws_bytes` bytes
 *    (see the *_workspace_bytes queries; ws must be 256-byte aligned).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Calls only enqueue work on it and return; they do not synchronise.
 *  - The return value reports host-side validation and launch errors (sdm_status).
 *    Errors found on the device (an index out of range, a bounded wait that ran
 *    out) are written to *dev_status (a device int the caller zeroes; the first
 *    error wins) and are read by the caller after synchronising.
 *  - dtype SDM_BF16: x, weights, sub-keys, M0, banks, q and v are bf16; SDM_F32: all
 *    fp32. alpha, beta, selection weights and y are always fp32, slot ids int32.
 *  - Supported shapes: d % 16 == 0; w in {8, 16, 32, 64}; w <= n_sub <= 512;
 *    dk even, dk/2 % 8 == 0, dk/2 <= 128. Others return SDM_EUNSUPPORTED.
 *    sdm_init_bank and sdm_scan need only d % 16 == 0, w in {8, 16, 32, 64} and
 *    w <= N (the recurrence does not depend on how the slots were chosen).
 */
#ifndef SDM_H_
#define SDM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SDM_API __attribute__((visibility("default")))
#else
#define SDM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDM_OK = 0,
    SDM_EINVAL = -1,        /* bad argument: null pointer, misaligned, negative size */
    SDM_EUNSUPPORTED = -2,  /* valid but outside the supported shapes above */
    SDM_ECUDA = -3,         /* a CUDA runtime or library call failed */
    SDM_ETIMEOUT = -4,      /* device: a bounded wait inside a kernel ran out */
    SDM_EWORKSPACE = -5,    /* ws_bytes smaller than the matching *_workspace_bytes */
    SDM_ERANGE = -6         /* device: a slot id outside [0, N) reached a kernel */
} sdm_status;

typedef enum { SDM_F32 = 0, SDM_BF16 = 1 } sdm_dtype;

/* Layer shape. N = n_sub * n_sub slots; the same w is used for writing and reading
 * (the pages give one active-slot count W = 64 for both). */
typedef struct sdm_cfg {
    int d;      /* slot width = model width */
    int n_sub;  /* rows of each sub-key table */
    int dk;     /* query width; halves of dk/2 are scored against K1 and K2 */
    int w;      /* active slots per token, write and read */
    int dtype;  /* sdm_dtype */
} sdm_cfg;

/* Layer parameters (device pointers, dtype of the cfg):
 *   W_qw [d, dk], W_qr [d, dk], W_v [d, d], K1 [n_sub, dk/2], K2 [n_sub, dk/2]. */
typedef struct sdm_weights {
    const void* W_qw;
    const void* W_qr;
    const void* W_v;
    const void* K1;
    const void* K2;
} sdm_weights;

/* Human-readable name of a status code (static string). */
SDM_API const char* sdm_status_string(int status);

/* Library version, e.g. "0.1.0". */
SDM_API const char* sdm_version(void);

/* SDM_OK if the shape is supported, else SDM_EINVAL / SDM_EUNSUPPORTED. */
SDM_API int sdm_check_cfg(const sdm_cfg* cfg);

/* Workspace needed by sdm_prefill / sdm_decode_step for B sequences of T tokens
 * (decode: T = 1), by sdm_address for ntok tokens, and by sdm_scan (and its two steps).
 * sdm_scan_min_workspace_bytes is the smallest workspace the scan accepts: without the
 * room for its forwarding ring (slot values handed from a writer still in flight to a
 * later token) it runs, with the same results, but a token whose slot was just written
 * by another in-flight token waits for that writer's bank store instead. */
SDM_API size_t sdm_workspace_bytes(const sdm_cfg* cfg, int B, int T);
SDM_API size_t sdm_address_workspace_bytes(const sdm_cfg* cfg, int64_t ntok);
SDM_API size_t sdm_scan_workspace_bytes(const sdm_cfg* cfg, int B, int T);
SDM_API size_t sdm_scan_min_workspace_bytes(const sdm_cfg* cfg, int B, int T);

/* Bank initialisation from the learned initial state ("Sparse Delta Memory",
 * Abstract: the initial state of the memory is learned and used as parametric
 * memory): banks[b] = M0 for b < B, a bit copy.
 *   M0 [N, d], banks [B, N, d] (slot-major: slot s of sequence b at banks + (b*N+s)*d).
 * M0 and banks must not overlap. */
SDM_API int sdm_init_bank(const sdm_cfg* cfg, const void* M0, void* banks, int B, void* stream);

/* Projections ("Write & Read": the token embedding is projected to write keys; a
 * separate query projection selects the read slots): for ntok tokens
 *   q_w = x W_qw [ntok, dk], q_r = x W_qr [ntok, dk], v = x W_v [ntok, d],
 * fp32 accumulation, rounded once (bf16 RNE in SDM_BF16). x [ntok, d]. The order of the
 * fp32 sums depends only on (cfg, ntok): the same shape always gives the same bits. */
SDM_API int sdm_project(const sdm_cfg* cfg, const sdm_weights* wts, const void* x, int64_t ntok,
                void* q_w, void* q_r, void* v, void* stream);

/* Product-key addressing ("Write & Read": two sub-keys -> outer sum -> top-k, softmax
 * weights) of ntok write queries q_w [ntok, dk] and read queries q_r [ntok, dk]:
 *   s1 = K1 q[0:dk/2], s2 = K2 q[dk/2:dk], c_ij = s1_i + s2_j, slot i*n_sub + j;
 *   keep the w largest c (ties: smaller slot id), weights = softmax of the kept c.
 * Outputs, per token t and kind (0 = write, 1 = read):
 *   idx [ntok, 2, w] int32 slot ids in ascending order, wsel [ntok, 2, w] fp32 weights.
 * Scores are fp32 (bf16 x bf16 products, fp32 sums). */
SDM_API int sdm_address(const sdm_cfg* cfg, const void* K1, const void* K2, const void* q_w,
                const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                size_t ws_bytes, int* dev_status, void* stream);

/* The recurrence ("Write & Read": selected columns are first decayed, then written
 * with the delta rule; the output is a weighted sum of the retrieved columns) for B
 * sequences of T tokens, in token order per sequence:
 *   u = M_S k;  M[S_j] <- alpha M[S_j] + beta k_j (v - alpha u)  (stored once, rounded)
 *   y = sum_j r_j M[R_j]                                          (post-write bank)
 * idx/wsel as produced by sdm_address for the B*T tokens (token b*T+t): each set of
 * w slot ids distinct and in ascending order. v [B*T, d], alpha, beta [B*T] fp32,
 * banks [B, N, d] updated in place, y [B*T, d] fp32. A slot id outside [0, N) is
 * skipped and reported as SDM_ERANGE in *dev_status. */
SDM_API int sdm_scan(const sdm_cfg* cfg, const int32_t* idx, const float* wsel, const void* v,
             const float* alpha, const float* beta, void* banks, float* y, int B, int T,
             void* ws, size_t ws_bytes, int* dev_status, void* stream);

/* sdm_scan in two steps, for callers that time or overlap them separately:
 * sdm_scan_prepare computes, into ws, the collision codes of the B*T tokens' slot
 * sets (for each slot reference, the distance to the latest earlier write of the same
 * slot within a short window, and its position there); sdm_scan_run then runs the
 * recurrence with those codes. The same ws and idx must be passed to both (ws_bytes at
 * least sdm_scan_min_workspace_bytes, sdm_scan_workspace_bytes for the forwarding
 * ring); sdm_scan == sdm_scan_prepare followed by sdm_scan_run. */
SDM_API int sdm_scan_prepare(const sdm_cfg* cfg, const int32_t* idx, int B, int T, void* ws,
                             size_t ws_bytes, int* dev_status, void* stream);
SDM_API int sdm_scan_run(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                         const void* v, const float* alpha, const float* beta, void* banks,
                         float* y, int B, int T, const void* ws, size_t ws_bytes,
                         int* dev_status, void* stream);

/* Failure detection of the recurrence, for tests: sdm_scan_run with two diagnostic
 * controls. spin_limit_cycles bounds every wait inside the kernel, in SM clock cycles
 * (<= 0: the default of about one second). skip_item >= 0 names one work item that the
 * kernel claims and drops -- token t of sequence b on row block rb, numbered
 * (t * B + b) * nrb + rb with nrb = ceil(d * element bytes / 1024) -- so that the tokens
 * depending on it wait for it until their bound runs out. Such a run records
 * SDM_ETIMEOUT in *dev_status, every warp leaves once the copies it started have landed,
 * and the call returns normally (banks and y are then undefined; the device stays
 * usable). skip_item < 0 withholds nothing. Other arguments as sdm_scan_run. */
SDM_API int sdm_scan_run_diag(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                              const void* v, const float* alpha, const float* beta, void* banks,
                              float* y, int B, int T, const void* ws, size_t ws_bytes,
                              long long spin_limit_cycles, long long skip_item, int* dev_status,
                              void* stream);

/* Size of the device array that sdm_scan_noalloc uses as its scratch: 8 MiB. A call
 * needs sdm_scan_min_workspace_bytes(cfg, B, T) of it: the collision codes (B * T * w * 4
 * bytes), four ordering masks per token (B * T * 32 bytes) and one progress flag per
 * token and 1 KB row block of a slot vector (B * T * ceil(d * elem / 1024) * 4 bytes),
 * plus under 1 KB of alignment and counters; at w = 64, d = 2048 bf16 that is
 * B * T <= 27592 tokens. When sdm_scan_workspace_bytes(cfg, B, T) fits too, the call
 * also uses the forwarding ring. */
#define SDM_SCAN_NOALLOC_MAX_BYTES (8u << 20)

/* sdm_scan without a caller workspace, for callers that cannot allocate device
 * memory: a plugin inside an application that owns all device memory through its own
 * pool or budget and hands this code no allocator, or a latency-critical loop where a
 * cudaMalloc/cudaFree would synchronise the device. The pages have no counterpart: it
 * is the same recurrence as sdm_scan, with the scratch (the collision codes) kept in a
 * library-owned device array of SDM_SCAN_NOALLOC_MAX_BYTES that every GPU loading the
 * library holds until the process exits. Arguments as sdm_scan, minus ws / ws_bytes.
 *  - Returns SDM_EWORKSPACE, before touching the GPU, if sdm_scan_min_workspace_bytes(cfg,
 *    B, T) exceeds SDM_SCAN_NOALLOC_MAX_BYTES.
 *  - Allocates nothing (no cudaMalloc, cudaFree or allocating library call); it clears
 *    the flags it uses with cudaMemsetAsync on `stream`.
 *  - The first call on a device looks up the array's device address (once per device,
 *    with that device current); make that first call before any stream capture. The
 *    address is kept for the life of the process: after a cudaDeviceReset of that device
 *    it is stale, so do not call this entry point on a device that has been reset.
 *  - Every call shares the one array: calls whose work overlaps on the GPU (other
 *    streams, other host threads) race on it and must be serialised by the caller. */
SDM_API int sdm_scan_noalloc(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                             const void* v, const float* alpha, const float* beta,
                             void* banks, float* y, int B, int T, int* dev_status,
                             void* stream);

/* Whole layer over a prefill of B sequences of T tokens: sdm_project, sdm_address and
 * sdm_scan in one call. All scratch lives in ws: the call (like sdm_decode_step)
 * allocates nothing and synchronises nothing, so it can be captured in a CUDA graph. x [B, T, d], alpha/beta [B, T], banks [B, N, d] (in place),
 * y [B, T, d] fp32. idx_out [B, T, 2, w] / w_out [B, T, 2, w] optional (NULL = not
 * returned). ws: sdm_workspace_bytes(cfg, B, T) bytes. */
SDM_API int sdm_prefill(const sdm_cfg* cfg, const sdm_weights* wts, const void* x, const float* alpha,
                const float* beta, void* banks, float* y, int B, int T, int32_t* idx_out,
                float* w_out, void* ws, size_t ws_bytes, int* dev_status, void* stream);

/* Bank initialisation fused into the recurrence. The learned initial state
 * ("Sparse Delta Memory: Scaling the State of Linear RNNs through Sparsity", Abstract)
 * is the same M0 for every sequence, and before token t a slot still holds M0 unless an
 * earlier token of its sequence wrote it. So instead of copying M0 into every bank
 * (sdm_init_bank, 2 * B * N * d elements of traffic), the scan loads M0 for those
 * references, and afterwards only the slots a sequence never wrote get M0's row. The
 * result is bit-identical to sdm_init_bank followed by the same calls without M0.
 *
 * sdm_first_touch: first_write [B, N] int32 <- for each sequence b and slot s, the first
 *   token t whose write set (idx[b*T+t][0][:]) holds s, or a value >= T if none;
 *   sdm_first_touch_bytes(cfg, B) = B * N * 4 bytes, 16-byte aligned, caller-owned.
 * sdm_scan_run_m0: sdm_scan_run with banks that start as M0 (their content on entry is
 *   read only for slots written earlier in the same call); M0 [N, d] must not overlap
 *   banks, first_write from sdm_first_touch on the same idx, B and T.
 * sdm_fill_untouched: banks[b][s] <- M0[s] wherever first_write[b][s] >= T.
 * sdm_prefill_m0: sdm_prefill from M0: the banks' content on entry is ignored; on
 *   return they hold the state after the T tokens, as after sdm_init_bank + sdm_prefill.
 *   ws: sdm_prefill_m0_workspace_bytes(cfg, B, T) (the prefill workspace plus the
 *   first-touch table). T = 0 copies M0 into the banks. */
SDM_API size_t sdm_first_touch_bytes(const sdm_cfg* cfg, int B);
SDM_API int sdm_first_touch(const sdm_cfg* cfg, const int32_t* idx, int B, int T,
                            int32_t* first_write, void* stream);
SDM_API int sdm_scan_run_m0(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                            const void* v, const float* alpha, const float* beta, const void* M0,
                            const int32_t* first_write, void* banks, float* y, int B, int T,
                            const void* ws, size_t ws_bytes, int* dev_status, void* stream);
SDM_API int sdm_fill_untouched(const sdm_cfg* cfg, const void* M0, const int32_t* first_write,
                               void* banks, int B, int T, void* stream);
SDM_API size_t sdm_prefill_m0_workspace_bytes(const sdm_cfg* cfg, int B, int T);
SDM_API int sdm_prefill_m0(const sdm_cfg* cfg, const sdm_weights* wts, const void* M0,
                           const void* x, const float* alpha, const float* beta, void* banks,
                           float* y, int B, int T, int32_t* idx_out, float* w_out, void* ws,
                           size_t ws_bytes, int* dev_status, void* stream);

/* Backward of the recurrence (the write and the read; the method is trained end to
 * end, "Sparse Delta Memory: Scaling the State of Linear RNNs through Sparsity",
 * Abstract). Two calls:
 * sdm_scan_run_train: sdm_scan_run (or sdm_scan_run_m0 when M0 / first_write are given,
 *   both or neither) that also records, per token, the pre-write values of its write
 *   slots: tape [B*T, w, d] in the state type, sdm_tape_bytes(cfg, B, T) bytes.
 * sdm_scan_backward: given dy [B*T, d] fp32 (the gradient of the loss with respect to y)
 *   and dbank [B, N, d] fp32 (in: with respect to the banks after the tokens, zeros if
 *   they do not enter the loss; out: with respect to the banks before the tokens --
 *   with banks from M0, dL/dM0 = sum over b of dbank[b]), it writes
 *   dv [B*T, d], dalpha, dbeta [B*T] and dwsel [B*T, 2, w] (write then read weights),
 *   all fp32. banks (in: the state after the tokens, as the forward left it; out: the
 *   state before them) are walked back with the tape. idx, wsel, v, alpha, beta as in
 *   the forward. ws: sdm_scan_backward_workspace_bytes(cfg, B, T) (per-block partial
 *   sums and per-token slot descriptors: row offsets and the slots shared with the
 *   neighbouring tokens). Every pointer
 *   is 16-byte aligned (SDM_EINVAL otherwise); N * d must be below 2^32
 *   (SDM_EUNSUPPORTED otherwise). The stored state's rounding is differentiated as
 *   the identity. */
SDM_API size_t sdm_tape_bytes(const sdm_cfg* cfg, int B, int T);
SDM_API int sdm_scan_run_train(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                               const void* v, const float* alpha, const float* beta,
                               const void* M0, const int32_t* first_write, void* banks, float* y,
                               int B, int T, const void* ws, size_t ws_bytes, void* tape,
                               int* dev_status, void* stream);
SDM_API size_t sdm_scan_backward_workspace_bytes(const sdm_cfg* cfg, int B, int T);
SDM_API int sdm_scan_backward(const sdm_cfg* cfg, const int32_t* idx, const float* wsel,
                              const void* v, const float* alpha, const float* beta,
                              const void* tape, void* banks, const float* dy, float* dbank,
                              float* dv, float* dalpha, float* dbeta, float* dwsel, int B, int T,
                              void* ws, size_t ws_bytes, void* stream);

/* Backward of the addressing: given dwsel [ntok, 2, w] fp32 (the gradient of the loss
 * with respect to the selection weights wsel of sdm_address, e.g. from
 * sdm_scan_backward), with the kept slots idx held fixed (the top-w selection is
 * piecewise constant), writes dq_w, dq_r [ntok, dk] and dK1, dK2 [n_sub, dk/2], fp32,
 * overwritten. q_w, q_r, K1, K2, idx, wsel as in sdm_address. Softmax backward per
 * token, then strict-fp32 GEMMs on the dense score gradients. ws:
 * sdm_address_backward_workspace_bytes(cfg, ntok), 256-byte aligned. */
SDM_API size_t sdm_address_backward_workspace_bytes(const sdm_cfg* cfg, int64_t ntok);
SDM_API int sdm_address_backward(const sdm_cfg* cfg, const void* K1, const void* K2,
                                 const void* q_w, const void* q_r, int64_t ntok,
                                 const int32_t* idx, const float* wsel, const float* dwsel,
                                 float* dq_w, float* dq_r, float* dK1, float* dK2, void* ws,
                                 size_t ws_bytes, void* stream);

/* Backward of the projections: with dq_w, dq_r [ntok, dk] and dv [ntok, d] fp32 (the
 * gradients with respect to sdm_project's outputs; their rounding is passed through),
 * writes dx [ntok, d] = dq_w W_qw^T + dq_r W_qr^T + dv W_v^T and dW_qw, dW_qr [d, dk],
 * dW_v [d, d] = x^T d(out), fp32, overwritten. GEMMs on fp32 copies of x and the
 * weights: strict fp32 for an fp32 layer; TF32 tensor cores for a bf16 layer (x and
 * the weights are exact in TF32, the incoming gradients are rounded to a relative
 * 2^-11, products summed in fp32). ws sdm_project_backward_workspace_bytes(cfg, ntok), 256-byte
 * aligned. With sdm_scan_backward and sdm_address_backward this completes the
 * gradients of one layer (dq_w, dq_r from the addressing, dv from the scan). */
SDM_API size_t sdm_project_backward_workspace_bytes(const sdm_cfg* cfg, int64_t ntok);
SDM_API int sdm_project_backward(const sdm_cfg* cfg, const sdm_weights* wts, const void* x,
                                 int64_t ntok, const float* dq_w, const float* dq_r,
                                 const float* dv, float* dx, float* dW_qw, float* dW_qr,
                                 float* dW_v, void* ws, size_t ws_bytes, void* stream);

/* Dense-state comparator (NOT the method: a measured reference point). The pages set
 * SDM against gated-delta-net: SDM's W = 64 active slot vectors per token are exactly the
 * size of GDN's whole dense state, at identical FLOPs per token ("Sparse Delta Memory"
 * blog, "Background", "How does SDM work?"). This runs the same gated delta rule on a
 * dense state of W columns that every token updates, per sequence:
 *   u = S k;  S <- alpha S + beta (v - alpha u) k^T;  y = S r     (fp32 throughout)
 * S0 / S_out [B, d, W] fp32 (row-major per row; S0 NULL = zeros, S_out NULL = not
 * returned), kw / kr: write / read weights of token b*T+t at kw + (b*T+t)*k_stride
 * (W fp32 each; e.g. the wsel of sdm_address with k_stride = 2W, kr = kw + W), v [B*T, d]
 * in the I/O type, alpha / beta [B*T], y [B*T, d] fp32. cfg: d % 16 == 0, w == 64.
 * The state never leaves the chip: its traffic is the per-token inputs and y. */
SDM_API int sdm_gdn_dense_scan(const sdm_cfg* cfg, const float* S0, const float* kw,
                               const float* kr, int64_t k_stride, const void* v,
                               const float* alpha, const float* beta, float* S_out, float* y,
                               int B, int T, void* stream);

/* Slot-access statistics, the pages' diagnostic of how the memory is used ("Sparse
 * Delta Memory" blog, "Memory Access Patterns on a Needle-in-a-Haystack Task": which
 * slots are written and read at each token position, and whether the slots written at
 * the needle are the ones read at the query). idx [B, T, 2, w] as from sdm_address.
 * Slot ids outside [0, N) are not counted.
 * sdm_slot_counts: counts [B, N] uint32 (overwritten) <- for each sequence b and slot s,
 *   the number of tokens t in [t0, t1) whose write (kind 0) or read (kind 1) set holds
 *   s. Counts over [0, t) are the pages' cumulative writes up to position t.
 * sdm_slot_overlap: out [B, 3] uint32 <- per sequence: the distinct slots written by the
 *   tokens in [w0, w1), the distinct slots read by the tokens in [r0, r1), and the
 *   distinct slots in both (the write-read bucket overlap). ws:
 *   sdm_slot_overlap_workspace_bytes(cfg, B) (two N-bit maps per sequence).
 * Windows must satisfy 0 <= lo <= hi <= T (SDM_EINVAL otherwise). */
SDM_API int sdm_slot_counts(const sdm_cfg* cfg, const int32_t* idx, int B, int T, int kind,
                            int t0, int t1, uint32_t* counts, void* stream);
SDM_API size_t sdm_slot_overlap_workspace_bytes(const sdm_cfg* cfg, int B);
SDM_API int sdm_slot_overlap(const sdm_cfg* cfg, const int32_t* idx, int B, int T, int w0, int w1,
                             int r0, int r1, uint32_t* out, void* ws, size_t ws_bytes,
                             void* stream);

/* One decode step: advance B independent sequences by one token each ("Sparse Delta
 * Memory" blog, "How does SDM work?": per token, select, write, then read).
 * x [B, d], alpha/beta [B], banks [B, N, d] (in place), y [B, d] fp32.
 * idx_out [B, 2, w] int32 / w_out [B, 2, w] fp32 optional (NULL = not returned): the
 * slot sets and selection weights this step used, as sdm_address reports them.
 * ws: sdm_workspace_bytes(cfg, B, 1) bytes. */
SDM_API int sdm_decode_step(const sdm_cfg* cfg, const sdm_weights* wts, const void* x,
                    const float* alpha, const float* beta, void* banks, float* y, int B,
                    int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes,
                    int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SDM_H_ */
