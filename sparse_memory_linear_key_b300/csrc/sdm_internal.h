// sdm_internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <mutex>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

// d must be a multiple of this (16-byte aligned rows for bf16 and fp32 alike)
constexpr int kRowAlign = 16;
// largest window of the collision codes (tokens): a slot reference records its latest
// earlier writer only if it lies at most `win` <= this many tokens back; older writers
// are guaranteed committed by the scan before the reference is loaded
constexpr int kMaxWindow = 128;
constexpr uint16_t kNoFwd = 0xFFFF;

// ---- bank initialisation (bank_init.cu)
cudaError_t launch_bank_init(const void* M0, void* banks, size_t bank_bytes, int B,
                             cudaStream_t s);

// ---- projections (proj_tc.cu): q_w, q_r, v of ntok tokens in one launch (bf16: tcgen05
// tensor cores; fp32: SIMT fp32)
// which: bit 0 q_w, bit 1 q_r, bit 2 v (the products to compute)
// early: the launch may overlap the kernel before it in the stream (programmatic
// dependent launch); the kernel touches no global memory until that one has completed
cudaError_t launch_project_tc(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                              void* q_w, void* q_r, void* v, cudaStream_t s, int which = 7,
                              bool early = false);

// ---- addressing (address.cu, score_tc.cu)
// z with P(Z > z) = p for a standard normal Z (a starting bracket for exact top-W searches)
float normal_upper_quantile(double p);
bool score_tc_supported(const sdm_cfg& c);
cudaError_t launch_score_tc(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                            const void* q_r, int64_t ntok, float* hv, int32_t* hi, int* status,
                            cudaStream_t s);
size_t address_ws_bytes(const sdm_cfg& c, int64_t ntok);
// early: the launch may overlap the kernel before it in the stream (programmatic
// dependent launch), which must not write K1 or K2; only the few-token kernel uses it.
// clear / clear_bytes (a multiple of 4): a buffer zeroed along the way, for the kernel
// after (the scan's flags), so that no memset lies between the two
cudaError_t launch_address(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                           const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                           int* status, cudaStream_t s, bool early = false,
                           void* clear = nullptr, size_t clear_bytes = 0);

// ---- scan (scan.cu, scan_codes.cu)
// Layout of the scan's workspace for B sequences of T tokens (byte offsets):
//   codes    [B*T, 2, w] uint16  collision codes
//   masks    [4][B*T] uint64     per token: fwdmask, deadmask, warmask (2 words)
//   flags    [B, nrb, T] int     progress of each (token, row block) item, then a
//                                work counter and an abort flag (256 bytes)
//   ring     [B*nrb, R, w, chunk] forwarding ring (R = min(T, 2*win) entries)
// `min_total` covers codes..flags: with a workspace that small the scan runs without
// the ring (a dependent reference then waits for its writer's bank store).
struct ScanWs {
    size_t codes, masks, flags, flags_bytes, ring, ring_bytes, min_total, total;
    int win, nrb, rb_rows, ring_entries, chunk_bytes;
};
ScanWs scan_ws_layout(const sdm_cfg& c, int B, int T);
cudaError_t launch_scan_codes(const sdm_cfg& c, const int32_t* idx, int B, int T, int win,
                              uint16_t* codes, unsigned long long* masks, int* status,
                              cudaStream_t s);
// Runs the recurrence; `ws` holds what launch_scan_codes wrote. ws_bytes >= L.total
// enables the forwarding ring.
// m0 / first_write non-null: the banks start as M0 without a copy (first_touch below)
cudaError_t launch_scan(const sdm_cfg& c, const int32_t* idx, const float* wsel, const void* v,
                        const float* alpha, const float* beta, void* banks, float* y, int B,
                        int T, void* ws, size_t ws_bytes, int* status, cudaStream_t s,
                        const void* m0 = nullptr, const int32_t* first_write = nullptr,
                        void* tape = nullptr, long long spin_limit = 0,
                        long long skip_item = -1, bool early = false);
// early (above): the flags are already clear (clear_scan_flags, issued earlier on the
// stream) and the kernel launches with programmatic dependent launch, overlapping the
// kernel before it until its first global access
cudaError_t clear_scan_flags(const sdm_cfg& c, int B, int T, void* ws, cudaStream_t s);
// One token a sequence (scan_step.cu): every (sequence, row block) item in one wave, same
// arithmetic and bits as launch_scan; bf16 state with w >= 16, no M0, no tape.
bool scan_step_supported(const sdm_cfg& c);
cudaError_t launch_scan_step(const sdm_cfg& c, const int32_t* idx, const float* wsel, const void* v,
                             const float* alpha, const float* beta, void* banks, float* y, int B,
                             int* status, cudaStream_t s, bool early);

// Backward of the recurrence (scan_bwd.cu): reverse token order over a gradient bank;
// ws holds per-block partial sums (scan_backward_ws_bytes).
size_t scan_backward_ws_bytes(const sdm_cfg& c, int B, int T);
cudaError_t launch_scan_backward(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                                 const void* v, const float* alpha, const float* beta,
                                 const void* tape, void* banks, const float* dy, float* dbank,
                                 float* dv, float* dalpha, float* dbeta, float* dwsel, int B,
                                 int T, void* ws, cudaStream_t s);

// first_write [B][N] <- the first token of each sequence that writes each slot, or a
// value >= T if none (bank_init.cu)
cudaError_t launch_first_touch(const sdm_cfg& c, const int32_t* idx, int B, int T,
                               int32_t* first_write, cudaStream_t s);
// row-major fp32 GEMM, C = op(A) op(B) + beta C, strict fp32, or on the tensor cores
// with the inputs rounded to TF32 (project.cu)
int gemm_f32_rm(cudaStream_t s, bool ta, bool tb, int M, int N, int K, const float* A, int lda,
                const float* B, int ldb, float* C, int ldc, float beta, bool tf32 = false);

// Backward of the addressing (addr_bwd.cu): selection-weight gradients -> dq, dK
size_t address_backward_ws_bytes(const sdm_cfg& c, int64_t ntok);
int launch_address_backward(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                            const void* q_r, int64_t ntok, const int32_t* idx, const float* wsel,
                            const float* dwsel, float* dq_w, float* dq_r, float* dK1, float* dK2,
                            void* ws, cudaStream_t s);

// Backward of the projections (addr_bwd.cu): dx, dW from dq_w, dq_r, dv
size_t project_backward_ws_bytes(const sdm_cfg& c, int64_t ntok);
int launch_project_backward(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                            const float* dq_w, const float* dq_r, const float* dv, float* dx,
                            float* dW_qw, float* dW_qr, float* dW_v, void* ws, cudaStream_t s);

// dense-state comparator (gdn_dense.cu): W = 64 columns, d % 16 == 0
cudaError_t launch_gdn_dense(bool bf_io, const float* S0, const float* kw, const float* kr,
                             int64_t ks, const void* v, const float* alpha, const float* beta,
                             float* S_out, float* y, int B, int T, int d, cudaStream_t s);

// slot-access statistics (slot_stats.cu)
size_t slot_overlap_ws_bytes(const sdm_cfg& c, int B);
cudaError_t launch_slot_counts(const sdm_cfg& c, const int32_t* idx, int B, int T, int kind,
                               int t0, int t1, uint32_t* counts, cudaStream_t s);
cudaError_t launch_slot_overlap(const sdm_cfg& c, const int32_t* idx, int B, int T, int w0, int w1,
                                int r0, int r1, uint32_t* out, void* ws, cudaStream_t s);

// banks[b][s] <- M0[s] for every slot sequence b never wrote (first_write >= T)
cudaError_t launch_fill_untouched(const sdm_cfg& c, const void* M0, const int32_t* first_write,
                                  void* banks, int B, int T, cudaStream_t s);

int num_sms_current_device();

}  // namespace sdm
