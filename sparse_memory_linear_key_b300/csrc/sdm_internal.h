// sdm_internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

// d must be a multiple of this (16-byte aligned rows for bf16 and fp32 alike)
constexpr int kRowAlign = 16;
// window of the collision codes (tokens): a slot reference records its latest earlier
// writer only if it lies at most this many tokens back; older writers are guaranteed
// committed by the scan before the reference is loaded
constexpr int kFwdWindow = 128;
constexpr uint16_t kNoFwd = 0xFFFF;

// ---- bank initialisation (bank_init.cu)
cudaError_t launch_bank_init(const void* M0, void* banks, size_t bank_bytes, int B,
                             cudaStream_t s);

// ---- projections (project.cu)
int launch_project(const sdm_cfg& c, const sdm_weights& w, const void* x, int64_t ntok,
                   void* q_w, void* q_r, void* v, cudaStream_t s);

// ---- addressing (address.cu)
size_t address_ws_bytes(const sdm_cfg& c, int64_t ntok);
cudaError_t launch_address(const sdm_cfg& c, const void* K1, const void* K2, const void* q_w,
                           const void* q_r, int64_t ntok, int32_t* idx, float* wsel, void* ws,
                           int* status, cudaStream_t s);
// collision codes for the scan: [B*T, 2, w] uint16 (dt << 8 | position, or kNoFwd)
size_t fwd_codes_smem_bytes(const sdm_cfg& c);
cudaError_t launch_fwd_codes(const sdm_cfg& c, const int32_t* idx, int B, int T,
                             uint16_t* codes, int* status, cudaStream_t s);

// ---- scan (scan.cu)
// Scratch of one scan over B sequences of T tokens, inside the scan workspace after the
// collision codes: per (sequence, row block, token) progress flags and a work counter.
size_t scan_flags_bytes(const sdm_cfg& c, int B, int T);
// Rows of one row block (one 1 KB chunk of a slot vector) and the number of blocks.
int scan_block_rows(const sdm_cfg& c);
int scan_row_blocks(const sdm_cfg& c);
// Clears the flags (flags_bytes at `flags`) and launches the scan kernel.
cudaError_t launch_scan(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                        const uint16_t* codes, const void* v, const float* alpha,
                        const float* beta, void* banks, float* y, int B, int T, void* flags,
                        int* status, cudaStream_t s);

int num_sms_current_device();

}  // namespace sdm
