// sdm_internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

// slot rows handled by one scan "machine" (a warp group owning 16 rows of a bank)
constexpr int kScanRows = 16;
// forwarding window of the collision codes (tokens); the scan uses G - 1 <= it
constexpr int kFwdWindow = 31;
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
cudaError_t launch_fwd_codes(const sdm_cfg& c, const int32_t* idx, int B, int T,
                             uint16_t* codes, int* status, cudaStream_t s);

// ---- scan (scan.cu)
struct ScanLaunch {
    int G;    // warps (tokens in flight) per machine
    int MPC;  // machines per block
};
ScanLaunch choose_scan_launch(int B, int T, int d, int num_sms);
cudaError_t launch_scan(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                        const uint16_t* codes, const void* v, const float* alpha,
                        const float* beta, void* banks, float* y, int B, int T, ScanLaunch L,
                        int* status, cudaStream_t s);

int num_sms_current_device();

}  // namespace sdm
