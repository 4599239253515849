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
// reverse; 4 groups of 64 threads share the W slots of a token (slot j in group j % 4).
// Sums over rows (dk, dr, dalpha, dbeta) are per-block partials, summed over the blocks
// of a sequence by a second kernel.
#include "sdm_common.cuh"
#include "sdm_internal.h"

namespace sdm {

namespace {

constexpr int kBRows = 64;
constexpr int kBThreads = 256;
constexpr int kBGroups = kBThreads / kBRows;

__device__ __forceinline__ float ld_state(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ld_state(const float* p) { return *p; }
__device__ __forceinline__ float ld_io(const bf16* p) { return __bfloat162float(__ldg(p)); }
__device__ __forceinline__ float ld_io(const float* p) { return __ldg(p); }

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

// partials: [nblk][B*T][2W + 2] = dk[W], dr[W], dalpha, dbeta of this block's rows
template <typename S, int W>
__global__ void __launch_bounds__(kBThreads) scan_bwd_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wsel, const S* __restrict__ v,
    const float* __restrict__ alpha, const float* __restrict__ beta, const S* __restrict__ tape,
    S* __restrict__ banks, const float* __restrict__ dy, float* __restrict__ dbank,
    float* __restrict__ dv, float* __restrict__ part, int B, int T, int d, int N)
{
    constexpr int SPG = W / kBGroups;         // slots a thread: j = grp + 4 i
    constexpr int P = 2 * W + 2;
    // Token t's slot ids, weights and gates sit in buffer t & 1 (written during token
    // t + 1), and so do its partial sums (cleared during token t + 1, after every thread
    // has written out token t + 2's).
    static_assert(2 * W <= kBThreads && P <= kBThreads, "one metadata entry a thread");
    __shared__ int sid[2][2][W];
    __shared__ float sw[2][2][W];
    __shared__ float gate[2][2];
    __shared__ float red[2][kBGroups][kBRows];
    __shared__ float acc[2][P];
    const int b = blockIdx.y;
    const int r = threadIdx.x % kBRows, grp = threadIdx.x / kBRows;
    const int row = blockIdx.x * kBRows + r;
    const bool act = row < d;
    const int lane = threadIdx.x & 31;
    const int e = threadIdx.x;                       // metadata entry of this thread
    S* bank = banks + (size_t)b * N * d;
    float* G = dbank + (size_t)b * N * d;
    if (T <= 0)
        return;
    // what a token needs besides the gradient bank, loaded one token ahead
    int nid = -1;
    float nw = 0.f, nal = 0.f, nbe = 0.f, ndy = 0.f, nv = 0.f;
    float nold[SPG];
    auto prefetch = [&](int64_t tk) {
        if (e < 2 * W) {
            nid = __ldg(idx + tk * 2 * W + e);
            nw = __ldg(wsel + tk * 2 * W + e);
        }
        if (e == 0) {
            nal = __ldg(alpha + tk);
            nbe = __ldg(beta + tk);
        }
        ndy = act ? __ldg(dy + tk * d + row) : 0.f;
        nv = act ? ld_io(v + tk * d + row) : 0.f;
#pragma unroll
        for (int i = 0; i < SPG; ++i)   // tape rows exist for every position, ids aside
            nold[i] = act ? ld_state(tape + ((size_t)tk * W + grp + kBGroups * i) * d + row) : 0.f;
    };
    auto publish = [&](int buf) {
        if (e < 2 * W) {
            sid[buf][e / W][e % W] = nid;
            sw[buf][e / W][e % W] = nw;
        }
        if (e == 0) {
            gate[buf][0] = nal;
            gate[buf][1] = nbe;
        }
    };
    prefetch((int64_t)b * T + T - 1);
    publish((T - 1) & 1);
    if (e < P) {
        acc[0][e] = 0.f;
        acc[1][e] = 0.f;
    }
    __syncthreads();
    for (int t = T - 1; t >= 0; --t) {
        const int64_t tok = (int64_t)b * T + t;
        const int cb = t & 1;
        const float dyr = ndy, vr = nv;
        float old[SPG];
#pragma unroll
        for (int i = 0; i < SPG; ++i)
            old[i] = nold[i];
        if (t > 0)
            prefetch(tok - 1);
        // ---- read: G[R_j] += r_j dy, dr_j = <M[R_j], dy> (M after this token's write).
        // All loads first, then the updates, then the sums over rows.
        float mv[SPG], gr[SPG];
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int s = sid[cb][1][grp + kBGroups * i];
            const bool ok = act && s >= 0 && s < N;
            mv[i] = ok ? ld_state(bank + (size_t)s * d + row) : 0.f;
            gr[i] = ok ? G[(size_t)s * d + row] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int j = grp + kBGroups * i;
            const int s = sid[cb][1][j];
            if (act && s >= 0 && s < N)
                G[(size_t)s * d + row] = fmaf(sw[cb][1][j], dyr, gr[i]);
        }
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const float pr = warp_sum(mv[i] * dyr);
            if (lane == 0)
                atomicAdd(&acc[cb][W + grp + kBGroups * i], pr);
        }
        __syncthreads();   // (A) a slot both read and written: its G update is visible below
        // every thread has written out token t + 1's partials (before A): clear them for
        // token t - 1, which starts after barrier C
        if (e < P)
            acc[cb ^ 1][e] = 0.f;
        // ---- write
        float gj[SPG];
        float gp = 0.f, up = 0.f;
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int j = grp + kBGroups * i;
            const int s = sid[cb][0][j];
            const bool ok = act && s >= 0 && s < N;
            if (!ok)
                old[i] = 0.f;
            gj[i] = ok ? G[(size_t)s * d + row] : 0.f;
            gp = fmaf(sw[cb][0][j], gj[i], gp);
            up = fmaf(sw[cb][0][j], old[i], up);
        }
        red[0][grp][r] = gp;
        red[1][grp][r] = up;
        __syncthreads();   // (B)
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int q = 0; q < kBGroups; ++q) {
            g += red[0][q][r];
            u += red[1][q][r];
        }
        const float al = gate[cb][0], be = gate[cb][1];
        const float c = vr - al * u;
        float pa = 0.f;
        float pk[SPG];
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const int j = grp + kBGroups * i;
            const int s = sid[cb][0][j];
            const float kj = sw[cb][0][j];
            pa = fmaf(gj[i], old[i] - be * kj * u, pa);
            pk[i] = be * gj[i] * c - al * be * g * old[i];
            if (act && s >= 0 && s < N) {
                G[(size_t)s * d + row] = al * (gj[i] - be * kj * g);
                // the tape value, stored back exactly (a stored value converts to fp32
                // and back unchanged)
                bank[(size_t)s * d + row] = S(old[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < SPG; ++i) {
            const float q = warp_sum(pk[i]);
            if (lane == 0)
                atomicAdd(&acc[cb][grp + kBGroups * i], q);
        }
        pa = warp_sum(pa);
        const float pb = warp_sum(grp == 0 ? g * c : 0.f);
        if (lane == 0) {
            atomicAdd(&acc[cb][2 * W], pa);
            atomicAdd(&acc[cb][2 * W + 1], pb);
        }
        if (grp == 0 && act)
            dv[tok * d + row] = be * g;
        // token t - 1's slot ids, weights and gates into the other buffer (token t + 1
        // finished with it before barrier A)
        if (t > 0)
            publish(cb ^ 1);
        __syncthreads();   // (C) partial sums complete; token t - 1's metadata visible
        if (e < P)
            part[((size_t)blockIdx.x * B * T + tok) * P + e] = acc[cb][e];
        // red is rewritten after token t - 1's barrier A, which every thread reaches only
        // after these reads; acc[cb] is cleared only after that barrier too
    }
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
cudaError_t launch_bwd_t(const int32_t* idx, const float* wsel, const void* v, const float* alpha,
                         const float* beta, const void* tape, void* banks, const float* dy,
                         float* dbank, float* dv, float* part, int B, int T, int d, int N,
                         cudaStream_t s)
{
    const dim3 grid((unsigned)((d + kBRows - 1) / kBRows), (unsigned)B);
    scan_bwd_kernel<S, W><<<grid, kBThreads, 0, s>>>(idx, wsel, (const S*)v, alpha, beta,
                                                     (const S*)tape, (S*)banks, dy, dbank, dv,
                                                     part, B, T, d, N);
    return cudaGetLastError();
}

}  // namespace

size_t scan_backward_ws_bytes(const sdm_cfg& c, int B, int T)
{
    const size_t nblk = (size_t)(c.d + kBRows - 1) / kBRows;
    return nblk * (size_t)B * T * (2 * c.w + 2) * sizeof(float);
}

cudaError_t launch_scan_backward(const sdm_cfg& c, const int32_t* idx, const float* wsel,
                                 const void* v, const float* alpha, const float* beta,
                                 const void* tape, void* banks, const float* dy, float* dbank,
                                 float* dv, float* dalpha, float* dbeta, float* dwsel, int B,
                                 int T, void* ws, cudaStream_t s)
{
    if (B <= 0 || T <= 0)
        return cudaSuccess;
    const int N = c.n_sub * c.n_sub;
    float* part = (float*)ws;
    const bool bf = c.dtype == SDM_BF16;
    cudaError_t e;
    switch (c.w) {
    case 8: e = bf ? launch_bwd_t<bf16, 8>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s)
                   : launch_bwd_t<float, 8>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s);
        break;
    case 16: e = bf ? launch_bwd_t<bf16, 16>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s)
                    : launch_bwd_t<float, 16>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s);
        break;
    case 32: e = bf ? launch_bwd_t<bf16, 32>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s)
                    : launch_bwd_t<float, 32>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s);
        break;
    case 64: e = bf ? launch_bwd_t<bf16, 64>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s)
                    : launch_bwd_t<float, 64>(idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, part, B, T, c.d, N, s);
        break;
    default: return cudaErrorInvalidValue;
    }
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
