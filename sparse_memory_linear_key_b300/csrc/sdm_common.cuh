// sdm_common.cuh -- device-side helpers shared by the SDM kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

using bf16 = __nv_bfloat16;

// Upper bound for every spin-wait inside a kernel, in SM clock cycles (about one
// second at 2 GHz). A wait that runs out records SDM_ETIMEOUT and the warp leaves.
constexpr long long kSpinLimitCycles = 2000000000LL;

__device__ __forceinline__ void report(int* status, int code)
{
    if (status != nullptr)
        atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ shared-memory flags

__device__ __forceinline__ int ld_acquire_cta(const int* p)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];"
                 : "=r"(v)
                 : "r"((uint32_t)__cvta_generic_to_shared(p))
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_release_cta(int* p, int v)
{
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(p)),
                 "r"(v)
                 : "memory");
}

// Spin until *flag >= target (acquire). Returns false if the wait ran out or another
// warp of the block raised *abort; then the caller must leave.
__device__ __forceinline__ bool wait_geq(const int* flag, int target, const int* abort,
                                         int* status)
{
    if (ld_acquire_cta(flag) >= target)
        return true;
    const long long t0 = clock64();
    while (true) {
        if (ld_acquire_cta(flag) >= target)
            return true;
        if (*(volatile const int*)abort)
            return false;
        if (clock64() - t0 > kSpinLimitCycles) {
            report(status, SDM_ETIMEOUT);
            *(volatile int*)abort = 1;
            return false;
        }
    }
}

// ------------------------------------------------------- 4-row vectors of state

// Four consecutive rows of one slot vector, in the storage type.
template <typename S>
struct Row4;

template <>
struct Row4<float> {
    using V = float4;
    static __device__ __forceinline__ V load_cg(const float* p) { return __ldcg((const float4*)p); }
    static __device__ __forceinline__ void store_cg(float* p, V v) { __stcg((float4*)p, v); }
    static __device__ __forceinline__ void to_f32(V v, float f[4])
    {
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    static __device__ __forceinline__ V from_f32(const float f[4])
    {
        return make_float4(f[0], f[1], f[2], f[3]);
    }
    static __device__ __forceinline__ V zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};

template <>
struct Row4<bf16> {
    using V = uint2;  // two packed bf16x2 words
    static __device__ __forceinline__ V load_cg(const bf16* p) { return __ldcg((const uint2*)p); }
    static __device__ __forceinline__ void store_cg(bf16* p, V v) { __stcg((uint2*)p, v); }
    static __device__ __forceinline__ void to_f32(V v, float f[4])
    {
        f[0] = __uint_as_float(v.x << 16);
        f[1] = __uint_as_float(v.x & 0xFFFF0000u);
        f[2] = __uint_as_float(v.y << 16);
        f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
    // round-to-nearest-even, once per value
    static __device__ __forceinline__ V from_f32(const float f[4])
    {
        __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
        V v;
        v.x = *reinterpret_cast<uint32_t*>(&a);
        v.y = *reinterpret_cast<uint32_t*>(&b);
        return v;
    }
    static __device__ __forceinline__ V zero() { return make_uint2(0u, 0u); }
};

// scalar load of the I/O type as fp32
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

// ------------------------------------------------------- ordered sort keys

// Monotone map of a float to uint32 (larger float -> larger key); -0 folds to +0.
__device__ __forceinline__ uint32_t float_order_bits(float f)
{
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_bits(uint32_t o)
{
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

// 64-bit key, ascending = larger score first, then smaller id.
__device__ __forceinline__ uint64_t desc_key(float score, uint32_t id)
{
    return ((uint64_t)(~float_order_bits(score)) << 32) | id;
}

__device__ __forceinline__ float key_score(uint64_t k)
{
    return float_from_order_bits(~(uint32_t)(k >> 32));
}

__device__ __forceinline__ uint32_t key_id(uint64_t k) { return (uint32_t)k; }

// Bitonic sort, ascending, of 32*E 64-bit keys held lane-major by one warp (lane l
// holds elements l*E .. l*E+E-1 in k[0..E-1]). E is a power of two.
template <int E, typename K>
__device__ __forceinline__ void warp_bitonic_sort(K (&k)[E])
{
    const int lane = threadIdx.x & 31;
    constexpr int P = 32 * E;
#pragma unroll
    for (int size = 2; size <= P; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < E) {
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    const int j = i ^ stride;
                    if (j > i) {
                        const int e = lane * E + i;
                        const bool up = (e & size) == 0;
                        K a = k[i], b = k[j];
                        const bool swap = up ? (a > b) : (a < b);
                        k[i] = swap ? b : a;
                        k[j] = swap ? a : b;
                    }
                }
            } else {
                const int lm = stride / E;
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    const int e = lane * E + i;
                    const K other = __shfl_xor_sync(0xFFFFFFFFu, k[i], lm);
                    const bool up = (e & size) == 0;
                    const bool lower = (e & stride) == 0;
                    const K mn = k[i] < other ? k[i] : other;
                    const K mx = k[i] < other ? other : k[i];
                    k[i] = (up == lower) ? mn : mx;
                }
            }
        }
    }
}

}  // namespace sdm

// ------------------------------------------------ global flags, mbarriers, bulk copies

namespace sdm {

__device__ __forceinline__ int ld_relaxed_gpu(const int* p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// *p = max(*p, v) with release semantics (monotone progress flags)
__device__ __forceinline__ void red_max_release_gpu(int* p, int v)
{
    asm volatile("red.release.gpu.global.max.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(int* p, int v)
{
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// orders this thread's earlier generic-proxy accesses of global memory before its later
// async-proxy (bulk copy) accesses, and vice versa
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream still runs, and
// griddep_wait() blocks until that kernel has completed and its memory is visible; a
// kernel launched without it passes straight through. griddep_launch() lets the next
// kernel start once every CTA of this one has issued it (or exited). Kernels of this
// library issue it only after their own wait, so a kernel that starts early overlaps
// only the kernel right before it, never work further back in the stream.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Declares `bytes` of the current phase's transactions done without a copy (used when
// copies that were counted will not be issued).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.complete_tx.shared::cta.relaxed.cta.b64 [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking: has the phase of parity `parity` completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// How often a wait that goes on looks at the global abort flag and its own bound: a
// read of the flag is a round trip to L2, and a wait that made one on every pass would
// notice its own barrier only that much later. Aborts come from errors alone, so a few
// microseconds' delay in seeing one costs nothing.
constexpr long long kAbortPollCycles = 4096;

// Bounded wait for the phase of parity `parity` of an mbarrier. Returns false if the
// global abort flag is raised (abort may be null: not watched) or the wait ran out;
// a wait that ran out records SDM_ETIMEOUT and raises the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* abort, int* status,
                                          long long limit = kSpinLimitCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    long long next = t0 + kAbortPollCycles;
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        const long long now = clock64();
        if (now < next)
            continue;
        next = now + kAbortPollCycles;
        if (abort != nullptr && ld_relaxed_gpu(abort) != 0)
            return false;
        if (now - t0 > limit) {
            report(status, SDM_ETIMEOUT);
            if (abort != nullptr)
                st_relaxed_gpu(abort, 1);
            return false;
        }
    }
}

// Bounded wait until *f >= target (relaxed reads; the caller follows a successful wait
// with fence_acq_rel_gpu() to make it an acquire).
__device__ __forceinline__ bool spin_geq_gpu(const int* f, int target, int* abort, int* status,
                                             long long limit = kSpinLimitCycles)
{
    if (ld_relaxed_gpu(f) >= target)
        return true;
    const long long t0 = clock64();
    long long next = t0 + kAbortPollCycles;
    while (true) {
        __nanosleep(32);
        if (ld_relaxed_gpu(f) >= target)
            return true;
        const long long now = clock64();
        if (now < next)
            continue;
        next = now + kAbortPollCycles;
        if (ld_relaxed_gpu(abort) != 0)
            return false;
        if (now - t0 > limit) {
            report(status, SDM_ETIMEOUT);
            st_relaxed_gpu(abort, 1);
            return false;
        }
    }
}

// Wait for an mbarrier phase for at most `limit` cycles, ignoring the abort flag and
// reporting nothing: used on the way out of an aborted kernel, to let copies this warp
// started land before the CTA's shared memory is released.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, long long limit)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - t0 <= limit) {
    }
}

// Bulk copy global -> shared (this CTA), completing `bytes` transactions on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 16-byte copy global -> shared through the load/store unit (L2 only, no L1).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has completed (the
// pending count is raised now and dropped on completion, so the phase waits for it).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One warp copies `bytes` (a multiple of 16, at most 1024) from src to dst.
__device__ __forceinline__ void warp_copy_chunk(uint32_t dst, const unsigned char* src, uint32_t bytes)
{
    const uint32_t lane = threadIdx.x & 31;
#pragma unroll
    for (uint32_t off = lane * 16; off < 1024; off += 512)
        if (off < bytes)
            cp_async16(dst + off, src + off);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace sdm
