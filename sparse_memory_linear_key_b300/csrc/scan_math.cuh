// scan_math.cuh -- the per-element arithmetic of the recurrence, shared by the
// persistent scan (scan.cu) and the one-token kernel (scan_step.cu) so that both compute
// the same bits ("Sparse Delta Memory" blog, "Write & Read": u = M_S k, the decayed delta
// write, the weighted read).
#pragma once

#include "sdm_common.cuh"

namespace sdm {

constexpr int kSG = 8;             // slot groups (lanes sharing a row group)

// 16 bytes of one slot vector (8 rows in bf16, 4 in fp32) as fp32 pairs, the operand
// of the packed two-lane fp32 FMA.
template <typename S>
struct Pack16;

template <>
struct Pack16<bf16> {
    static constexpr int R = 8;   // rows
    static constexpr int H = 4;   // fp32 pairs
    static __device__ __forceinline__ void unpack(const uint4& q, float2 (&f)[H])
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
    // round-to-nearest-even, once per value
    static __device__ __forceinline__ uint4 pack(const float2 (&f)[H])
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __float22bfloat162_rn(f[i]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Pack16<float> {
    static constexpr int R = 4;
    static constexpr int H = 2;
    static __device__ __forceinline__ void unpack(const uint4& q, float2 (&f)[H])
    {
        f[0] = make_float2(__uint_as_float(q.x), __uint_as_float(q.y));
        f[1] = make_float2(__uint_as_float(q.z), __uint_as_float(q.w));
    }
    static __device__ __forceinline__ uint4 pack(const float2 (&f)[H])
    {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                          __float_as_uint(f[1].y));
    }
};

// sum of a pair over the eight slot groups of a row group (lanes 4 apart)
__device__ __forceinline__ float2 slot_group_sum(float2 v)
{
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1)
        v = __fadd2_rn(v, make_float2(__shfl_xor_sync(0xFFFFFFFFu, v.x, o),
                                      __shfl_xor_sync(0xFFFFFFFFu, v.y, o)));
    return v;
}


// the part of a weight that column `part` of the B fragment holds: 0 the nearest bf16, 1
// the nearest bf16 of what that leaves (together about 16 bits of the fp32 weight)
__device__ __forceinline__ uint32_t weight_part_bits(float w, int part)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
    const __nv_bfloat16 v = part == 0 ? hi : lo;
    return part < 2 ? (uint32_t)*reinterpret_cast<const unsigned short*>(&v) : 0u;
}


}  // namespace sdm
