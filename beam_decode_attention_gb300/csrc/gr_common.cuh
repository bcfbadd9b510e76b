// gr_common.cuh -- small device helpers shared by the kernels of libgrattn.so.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gr_internal.h"

namespace gr {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// N consecutive bf16 (N = 2, 4 or 8; 4N-byte aligned) widened to fp32.
template <int N>
__device__ __forceinline__ void load_bf16(const uint16_t *p, float (&f)[N]) {
    static_assert(N == 2 || N == 4 || N == 8, "vector width");
    if constexpr (N == 2) {
        uint32_t u = __ldg(reinterpret_cast<const unsigned int *>(p));
        f[0] = __uint_as_float(u << 16);
        f[1] = __uint_as_float(u & 0xffff0000u);
    } else if constexpr (N == 4) {
        uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
        f[4] = __uint_as_float(u.z << 16); f[5] = __uint_as_float(u.z & 0xffff0000u);
        f[6] = __uint_as_float(u.w << 16); f[7] = __uint_as_float(u.w & 0xffff0000u);
    }
}

// Two fp32 -> packed bf16x2 (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int N>
__device__ __forceinline__ void store_bf16(uint16_t *p, const float (&f)[N]) {
    static_assert(N == 2 || N == 4 || N == 8, "vector width");
    if constexpr (N == 2) {
        *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(f[0], f[1]);
    } else if constexpr (N == 4) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
    } else {
        *reinterpret_cast<uint4 *>(p) = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                   pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
}

template <int N>
__device__ __forceinline__ void load_f32(const float *p, float (&f)[N]) {
    static_assert(N == 2 || N == 4, "vector width");
    if constexpr (N == 2) {
        float2 v = *reinterpret_cast<const float2 *>(p);
        f[0] = v.x; f[1] = v.y;
    } else {
        float4 v = *reinterpret_cast<const float4 *>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
}

template <int N>
__device__ __forceinline__ void store_f32(float *p, const float (&f)[N]) {
    static_assert(N == 2 || N == 4, "vector width");
    if constexpr (N == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(f[0], f[1]);
    } else {
        *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

__device__ __forceinline__ void raise_device_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

}  // namespace gr
