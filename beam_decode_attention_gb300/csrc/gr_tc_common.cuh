// gr_tc_common.cuh -- device helpers shared by the two tensor-core context
// kernels (the tile-pair kernel in gr_ctx_tc.cu and the persistent kernel in
// gr_ctx_pk.cu): bounded mbarrier waits, context-key coordinates for the
// dense and paged layouts, and the mixed-precision chain-score FMA.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gr_common.cuh"
#include "gr_ptx.cuh"

namespace gr {
namespace tc {

constexpr int kBM = 128;   // rows per tile = TMEM lanes
constexpr int kBN = 128;   // keys per block

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Warp-uniform bounded wait for an mbarrier phase: gives up after kSpinLimit
// polls or one second, or as soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    long long it = 0;
    uint64_t t0 = 0;
    while (true) {
        const bool ok = ptx::mbar_try_wait(bar, parity);
        if (__all_sync(kFullMask, ok)) return true;
        ++it;
        bool stop = (abort_flag != nullptr && *abort_flag != 0);
        if ((it & 4095) == 0) {   // slow path: only long waits read the clock
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > 1000000000ull) stop = true;
            if (it > kSpinLimit) stop = true;
        }
        if (__any_sync(kFullMask, stop)) return false;
    }
}

// Bounded wait by a single thread (the MMA issuer): same limits as wait_warp.
__device__ __forceinline__ bool wait_lane(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    long long it = 0;
    uint64_t t0 = 0;
    while (!ptx::mbar_try_wait(bar, parity)) {
        ++it;
        if (abort_flag != nullptr && *abort_flag != 0) return false;
        if ((it & 4095) == 0) {
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > 1000000000ull || it > kSpinLimit) return false;
        }
    }
    return true;
}

// Tensor-map coordinates (position, request-or-page) of context key `key`
// of request r: the dense layout [R, Hkv, Lc_max, D], or a paged pool
// [num_pages, Hkv, page_size, D] through the request's block table (page
// sizes are multiples of the 128-key block, so a block never straddles two
// pages).  A page index outside the pool lands outside the tensor map, where
// TMA reads zeros.
__device__ __forceinline__ void kv_coords(const CtxArgs &a, int r, int key, int &c1, int &c3) {
    if (a.page_size == 0) {
        c1 = key;
        c3 = r;
    } else {
        c1 = key % a.page_size;
        c3 = a.block_table[(long long)r * a.pages_per_req + key / a.page_size];
    }
}

// dlo += lo(a) * lo(b) and dhi += hi(a) * hi(b) for two packed bf16 pairs, in
// fp32: the mixed-precision FMA takes the bf16 halves directly (bf16 -> fp32
// is exact, so this equals fmaf on the widened values) with no unpacking.
__device__ __forceinline__ void fma_bf16x2(float &dlo, float &dhi, uint32_t a, uint32_t b) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
        : "+f"(dlo), "+f"(dhi)
        : "r"(a), "r"(b));
}

}  // namespace tc

// Host: the driver's tensor-map encoder (resolved at run time, so the library
// loads without a driver) and a 4-D tiled map with 128-byte swizzle (bf16
// unless another element type is given).
bool encode_4d(CUtensorMap *m, const void *base, const uint64_t dims[4], const uint64_t strides_bytes[3],
               const uint32_t box[4], CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

}  // namespace gr
