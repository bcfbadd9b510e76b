// gr_ctx_simt.cu -- shared (context) stage on CUDA cores.
//
// The straightforward form of the shared stage: each CTA stages a block of
// the request's ContextKV in shared memory once and serves 16 query rows of
// the same (request, kv head) from it, with an online softmax over the key
// blocks (xGR review, "xAttention": online softmax, FlashAttention-style
// blocking).  It writes one normalised partial (output, LSE) per key split.
// It is the simple cross-check of the tensor-core kernel (gr_ctx_tc.cu) and
// is selected only when GR_ATTN_FORCE_PATH=simt.
#include <cmath>

#include "gr_common.cuh"

namespace gr {

namespace {

constexpr int kKeys = 32;        // keys per shared-memory block
constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 4;
constexpr int kRows = kWarps * kRowsPerWarp;

template <int D>
__global__ void __launch_bounds__(kWarps * 32) ctx_simt_kernel(const CtxArgs a) {
    constexpr int V = D / 32;
    constexpr int PAD = D + 8;   // row stride in bf16 elements: 16-byte lane reads hit distinct banks
    __shared__ __align__(16) uint16_t sk[kKeys * PAD];
    __shared__ __align__(16) uint16_t sv[kKeys * PAD];
    __shared__ float sq[kRows][D];

    const Geometry &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kvh = blockIdx.y % g.Hkv, r = blockIdx.y / g.Hkv, sp = blockIdx.z;
    const int M = g.W_s * g.G;                // rows of this (request, kv head)
    const int m0 = blockIdx.x * kRows;
    const long long n_rows = (long long)g.R * g.W_s * g.Hq;

    // query rows, pre-scaled into base-2 score units
    for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
        const int rr = idx / D, d = idx % D, m = m0 + rr;
        float v = 0.f;
        if (m < M) {
            const int b = m / g.G, h = kvh * g.G + m % g.G;
            v = bf16_bits_to_float(a.q[(((long long)r * g.W_s + b) * g.Hq + h) * D + d]) * g.scale_log2;
        }
        sq[rr][d] = v;
    }

    int len = a.ctx_len[r];
    len = len < 0 ? 0 : (len > g.Lc_max ? g.Lc_max : len);
    const int lo = sp * a.sp.split_len;
    const int hi = min(lo + a.sp.split_len, len);
    const uint16_t *kbase = a.ctx_k + ((long long)r * g.Hkv + kvh) * g.Lc_max * D;
    const uint16_t *vbase = a.ctx_v + ((long long)r * g.Hkv + kvh) * g.Lc_max * D;

    float m_run[kRowsPerWarp], l_run[kRowsPerWarp], acc[kRowsPerWarp][V];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        m_run[i] = -INFINITY; l_run[i] = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[i][v] = 0.f;
    }

    for (int k0 = lo; k0 < hi; k0 += kKeys) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kKeys * D / 8; idx += blockDim.x) {
            const int kr = idx / (D / 8), c = idx % (D / 8);
            uint4 kk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
            if (k0 + kr < hi) {   // positions past the context are never read
                kk = __ldg(reinterpret_cast<const uint4 *>(kbase + (long long)(k0 + kr) * D) + c);
                vv = __ldg(reinterpret_cast<const uint4 *>(vbase + (long long)(k0 + kr) * D) + c);
            }
            *reinterpret_cast<uint4 *>(&sk[kr * PAD + c * 8]) = kk;
            *reinterpret_cast<uint4 *>(&sv[kr * PAD + c * 8]) = vv;
        }
        __syncthreads();
        const bool valid = (k0 + lane) < hi;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int rr = warp * kRowsPerWarp + i;
            float x = 0.f;
#pragma unroll 4
            for (int d = 0; d < D; d += 8) {
                float kf[8];
                const uint4 u = *reinterpret_cast<const uint4 *>(&sk[lane * PAD + d]);
                kf[0] = __uint_as_float(u.x << 16); kf[1] = __uint_as_float(u.x & 0xffff0000u);
                kf[2] = __uint_as_float(u.y << 16); kf[3] = __uint_as_float(u.y & 0xffff0000u);
                kf[4] = __uint_as_float(u.z << 16); kf[5] = __uint_as_float(u.z & 0xffff0000u);
                kf[6] = __uint_as_float(u.w << 16); kf[7] = __uint_as_float(u.w & 0xffff0000u);
#pragma unroll
                for (int e = 0; e < 8; ++e) x = fmaf(sq[rr][d + e], kf[e], x);
            }
            x = valid ? x : -INFINITY;
            const float m_new = fmaxf(m_run[i], warp_max(x));   // lane 0 is always valid
            const float c = exp2f(m_run[i] - m_new);
            const float p = exp2f(x - m_new);
            l_run[i] = l_run[i] * c + warp_sum(p);
#pragma unroll
            for (int v = 0; v < V; ++v) acc[i][v] *= c;
            for (int j = 0; j < kKeys; ++j) {
                const float pj = __shfl_sync(kFullMask, p, j);
                const uint16_t *vr = &sv[j * PAD + lane * V];
#pragma unroll
                for (int v = 0; v < V; ++v) acc[i][v] = fmaf(pj, bf16_bits_to_float(vr[v]), acc[i][v]);
            }
            m_run[i] = m_new;
        }
    }

#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int m = m0 + warp * kRowsPerWarp + i;
        if (m >= M) continue;
        const int b = m / g.G, h = kvh * g.G + m % g.G;
        const long long row = ((long long)r * g.W_s + b) * g.Hq + h;
        float o[V];
        const bool any = l_run[i] > 0.f;
        const float inv = any ? 1.f / l_run[i] : 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) o[v] = acc[i][v] * inv;
        store_f32<V>(a.part_o + ((long long)sp * n_rows + row) * D + lane * V, o);
        if (lane == 0)
            a.part_lse[(long long)sp * n_rows + row] = any ? (m_run[i] + log2f(l_run[i])) * kLn2 : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_ctx_simt(const CtxArgs &a, cudaStream_t s) {
    const int M = a.g.W_s * a.g.G;
    dim3 grid((M + kRows - 1) / kRows, a.g.R * a.g.Hkv, a.sp.n_splits);
    if (a.g.D == 128)
        ctx_simt_kernel<128><<<grid, kWarps * 32, 0, s>>>(a);
    else
        ctx_simt_kernel<64><<<grid, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gr
