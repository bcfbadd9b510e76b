// gr_beam_merge.cu -- the per-beam (unshared) stage, the log-sum-exp merge,
// and the BeamPath utilities, on CUDA cores.
//
// Per-beam stage: every (request, beam, query head) row attends to its own
// s+1 decoded tokens, found by following BeamPath parent slots back to step 0
// (GR-Inference blog, "kernel design": BeamKV is read on CUDA cores along
// BeamPath).  Merge: the context-stage partials (one per key split) and the
// per-beam partial are combined exactly by log-sum-exp (GR-Inference blog,
// "kernel design"; xGR review, "xAttention", merging stage).
#include <cmath>

#include "gr_common.cuh"

namespace gr {

namespace {

constexpr int kMergeWarps = 8;

// One warp per (request r, beam b, kv head g); it serves the G query heads of
// the group, which share the chain's K/V.  Lane l holds elements
// [l*V, l*V + V) of a D-vector (V = D/32), so every vector access of the warp
// covers D contiguous elements.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) beam_merge_kernel(const MergeArgs a) {
    constexpr int V = D / 32;
    const Geometry &g = a.g;
    __shared__ int s_chain[kMergeWarps][kMaxSteps];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * kMergeWarps + warp;
    if (item >= (long long)g.R * g.W_s * g.Hkv) return;
    const int kvh = (int)(item % g.Hkv);
    const long long rb = item / g.Hkv;
    const int b = (int)(rb % g.W_s);
    const int r = (int)(rb / g.W_s);
    if (b >= width_of(g, r, g.step)) return;   // a row past its request's width (per-request widths)

    // ancestor walk: a_s = b, a_{t-1} = BeamPath[r, t, a_t]
    int ok = 1;
    if (lane == 0) {
        int slot = b;
        s_chain[warp][g.step] = slot;
        for (int t = g.step; t >= 1; --t) {
            const int p = __ldg(a.beam_path + ((long long)r * g.S_max + t) * g.W_max + slot);
            if (p < 0 || p >= width_of(g, r, t - 1)) { ok = 0; break; }
            slot = p;
            s_chain[warp][t - 1] = slot;
        }
    }
    ok = __shfl_sync(kFullMask, ok, 0);
    __syncwarp();

    const long long n_rows = (long long)g.R * g.W_s * g.Hq;
    for (int jj = 0; jj < g.G; ++jj) {
        const int h = kvh * g.G + jj;
        const long long row = ((long long)r * g.W_s + b) * g.Hq + h;
        float o[V];
        if (!ok) {
            // broken precondition: no out-of-range read, NaN marks the row
#pragma unroll
            for (int i = 0; i < V; ++i) o[i] = __int_as_float(0x7fc00000);
            store_bf16<V>(a.out + row * D + lane * V, o);
            if (lane == 0) a.lse[row] = __int_as_float(0x7fc00000);
            continue;
        }
        float qf[V];
        load_bf16<V>(a.q + row * D + lane * V, qf);

        // per-beam partial, online softmax in base-2 units
        float m = -INFINITY, l = 0.f, acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        for (int t = 0; t <= g.step; ++t) {
            const long long kv =
                ((((long long)r * g.S_max + t) * g.W_max + s_chain[warp][t]) * g.Hkv + kvh) * D + lane * V;
            float kf[V], vf[V];
            load_bf16<V>(a.beam_k + kv, kf);
            load_bf16<V>(a.beam_v + kv, vf);
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) d = fmaf(qf[i], kf[i], d);
            const float x = warp_sum(d) * g.scale_log2;
            const float m_new = fmaxf(m, x);
            const float c = exp2f(m - m_new);
            const float p = exp2f(x - m_new);
            l = l * c + p;
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = fmaf(p, vf[i], acc[i] * c);
            m = m_new;
        }
        // the beam partial always holds >= 1 token, so l >= 1
        const float lse_beam = m + log2f(l);
        float top = lse_beam;
        for (int sp = 0; sp < a.n_splits; ++sp)
            top = fmaxf(top, __ldg(a.part_lse + sp * n_rows + row) * kLog2e);
        float wsum = exp2f(lse_beam - top);
        const float wb = wsum / l;
#pragma unroll
        for (int i = 0; i < V; ++i) o[i] = acc[i] * wb;
        for (int sp = 0; sp < a.n_splits; ++sp) {
            const float li = __ldg(a.part_lse + sp * n_rows + row) * kLog2e;
            const float wi = exp2f(li - top);   // empty split: lse = -inf -> 0
            float po[V];
            load_f32<V>(a.part_o + (sp * n_rows + row) * D + lane * V, po);
#pragma unroll
            for (int i = 0; i < V; ++i) o[i] = fmaf(wi, po[i], o[i]);
            wsum += wi;
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int i = 0; i < V; ++i) o[i] *= inv;
        store_bf16<V>(a.out + row * D + lane * V, o);
        if (lane == 0) a.lse[row] = (top + log2f(wsum)) * kLn2;
    }
    if (!ok && lane == 0) raise_device_error(a.err, kDevErrBadParent);
}

__global__ void ancestors_kernel(const Geometry g, const int32_t *__restrict__ beam_path,
                                 int32_t *__restrict__ anc) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)g.R * g.W_s) return;
    const int b = (int)(i % g.W_s), r = (int)(i / g.W_s);
    int32_t *row = anc + i * (g.step + 1);
    int slot = b;
    row[g.step] = slot;
    int t = g.step;
    for (; t >= 1; --t) {
        const int p = __ldg(beam_path + ((long long)r * g.S_max + t) * g.W_max + slot);
        if (p < 0 || p >= g.widths[t - 1]) break;
        slot = p;
        row[t - 1] = slot;
    }
    // a parent out of range: this step and every earlier one are unknown
    for (int u = t - 1; u >= 0; --u) row[u] = -1;
}

__global__ void validate_kernel(const Geometry g, const int32_t *__restrict__ beam_path,
                                const int32_t *__restrict__ ctx_len, int32_t *bad_count) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long n_path = (long long)g.R * g.step * g.W_max;
    int bad = 0;
    if (i < n_path) {
        const int b = (int)(i % g.W_max);
        const long long rt = i / g.W_max;
        const int t = 1 + (int)(rt % g.step);
        const int r = (int)(rt / g.step);
        if (b < g.widths[t]) {
            const int p = beam_path[((long long)r * g.S_max + t) * g.W_max + b];
            bad = (p < 0 || p >= g.widths[t - 1]);
        }
    } else if (i < n_path + g.R) {
        const int c = ctx_len[i - n_path];
        bad = (c < 0 || c > g.Lc_max);
    }
    const unsigned vote = __ballot_sync(kFullMask, bad);
    if ((threadIdx.x & 31) == 0 && vote) atomicAdd(bad_count, __popc(vote));
}

}  // namespace

cudaError_t launch_beam_merge(const MergeArgs &a, cudaStream_t s) {
    const long long items = (long long)a.g.R * a.g.W_s * a.g.Hkv;
    const unsigned blocks = (unsigned)((items + kMergeWarps - 1) / kMergeWarps);
    if (a.g.D == 128)
        beam_merge_kernel<128><<<blocks, kMergeWarps * 32, 0, s>>>(a);
    else
        beam_merge_kernel<64><<<blocks, kMergeWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ancestors(const Geometry &g, const int32_t *beam_path, int32_t *anc,
                             cudaStream_t s) {
    const long long n = (long long)g.R * g.W_s;
    ancestors_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(g, beam_path, anc);
    return cudaGetLastError();
}

cudaError_t launch_validate(const Geometry &g, const int32_t *beam_path, const int32_t *ctx_len,
                            int32_t *bad_count, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(bad_count, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    const long long n = (long long)g.R * g.step * g.W_max + g.R;
    validate_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(g, beam_path, ctx_len, bad_count);
    return cudaGetLastError();
}

}  // namespace gr
