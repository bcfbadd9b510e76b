// gr_reorder.cu -- BeamKV maintenance between decode steps: the append of
// each step's new K/V, and the per-beam cache reordered so that every beam's
// chain is contiguous (xGR review, "xAttention": the unshared cache is rearranged in
// place after each beam selection, an alternative to following BeamPath
// indirections; the review's update formula is garbled, so this takes the
// plain reading, out of place):
//
//   out_k/out_v[r, t, b] = beam_k/beam_v[r, t, a_t(b)]   for t = 0..s, b < W_s
//   out_path[r, t, b]    = b                              (t >= 1; 0 at t = 0)
//
// with a_s = b, a_{t-1} = BeamPath[r, t, a_t].  Decode attention over the
// reordered cache with the identity path (and every level W_s wide) gives
// the same rows as over the original cache with BeamPath.  A broken chain
// (a parent outside [0, W_{t-1})) is not followed: the levels below the break
// are not written, and the device error word is set.
#include <cstdint>

#include "gr_common.cuh"
#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kReorderThreads = 128;
constexpr int kInplaceThreads = 256;
constexpr int kAppendThreads = 256;
constexpr size_t kInplaceSmemTarget = 100 * 1024;   // two CTAs per SM
constexpr size_t kInplaceSmemMax = 220 * 1024;

// One CTA per (request, beam): walk the chain, then copy each level's K and V
// rows (Hkv * D contiguous bf16 each) with 16-byte loads and stores.
__global__ void __launch_bounds__(kReorderThreads) reorder_kernel(Geometry g, const uint16_t *beam_k,
                                                                  const uint16_t *beam_v, const int32_t *beam_path,
                                                                  uint16_t *out_k, uint16_t *out_v, int32_t *out_path,
                                                                  int *err) {
    const int r = blockIdx.y, b = blockIdx.x;
    if (b >= g.W_s) return;
    const long long row_elems = (long long)g.Hkv * g.D;   // one (r, t, slot) row
    int slot = b;
    for (int t = g.step; t >= 0; --t) {
        const long long src = (((long long)r * g.S_max + t) * g.W_max + slot) * row_elems;
        const long long dst = (((long long)r * g.S_max + t) * g.W_max + b) * row_elems;
        const uint4 *sk = reinterpret_cast<const uint4 *>(beam_k + src), *sv = reinterpret_cast<const uint4 *>(beam_v + src);
        uint4 *dk = reinterpret_cast<uint4 *>(out_k + dst), *dv = reinterpret_cast<uint4 *>(out_v + dst);
        for (int i = threadIdx.x; i < row_elems / 8; i += blockDim.x) {
            dk[i] = __ldg(sk + i);
            dv[i] = __ldg(sv + i);
        }
        if (threadIdx.x == 0) out_path[((long long)r * g.S_max + t) * g.W_max + b] = t > 0 ? b : 0;
        if (t == 0) break;
        const int par = __ldg(beam_path + ((long long)r * g.S_max + t) * g.W_max + slot);
        if (par < 0 || par >= g.widths[t - 1]) {
            if (threadIdx.x == 0) raise_device_error(err, kDevErrBadParent);
            return;
        }
        slot = par;
    }
}

// In place.  One CTA owns one column tile of one (request, level, tensor):
// the same 16-byte chunks of every slot's row at that level.  It stages the
// level's source rows (slots below W_t, the only ones a parent can name) in
// shared memory, waits for the whole CTA, and writes each beam's row from
// its ancestor's copy, so no other CTA touches these bytes and nothing is
// read after it is overwritten.  Rows whose ancestor is their own slot are
// not rewritten; a broken chain leaves the beam's rows below the break as
// they were.  Level `step` maps every slot to itself and has no CTA.
__global__ void __launch_bounds__(kInplaceThreads) reorder_inplace_kernel(Geometry g, uint16_t *beam_k,
                                                                          uint16_t *beam_v,
                                                                          const int32_t *beam_path,
                                                                          int tile_chunks, int *err) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int r = blockIdx.y / g.step, t = blockIdx.y % g.step;
    const int row_chunks = g.Hkv * g.D / 8;   // 16-byte chunks in one (r, t, slot) row
    const int c0 = blockIdx.x * tile_chunks;
    const int nc = min(tile_chunks, row_chunks - c0);
    const int W_t = g.widths[t], W_s = g.W_s;
    uint4 *stage = reinterpret_cast<uint4 *>(smem_raw);
    int *anc = reinterpret_cast<int *>(stage + (size_t)W_t * tile_chunks);

    for (int b = threadIdx.x; b < W_s; b += blockDim.x) {
        int slot = b;
        for (int u = g.step; u > t; --u) {
            const int par = __ldg(beam_path + ((long long)r * g.S_max + u) * g.W_max + slot);
            if (par < 0 || par >= g.widths[u - 1]) {
                slot = -1;
                break;
            }
            slot = par;
        }
        anc[b] = slot;
        if (slot < 0 && blockIdx.x == 0 && blockIdx.z == 0) raise_device_error(err, kDevErrBadParent);
    }
    uint4 *level = reinterpret_cast<uint4 *>((blockIdx.z ? beam_v : beam_k) +
                                             ((long long)r * g.S_max + t) * g.W_max * (long long)g.Hkv * g.D) + c0;
    for (int i = threadIdx.x; i < W_t * nc; i += blockDim.x) {
        const int row = i / nc, c = i - row * nc;
        stage[row * tile_chunks + c] = level[(long long)row * row_chunks + c];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < W_s * nc; i += blockDim.x) {
        const int b = i / nc, c = i - b * nc;
        const int a = anc[b];
        if (a >= 0 && a != b) level[(long long)b * row_chunks + c] = stage[a * tile_chunks + c];
    }
}

// The identity path after an in-place reorder: beam_path[r, t, b] = b for
// t = 1..step, b < W_s.  Runs after reorder_inplace_kernel (stream order), the
// last reader of the old path.
__global__ void identity_path_kernel(Geometry g, int32_t *beam_path) {
    const int r = blockIdx.y / g.step, t = 1 + blockIdx.y % g.step;
    int32_t *row = beam_path + ((long long)r * g.S_max + t) * g.W_max;
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < g.W_s; b += gridDim.x * blockDim.x) row[b] = b;
}

// BeamKV append: row (r, b) of the new K and V (Hkv * D bf16, rows src_stride
// elements apart) goes to slot b of request r's step plane.  One thread per
// 16-byte chunk, grid-stride.
__global__ void __launch_bounds__(kAppendThreads) append_kernel(int R, int W_s, int S_max, int W_max, int row_chunks,
                                                                int step, const uint16_t *k_new,
                                                                const uint16_t *v_new, long long src_stride,
                                                                uint16_t *beam_k, uint16_t *beam_v) {
    const long long total = (long long)R * W_s * row_chunks;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / row_chunks;
        const int c = (int)(i - row * row_chunks);
        const int r = (int)(row / W_s), b = (int)(row - (long long)r * W_s);
        const long long src = row * src_stride + c * 8;
        const long long dst = (((long long)r * S_max + step) * W_max + b) * row_chunks * 8 + c * 8;
        const uint4 kk = __ldcs(reinterpret_cast<const uint4 *>(k_new + src));
        const uint4 vv = __ldcs(reinterpret_cast<const uint4 *>(v_new + src));
        *reinterpret_cast<uint4 *>(beam_k + dst) = kk;
        *reinterpret_cast<uint4 *>(beam_v + dst) = vv;
    }
}

}  // namespace

// Column-tile width (16-byte chunks per row) of the in-place reorder: the
// widest power of two up to 8 whose staging (every source slot of the widest
// level) plus the ancestor table fits kInplaceSmemTarget, so that two CTAs
// share an SM; down to one chunk within the opt-in limit.  0: too wide.
int inplace_tile_chunks(const Geometry &g, size_t *smem_bytes) {
    int w_src = 1;
    for (int t = 0; t < g.step; ++t) w_src = g.widths[t] > w_src ? g.widths[t] : w_src;
    const int row_chunks = g.Hkv * g.D / 8;
    for (int tc = 8; tc >= 1; tc /= 2) {
        const size_t bytes = (size_t)w_src * tc * 16 + (size_t)g.W_s * 4;
        if (tc > row_chunks) continue;
        if (bytes <= kInplaceSmemTarget || (tc == 1 && bytes <= kInplaceSmemMax)) {
            *smem_bytes = bytes;
            return tc;
        }
    }
    return 0;
}

cudaError_t launch_reorder_inplace(const Geometry &g, uint16_t *beam_k, uint16_t *beam_v, int32_t *beam_path,
                                   int *err, cudaStream_t s) {
    if (g.step == 0) return cudaSuccess;   // one level, already in place; the path has no entry to set
    size_t smem = 0;
    const int tc = inplace_tile_chunks(g, &smem);
    if (tc == 0) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(reorder_inplace_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int row_chunks = g.Hkv * g.D / 8;
    dim3 grid((row_chunks + tc - 1) / tc, g.R * g.step, 2);
    reorder_inplace_kernel<<<grid, kInplaceThreads, smem, s>>>(g, beam_k, beam_v, beam_path, tc, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 pgrid((g.W_s + 255) / 256, g.R * g.step);
    identity_path_kernel<<<pgrid, 256, 0, s>>>(g, beam_path);
    return cudaGetLastError();
}

cudaError_t launch_append(int R, int W_s, int S_max, int W_max, int Hkv, int D, int step, const uint16_t *k_new,
                          const uint16_t *v_new, long long src_stride, uint16_t *beam_k, uint16_t *beam_v,
                          int sm_count, cudaStream_t s) {
    const int row_chunks = Hkv * D / 8;
    const long long total = (long long)R * W_s * row_chunks;
    const long long want = (total + kAppendThreads - 1) / kAppendThreads;
    const long long cap = (long long)sm_count * 8;
    const int blocks = (int)(want < cap ? want : cap);
    append_kernel<<<blocks, kAppendThreads, 0, s>>>(R, W_s, S_max, W_max, row_chunks, step, k_new, v_new, src_stride,
                                                    beam_k, beam_v);
    return cudaGetLastError();
}

cudaError_t launch_reorder(const Geometry &g, const uint16_t *beam_k, const uint16_t *beam_v,
                           const int32_t *beam_path, uint16_t *out_k, uint16_t *out_v, int32_t *out_path, int *err,
                           cudaStream_t s) {
    dim3 grid(g.W_s, g.R);
    reorder_kernel<<<grid, kReorderThreads, 0, s>>>(g, beam_k, beam_v, beam_path, out_k, out_v, out_path, err);
    return cudaGetLastError();
}

}  // namespace gr
