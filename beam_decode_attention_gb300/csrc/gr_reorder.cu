// gr_reorder.cu -- the per-beam cache reordered so that every beam's chain is
// contiguous (xGR review, "xAttention": the unshared cache is rearranged in
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

}  // namespace

cudaError_t launch_reorder(const Geometry &g, const uint16_t *beam_k, const uint16_t *beam_v,
                           const int32_t *beam_path, uint16_t *out_k, uint16_t *out_v, int32_t *out_path, int *err,
                           cudaStream_t s) {
    dim3 grid(g.W_s, g.R);
    reorder_kernel<<<grid, kReorderThreads, 0, s>>>(g, beam_k, beam_v, beam_path, out_k, out_v, out_path, err);
    return cudaGetLastError();
}

}  // namespace gr
