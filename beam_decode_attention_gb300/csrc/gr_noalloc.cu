// gr_noalloc.cu -- gr_decode_attn_noalloc: the decode attention for callers
// that cannot allocate device memory.
//
// gr_decode_attn asks its caller for a device workspace, where the
// context-stage kernel keeps its per-split partial results (an fp32 output
// and a log-sum-exp per row and split) until the merge kernel combines them.
// Some callers have no way to provide one: code that runs where CUDA API
// calls that allocate are not allowed (a host callback enqueued on a
// stream), code inside an engine whose memory pool has already reserved the
// device memory (an extra cudaMalloc fails or breaks its accounting), and
// latency-critical paths that cannot pay for cudaMalloc's implicit device
// synchronisation.  For them this file keeps that scratch in a fixed-size
// array in the library's own device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// this library holds GR_NOALLOC_SCRATCH_BYTES of device memory for it until
// the process exits.  Host code cannot use the array's name as a device
// address (on the host it names a stand-in object), so the first call on
// each device looks the address up with cudaGetSymbolAddress while that
// device is current, and later calls reuse it.
#include <mutex>

#include "gr_attn.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[GR_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up runs
// once per device).  Returns GR_ERR_CUDA if the lookup fails.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GR_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GR_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GR_OK;
}

}  // namespace

extern "C" int gr_decode_attn_noalloc(const gr_attn_shape *shape, const void *q, const void *ctx_k,
                                      const void *ctx_v, const int32_t *ctx_len, const void *beam_k,
                                      const void *beam_v, const int32_t *beam_path,
                                      const int32_t *widths, int32_t step, void *out, float *lse,
                                      gr_stream_t stream) {
    if (!shape || !widths) return GR_ERR_NULL_ARG;
    // The plan for this call decides how much scratch it needs; a call that
    // needs more than the static array holds is refused before anything is
    // enqueued.  A bad shape makes the size query return 0, and
    // gr_decode_attn below reports the precise error.
    const size_t need = gr_decode_attn_workspace_size(shape, widths, step);
    if (need > (size_t)GR_NOALLOC_SCRATCH_BYTES) return GR_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != GR_OK) return rc;
    // Every entry of the scratch that the kernels read is written earlier in
    // the same call, so the previous call's leftovers need no clearing.
    return gr_decode_attn(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step,
                          out, lse, scratch, GR_NOALLOC_SCRATCH_BYTES, stream);
}
