// gr_noalloc.cu -- gr_decode_attn_noalloc: the decode attention for callers
// that cannot allocate device memory.
//
// gr_decode_attn asks its caller for a device workspace, where the
// context-stage kernel keeps its per-split partial results (an fp32 output
// and a log-sum-exp per row and split) until the merge kernel combines them.
// Some callers have no way to provide one: code inside an engine whose
// memory pool has already reserved the device memory (an extra cudaMalloc
// fails or breaks its accounting), and latency-critical paths that cannot
// pay for cudaMalloc's implicit device synchronisation.  For them this file
// keeps that scratch in a fixed-size array in the library's own device
// memory.  (Code running inside a stream callback cannot use this entry
// point either: CUDA forbids every CUDA call there, launches included.)
//
// The array is a file-scope __device__ variable, so every GPU that loads
// this library holds GR_NOALLOC_SCRATCH_BYTES of device memory for it until
// the process exits.  Host code cannot use the array's name as a device
// address (on the host it names a stand-in object), so the first call on
// each device looks the address up with cudaGetSymbolAddress while that
// device is current, and later calls reuse it.
#include <mutex>

#include "gr_attn.h"
#include "gr_internal.h"

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
    // Every check gr_decode_attn makes, in its order (shapes, pointers,
    // alignment, the device), runs first, so both entry points report the
    // same error for the same arguments.  Then the plan's scratch need is
    // compared with the static array: a call that needs more is refused
    // before anything is enqueued.
    size_t need = 0;
    int rc = gr::decode_scratch_bytes(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step,
                                      out, lse, &need);
    if (rc != GR_OK) return rc;
    if (need > (size_t)GR_NOALLOC_SCRATCH_BYTES) return GR_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != GR_OK) return rc;
    // Every entry of the scratch that the kernels read is written earlier in
    // the same call, so the previous call's leftovers need no clearing.
    return gr_decode_attn(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step,
                          out, lse, scratch, GR_NOALLOC_SCRATCH_BYTES, stream);
}
