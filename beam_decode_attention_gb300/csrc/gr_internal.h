// gr_internal.h -- launch parameters shared by the host front end and the
// kernels of libgrattn.so (not installed; the public ABI is include/gr_attn.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gr_attn.h"

namespace gr {

// Decode steps a call may name (widths travel to the kernels by value).
constexpr int kMaxSteps = 64;

// Bounded waits: a kernel that polls an mbarrier more often than this sets
// the device error word and returns instead of hanging the GPU.
constexpr long long kSpinLimit = 1LL << 25;

// Device error codes written to the error word (first writer wins).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrBadParent = 2;

// Geometry of one call, resolved on the host.
struct Geometry {
    int R, Hq, Hkv, G, D;
    int Lc_max, S_max, W_max;
    int step, W_s;
    float scale;        // softmax scale applied to q.k (natural-log units)
    float scale_log2;   // softmax scale * log2(e)
    int widths[kMaxSteps];   // per step; with per-request widths, the largest over requests
    // per-request widths (device int32 [R, S_max]; null: every request has
    // widths[t]): rows b >= width(r, step) are not computed, and parents are
    // checked against width(r, t - 1)
    const int32_t *req_widths;
};

// the active width of request r at step t
__host__ __device__ inline int width_of(const Geometry &g, int r, int t) {
    // a per-request width never exceeds the step's padded width, so a device
    // copy that disagrees with the host's cannot index past the tensors
    if (!g.req_widths) return g.widths[t];
    const int w = g.req_widths[(long long)r * g.S_max + t];
    return w < g.widths[t] ? w : g.widths[t];
}

// Context-stage split of the key axis: split sp covers context positions
// [sp * split_len, (sp + 1) * split_len) clipped to ctx_len[r].
struct SplitPlan {
    int n_splits;   // >= 1 when Lc_max > 0, 0 when there is no context
    int split_len;  // multiple of the key-block size
    int persistent; // 1: one split on the persistent kernel (gr_ctx_pk.cu)
};

struct CtxArgs {
    Geometry g;
    SplitPlan sp;
    const uint16_t *q, *ctx_k, *ctx_v;
    const int32_t *ctx_len;
    float *part_o;    // fp32 [n_splits, R, W_s, Hq, D]  partial output, normalised
    float *part_lse;  // fp32 [n_splits, R, W_s, Hq]     partial LSE (natural log)
    int *err;
    // fused epilogue (one key split): the kernel also runs the per-beam
    // stage and the merge, and writes the final rows
    int fused;
    // split merge in the kernel (several key splits, chain short enough for
    // the fused epilogue): split 0 also runs the per-beam stage and folds the
    // chain into its partial; every split writes its partial and arrives on
    // its (request, kv head, tile pair) counter, and the last to arrive
    // merges the partials into the final rows.  The counters are zero when
    // the kernel starts.
    int split_merge;
    int *counters;    // int32 [R * Hkv * pairs]
    const uint16_t *beam_k, *beam_v;
    const int32_t *beam_path;
    uint16_t *out;
    float *lse;
    // paged ContextKV (page_size 0: the dense [R, Hkv, Lc_max, D] layout):
    // position j of request r sits in page block_table[r * pages_per_req +
    // j / page_size] of a pool [num_pages, Hkv, page_size, D], at j % page_size
    const int32_t *block_table = nullptr;
    int page_size = 0, pages_per_req = 0, num_pages = 0;
};

struct MergeArgs {
    Geometry g;
    int n_splits;
    const uint16_t *q, *beam_k, *beam_v;
    const int32_t *beam_path;
    const float *part_o, *part_lse;
    uint16_t *out;
    float *lse;
    int *err;
};

// gr_host.cu: every host-side check gr_decode_attn makes except the
// workspace size, in the same order; on GR_OK *need is the workspace the
// call's plan uses
int decode_scratch_bytes(const gr_attn_shape *shape, const void *q, const void *ctx_k, const void *ctx_v,
                         const int32_t *ctx_len, const void *beam_k, const void *beam_v, const int32_t *beam_path,
                         const int32_t *widths, int32_t step, const void *out, const float *lse, size_t *need);

// gr_beam_merge.cu
cudaError_t launch_beam_merge(const MergeArgs &a, cudaStream_t s);
cudaError_t launch_ancestors(const Geometry &g, const int32_t *beam_path, int32_t *anc,
                             cudaStream_t s);
cudaError_t launch_validate(const Geometry &g, const int32_t *beam_path, const int32_t *ctx_len,
                            int32_t *bad_count, cudaStream_t s);

// gr_ctx_simt.cu  (CUDA-core context stage)
cudaError_t launch_ctx_simt(const CtxArgs &a, cudaStream_t s);

// gr_ctx_tc.cu  (tensor-core context stage)
int tc_beams_per_tile(int G);
int tc_fused_max_steps(int G);  // the fused epilogue holds chains of steps < this
int tc_merge_max_splits();      // the in-kernel split merge takes at most this many splits
cudaError_t launch_ctx_tc(const CtxArgs &a, int sm_count, cudaStream_t s);

// gr_ctx_pk.cu  (persistent tensor-core kernel: the whole call over 128-row tiles, one key split)
int pk_max_steps();   // chains of steps < this
cudaError_t launch_ctx_pk(const CtxArgs &a, int sm_count, cudaStream_t s);

// gr_reorder.cu  (BeamKV append; per-beam cache reordered along BeamPath)
cudaError_t launch_reorder(const Geometry &g, const uint16_t *beam_k, const uint16_t *beam_v,
                           const int32_t *beam_path, uint16_t *out_k, uint16_t *out_v, int32_t *out_path, int *err,
                           cudaStream_t s);
int inplace_tile_chunks(const Geometry &g, size_t *smem_bytes);   // 0: a level too wide to stage
cudaError_t launch_reorder_inplace(const Geometry &g, uint16_t *beam_k, uint16_t *beam_v, int32_t *beam_path,
                                   int *err, cudaStream_t s);
cudaError_t launch_append(int R, int W_s, int S_max, int W_max, int Hkv, int D, int step, const uint16_t *k_new,
                          const uint16_t *v_new, long long src_stride, uint16_t *beam_k, uint16_t *beam_v,
                          int sm_count, cudaStream_t s);

// gr_select.cu  (beam selection)
size_t select_list_bytes(int R, int W, int V, int next_width);
int select_max_width();
int select_max_beams();
size_t trie_select_bytes(int R, int W, int next_width);
cudaError_t launch_trie_select(int R, int W, int V, int next_width, int num_nodes, int num_edges,
                               const float *logits, const float *beam_scores, const int32_t *beam_node,
                               const int32_t *offsets, const int32_t *tokens, const int32_t *children,
                               int32_t *next_parent, long long parent_stride, int32_t *next_token,
                               float *next_score, int32_t *next_node, void *workspace, cudaStream_t s,
                               cudaEvent_t between = nullptr);
// `between` (may be null) is recorded on `s` between the two kernels
cudaError_t launch_beam_select(int R, int W, int V, int next_width, const float *logits,
                               const float *beam_scores, int32_t *next_parent, long long parent_stride,
                               int32_t *next_token, float *next_score, void *workspace, cudaStream_t s,
                               cudaEvent_t between = nullptr);

}  // namespace gr
