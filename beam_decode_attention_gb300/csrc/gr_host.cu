// gr_host.cu -- the C ABI of libgrattn.so (include/gr_attn.h): argument
// checks, the split planner, workspace carve-up and kernel launches.
//
// The call follows the three stages of the pages' decode attention: shared
// (context) stage, unshared (per-beam) stage, log-sum-exp merge (GR-Inference
// blog, "kernel design"; xGR review, "xAttention").
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gr_attn.h"
#include "gr_internal.h"

namespace gr {

// Device error word: kernels that give up a bounded wait, or meet a broken
// precondition, record a code here (see raise_device_error).
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    int *err_ptr = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device facts, looked up once with that device current.
int device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GR_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GR_ERR_CUDA;
        }
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
            cudaGetLastError();
            return GR_ERR_CUDA;
        }
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        d.err_ptr = static_cast<int *>(p);
        d.ready = true;
    }
    *out = d;
    return d.supported ? GR_OK : GR_ERR_UNSUPPORTED;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// true when the byte ranges [a, a + na) and [b, b + nb) share a byte
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

int make_geometry(const gr_attn_shape *s, const int32_t *widths, int32_t step, Geometry *g) {
    if (!s || !widths) return GR_ERR_NULL_ARG;
    if (s->num_requests < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->ctx_capacity < 0 ||
        s->step_capacity < 1 || s->beam_capacity < 1)
        return GR_ERR_BAD_SHAPE;
    if (s->num_q_heads % s->num_kv_heads != 0) return GR_ERR_BAD_SHAPE;
    if (s->head_dim != 64 && s->head_dim != 128) return GR_ERR_UNSUPPORTED;
    if (s->num_q_heads / s->num_kv_heads > 128) return GR_ERR_UNSUPPORTED;
    if (!(std::isfinite(s->softmax_scale)) || !(s->softmax_scale > 0.f)) return GR_ERR_BAD_SHAPE;
    if (step < 0 || step >= s->step_capacity) return GR_ERR_BAD_SHAPE;
    if (step >= kMaxSteps) return GR_ERR_UNSUPPORTED;
    std::memset(g, 0, sizeof *g);
    for (int t = 0; t <= step; ++t) {
        if (widths[t] < 1 || widths[t] > s->beam_capacity) return GR_ERR_BAD_SHAPE;
        g->widths[t] = widths[t];
    }
    g->R = s->num_requests;
    g->Hq = s->num_q_heads;
    g->Hkv = s->num_kv_heads;
    g->G = s->num_q_heads / s->num_kv_heads;
    g->D = s->head_dim;
    g->Lc_max = s->ctx_capacity;
    g->S_max = s->step_capacity;
    g->W_max = s->beam_capacity;
    g->step = step;
    g->W_s = widths[step];
    g->scale = s->softmax_scale;
    g->scale_log2 = s->softmax_scale * 1.4426950408889634f;
    // every index the kernels form must fit comfortably in 64-bit arithmetic
    // and every grid dimension in its hardware limit
    const double rows = (double)g->R * g->W_s * g->Hq;
    if (rows * g->D > 4.0e15 || (double)g->R * g->Hkv > 65535.0) return GR_ERR_BAD_SHAPE;
    return GR_OK;
}

enum class Path { kTensorCore, kSimt };

// GR_ATTN_FORCE_PATH=simt selects the CUDA-core context stage (a cross-check
// of the tensor-core kernels in tests); the tensor-core stage is the default.
Path chosen_path() {
    const char *e = std::getenv("GR_ATTN_FORCE_PATH");
    if (e && std::strcmp(e, "simt") == 0) return Path::kSimt;
    return Path::kTensorCore;
}

// GR_ATTN_FORCE_PATH=pair keeps single-split calls on the tile-pair kernel,
// GR_ATTN_FORCE_PATH=persistent puts them on the persistent one whatever the
// cost model says (tests compare the two).
bool pair_forced() {
    const char *e = std::getenv("GR_ATTN_FORCE_PATH");
    return e && std::strcmp(e, "pair") == 0;
}

bool persistent_forced() {
    const char *e = std::getenv("GR_ATTN_FORCE_PATH");
    return e && std::strcmp(e, "persistent") == 0;
}

int forced_splits() {
    const char *e = std::getenv("GR_ATTN_FORCE_SPLITS");
    if (!e) return 0;
    int v = std::atoi(e);
    return v > 0 ? v : 0;
}

// Split plan for the CUDA-core context stage.
SplitPlan plan_simt(const Geometry &g, int sm_count) {
    SplitPlan p{0, 0, 0};
    if (g.Lc_max == 0) return p;
    constexpr int kKeyBlock = 32;
    const int blocks = (g.Lc_max + kKeyBlock - 1) / kKeyBlock;
    const long long ctas = (long long)((g.W_s * g.G + 15) / 16) * g.R * g.Hkv;
    int n = forced_splits();
    if (n == 0) {
        const long long target = 4LL * sm_count;
        n = (int)std::min<long long>(blocks, std::max<long long>(1, (target + ctas - 1) / ctas));
    }
    n = std::min(n, blocks);
    const int per = (blocks + n - 1) / n;
    p.split_len = per * kKeyBlock;
    p.n_splits = (g.Lc_max + p.split_len - 1) / p.split_len;
    return p;
}

// Tile geometry of the tensor-core kernels: beams per 128-row tile, tiles
// per (request, kv head), and tile pairs (one tile-pair CTA per pair and split).
struct TcShape {
    int bpt, tiles, pairs;
};

TcShape tc_shape(const Geometry &g) {
    TcShape t;
    t.bpt = tc_beams_per_tile(g.G);
    t.tiles = (g.W_s + t.bpt - 1) / t.bpt;
    t.pairs = (t.tiles + 1) / 2;
    return t;
}

// Whether a call with this many key splits keeps the split merge in the
// context kernel (the chain must fit the fused epilogue's tables).
bool tc_split_merge(const Geometry &g, int n_splits) {
    return n_splits > 1 && n_splits <= tc_merge_max_splits() && g.step < tc_fused_max_steps(g.G);
}

// Whether a single-split call runs on the persistent kernel (chains short
// enough for its epilogue tables, not forced onto the tile-pair kernel).
bool tc_persistent(const Geometry &g, int n_splits) {
    return n_splits == 1 && g.step < pk_max_steps() && !pair_forced();
}

// Kernel and split count for the tensor-core context stage, from a cost
// model of one call (in microseconds, measured on GB300 with one CTA per
// SM).  The tile-pair kernel: a CTA costs kFixed (set-up, first S,
// epilogue) plus kPerBlock per 128-key block of its split, CTAs run in waves
// of sm_count, and several splits add the merge, kMergeIn (in the kernel
// while the chain fits its tables) or kMergeKernel (a second kernel).  The
// persistent kernel (one split, 128-row tiles) is a candidate while every
// tile has an SM of its own: one round of kPkFixed plus kPkPerBlock per
// block.  Past one round the tile-pair kernel measured faster (each 128-row
// tile then streams the whole context per block on its own SM, where a tile
// pair shares it).  Fewer splits win ties.
SplitPlan plan_tc(const Geometry &g, int sm_count) {
    SplitPlan p{0, 0, 0};
    if (g.Lc_max == 0) return p;
    constexpr int kKeyBlock = 128;
    constexpr double kFixed = 9.0, kPerBlock = 1.8, kMergeIn = 15.0, kMergeKernel = 17.0;
    constexpr double kPkFixed = 8.0, kPkPerBlock = 1.5;
    const int blocks = (g.Lc_max + kKeyBlock - 1) / kKeyBlock;
    const TcShape sh = tc_shape(g);
    const long long ctas = (long long)sh.pairs * g.R * g.Hkv;
    const long long items = (long long)sh.tiles * g.R * g.Hkv;
    const int sms = std::max(1, sm_count);
    int n = forced_splits();
    bool pk = false;
    if (n == 0 && persistent_forced() && tc_persistent(g, 1)) {
        n = 1;
        pk = true;
    } else if (n == 0) {
        double best = 0.0;
        for (int c = 1; c <= std::min(blocks, 32); ++c) {
            const int per = (blocks + c - 1) / c;
            const long long waves = (ctas * c + sms - 1) / sms;
            const double t = (double)waves * (kFixed + kPerBlock * per) +
                             (c > 1 ? (tc_split_merge(g, c) ? kMergeIn : kMergeKernel) : 0.0);
            if (c == 1 || t < best - 1e-9) {
                best = t;
                n = c;
            }
        }
        if (tc_persistent(g, 1) && items <= sms && kPkFixed + kPkPerBlock * blocks < best - 1e-9) {
            n = 1;
            pk = true;
        }
    } else if (n == 1 && tc_persistent(g, 1) && persistent_forced()) {
        pk = true;
    }
    n = std::min(n, blocks);
    const int per = (blocks + n - 1) / n;
    p.split_len = per * kKeyBlock;
    p.n_splits = (g.Lc_max + p.split_len - 1) / p.split_len;
    p.persistent = (pk && p.n_splits == 1) ? 1 : 0;
    return p;
}

SplitPlan plan(const Geometry &g, int sm_count) {
    return chosen_path() == Path::kSimt ? plan_simt(g, sm_count) : plan_tc(g, sm_count);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    size_t part_o, part_lse, counters, counter_bytes, total;
};

// With a single key split (and a chain short enough for the kernel's
// shared-memory scratch), the tensor-core kernel runs the per-beam stage and
// the merge itself: no partials, no workspace, one kernel.
bool fused_merge(const Geometry &g, const SplitPlan &p) {
    return chosen_path() == Path::kTensorCore && p.n_splits == 1 && g.step < tc_fused_max_steps(g.G);
}

// The planner's choice of the persistent kernel.
bool persistent(const Geometry &, const SplitPlan &p) {
    return chosen_path() == Path::kTensorCore && p.persistent != 0;
}

// With several key splits and such a chain, the split merge also stays in
// the context kernel: partials and arrival counters in the workspace, one
// kernel (plus the counters' reset).
bool split_merge(const Geometry &g, const SplitPlan &p) {
    return chosen_path() == Path::kTensorCore && tc_split_merge(g, p.n_splits);
}

long long context_ctas(const Geometry &g, const SplitPlan &sp, int sm_count) {
    if (sp.n_splits == 0) return 0;
    if (chosen_path() == Path::kSimt) return (long long)((g.W_s * g.G + 15) / 16) * g.R * g.Hkv * sp.n_splits;
    if (persistent(g, sp)) return std::min<long long>((long long)tc_shape(g).tiles * g.R * g.Hkv, (long long)sm_count);
    return (long long)tc_shape(g).pairs * g.R * g.Hkv * sp.n_splits;
}

Layout workspace_layout(const Geometry &g, const SplitPlan &p) {
    Layout l{0, 0, 0, 0, 0};
    if (fused_merge(g, p)) return l;
    const size_t rows = (size_t)g.R * g.W_s * g.Hq;
    const size_t o_bytes = (size_t)p.n_splits * rows * g.D * sizeof(float);
    const size_t lse_bytes = (size_t)p.n_splits * rows * sizeof(float);
    l.part_o = 0;
    l.part_lse = align256(o_bytes);
    l.counters = align256(l.part_lse + lse_bytes);
    l.counter_bytes = split_merge(g, p) ? (size_t)tc_shape(g).pairs * g.R * g.Hkv * sizeof(int) : 0;
    l.total = p.n_splits ? align256(l.counters + l.counter_bytes) : 0;
    return l;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GR_OK;
    cudaGetLastError();
    return GR_ERR_CUDA;
}

}  // namespace
}  // namespace gr

using namespace gr;

extern "C" {

int gr_version(void) { return 100; }

const char *gr_status_string(int status) {
    switch (status) {
        case GR_OK: return "ok";
        case GR_ERR_NULL_ARG: return "a required pointer is NULL";
        case GR_ERR_BAD_SHAPE: return "inconsistent or out-of-range sizes";
        case GR_ERR_UNSUPPORTED: return "unsupported head_dim, head grouping or device";
        case GR_ERR_MISALIGNED: return "a device pointer is not 16-byte aligned";
        case GR_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than gr_decode_attn_workspace_size()";
        case GR_ERR_CUDA: return "a CUDA call failed";
        case GR_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
        case GR_ERR_BAD_BEAM_PATH: return "a BeamPath parent slot was out of range";
        default: return "unknown status";
    }
}

size_t gr_decode_attn_workspace_size(const gr_attn_shape *shape, const int32_t *widths, int32_t step) {
    Geometry g;
    if (make_geometry(shape, widths, step, &g) != GR_OK) return 0;
    DeviceInfo dev;
    if (device_info(&dev) != GR_OK) return 0;
    return workspace_layout(g, plan(g, dev.sm_count)).total;
}

}  // extern "C"

namespace {

// Everything gr_decode_attn decides before it enqueues work: the geometry,
// the split plan, the workspace layout and the device facts.
struct DecodeCall {
    Geometry g;
    SplitPlan sp;
    Layout lay;
    DeviceInfo dev;
};

// Every host-side check of a decode call except the workspace size, in the
// order the entry points report them: shape and widths, paged and
// per-request-width descriptors, NULL pointers, alignment, then the device.
int prepare_decode(const gr_attn_shape *shape, const void *q, const void *ctx_k, const void *ctx_v,
                   const int32_t *ctx_len, const void *beam_k, const void *beam_v, const int32_t *beam_path,
                   const int32_t *widths, int32_t step, const void *out, const float *lse, const void *workspace,
                   const gr_ctx_pages *pages, const int32_t *block_table, const int32_t *req_widths,
                   DecodeCall *dc) {
    Geometry &g = dc->g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (req_widths) {
        if (misaligned(req_widths)) return GR_ERR_MISALIGNED;
        if (chosen_path() == Path::kSimt) return GR_ERR_UNSUPPORTED;   // the cross-check path: shared widths only
        g.req_widths = req_widths;
    }
    if (pages) {
        if (pages->page_size < 128 || pages->page_size % 128 != 0 || pages->num_pages < 1 ||
            pages->pages_per_request < 1 ||
            (long long)pages->pages_per_request * pages->page_size < (long long)g.Lc_max)
            return GR_ERR_BAD_SHAPE;
        if (!block_table) return GR_ERR_NULL_ARG;
        if (misaligned(block_table)) return GR_ERR_MISALIGNED;
        if (chosen_path() == Path::kSimt) return GR_ERR_UNSUPPORTED;   // the cross-check path reads dense only
    }
    if (!q || !ctx_len || !beam_k || !beam_v || !beam_path || !out || !lse) return GR_ERR_NULL_ARG;
    if (g.Lc_max > 0 && (!ctx_k || !ctx_v)) return GR_ERR_NULL_ARG;
    if (misaligned(q) || misaligned(ctx_k) || misaligned(ctx_v) || misaligned(ctx_len) ||
        misaligned(beam_k) || misaligned(beam_v) || misaligned(beam_path) || misaligned(out) ||
        misaligned(lse) || misaligned(workspace))
        return GR_ERR_MISALIGNED;
    rc = device_info(&dc->dev);
    if (rc != GR_OK) return rc;
    dc->sp = plan(g, dc->dev.sm_count);
    dc->lay = workspace_layout(g, dc->sp);
    return GR_OK;
}

int run_decode(const gr_attn_shape *shape, const void *q, const void *ctx_k, const void *ctx_v,
               const int32_t *ctx_len, const void *beam_k, const void *beam_v,
               const int32_t *beam_path, const int32_t *widths, int32_t step, void *out, float *lse,
               void *workspace, size_t workspace_bytes, gr_stream_t stream,
               gr_event_t const *events, const gr_ctx_pages *pages = nullptr,
               const int32_t *block_table = nullptr, const int32_t *req_widths = nullptr) {
    DecodeCall dc;
    int rc = prepare_decode(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step, out, lse,
                            workspace, pages, block_table, req_widths, &dc);
    if (rc != GR_OK) return rc;
    const Geometry &g = dc.g;
    const SplitPlan &sp = dc.sp;
    const Layout &lay = dc.lay;
    const DeviceInfo &dev = dc.dev;
    if (lay.total > 0 && (!workspace || workspace_bytes < lay.total)) return GR_ERR_WORKSPACE_TOO_SMALL;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto mark = [&](int i) -> int {
        if (!events || !events[i]) return GR_OK;
        return cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s));
    };
    char *ws = static_cast<char *>(workspace);
    float *part_o = sp.n_splits ? reinterpret_cast<float *>(ws + lay.part_o) : nullptr;
    float *part_lse = sp.n_splits ? reinterpret_cast<float *>(ws + lay.part_lse) : nullptr;

    if ((rc = mark(0)) != GR_OK) return rc;
    if (sp.n_splits > 0) {
        CtxArgs c;
        c.g = g;
        c.sp = sp;
        c.q = static_cast<const uint16_t *>(q);
        c.ctx_k = static_cast<const uint16_t *>(ctx_k);
        c.ctx_v = static_cast<const uint16_t *>(ctx_v);
        c.ctx_len = ctx_len;
        c.part_o = part_o;
        c.part_lse = part_lse;
        c.err = dev.err_ptr;
        c.fused = fused_merge(g, sp) ? 1 : 0;
        c.split_merge = split_merge(g, sp) ? 1 : 0;
        c.counters = c.split_merge ? reinterpret_cast<int *>(ws + lay.counters) : nullptr;
        c.beam_k = static_cast<const uint16_t *>(beam_k);
        c.beam_v = static_cast<const uint16_t *>(beam_v);
        c.beam_path = beam_path;
        c.out = static_cast<uint16_t *>(out);
        c.lse = lse;
        if (pages) {
            c.block_table = block_table;
            c.page_size = pages->page_size;
            c.pages_per_req = pages->pages_per_request;
            c.num_pages = pages->num_pages;
        }
        if (c.split_merge) {
            // the arrival counters start at zero in every call
            rc = cuda_status(cudaMemsetAsync(c.counters, 0, lay.counter_bytes, s));
            if (rc != GR_OK) return rc;
        }
        if (persistent(g, sp))
            rc = cuda_status(launch_ctx_pk(c, dev.sm_count, s));
        else
            rc = cuda_status(chosen_path() == Path::kSimt ? launch_ctx_simt(c, s) : launch_ctx_tc(c, dev.sm_count, s));
        if (rc != GR_OK) return rc;
    }
    if ((rc = mark(1)) != GR_OK) return rc;
    if (fused_merge(g, sp) || split_merge(g, sp)) return mark(2);
    MergeArgs m;
    m.g = g;
    m.n_splits = sp.n_splits;
    m.q = static_cast<const uint16_t *>(q);
    m.beam_k = static_cast<const uint16_t *>(beam_k);
    m.beam_v = static_cast<const uint16_t *>(beam_v);
    m.beam_path = beam_path;
    m.part_o = part_o;
    m.part_lse = part_lse;
    m.out = static_cast<uint16_t *>(out);
    m.lse = lse;
    m.err = dev.err_ptr;
    rc = cuda_status(launch_beam_merge(m, s));
    if (rc != GR_OK) return rc;
    return mark(2);
}

}  // namespace

namespace gr {

int decode_scratch_bytes(const gr_attn_shape *shape, const void *q, const void *ctx_k, const void *ctx_v,
                         const int32_t *ctx_len, const void *beam_k, const void *beam_v, const int32_t *beam_path,
                         const int32_t *widths, int32_t step, const void *out, const float *lse, size_t *need) {
    DecodeCall dc;
    const int rc = prepare_decode(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step, out,
                                  lse, nullptr, nullptr, nullptr, nullptr, &dc);
    if (rc == GR_OK) *need = dc.lay.total;
    return rc;
}

}  // namespace gr

extern "C" {

int gr_decode_attn(const gr_attn_shape *shape, const void *q, const void *ctx_k, const void *ctx_v,
                   const int32_t *ctx_len, const void *beam_k, const void *beam_v,
                   const int32_t *beam_path, const int32_t *widths, int32_t step, void *out,
                   float *lse, void *workspace, size_t workspace_bytes, gr_stream_t stream) {
    return run_decode(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step, out,
                      lse, workspace, workspace_bytes, stream, nullptr);
}

int gr_decode_attn_paged(const gr_attn_shape *shape, const gr_ctx_pages *pages, const void *q,
                         const void *ctx_k_pool, const void *ctx_v_pool, const int32_t *ctx_len,
                         const int32_t *block_table, const void *beam_k, const void *beam_v,
                         const int32_t *beam_path, const int32_t *widths, int32_t step, void *out,
                         float *lse, void *workspace, size_t workspace_bytes, gr_stream_t stream) {
    if (!pages) return GR_ERR_NULL_ARG;
    return run_decode(shape, q, ctx_k_pool, ctx_v_pool, ctx_len, beam_k, beam_v, beam_path, widths, step, out,
                      lse, workspace, workspace_bytes, stream, nullptr, pages, block_table);
}

int gr_decode_attn_ragged(const gr_attn_shape *shape, const void *q, const void *ctx_k, const void *ctx_v,
                          const int32_t *ctx_len, const void *beam_k, const void *beam_v,
                          const int32_t *beam_path, const int32_t *req_widths_host,
                          const int32_t *req_widths, int32_t step, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, gr_stream_t stream) {
    if (!shape || !req_widths_host || !req_widths) return GR_ERR_NULL_ARG;
    if (shape->num_requests < 1 || step < 0 || step >= shape->step_capacity || step >= kMaxSteps)
        return GR_ERR_BAD_SHAPE;
    // the layout (and the plan) takes each step's largest width
    int32_t wmax[kMaxSteps];
    for (int t = 0; t <= step; ++t) {
        wmax[t] = 0;
        for (int r = 0; r < shape->num_requests; ++r) {
            const int32_t w = req_widths_host[(long long)r * (step + 1) + t];
            if (w < 1 || w > shape->beam_capacity) return GR_ERR_BAD_SHAPE;
            wmax[t] = w > wmax[t] ? w : wmax[t];
        }
    }
    return run_decode(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, wmax, step, out, lse,
                      workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, req_widths);
}

int gr_decode_attn_timed(const gr_attn_shape *shape, const void *q, const void *ctx_k,
                         const void *ctx_v, const int32_t *ctx_len, const void *beam_k,
                         const void *beam_v, const int32_t *beam_path, const int32_t *widths,
                         int32_t step, void *out, float *lse, void *workspace,
                         size_t workspace_bytes, gr_stream_t stream, gr_event_t const *events) {
    if (!events || !events[0] || !events[2]) return GR_ERR_NULL_ARG;   // events[1] may be NULL
    return run_decode(shape, q, ctx_k, ctx_v, ctx_len, beam_k, beam_v, beam_path, widths, step, out,
                      lse, workspace, workspace_bytes, stream, events);
}

int gr_decode_attn_plan(const gr_attn_shape *shape, const int32_t *widths, int32_t step,
                        gr_plan_info *info) {
    Geometry g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (!info) return GR_ERR_NULL_ARG;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    const SplitPlan sp = plan(g, dev.sm_count);
    info->path = chosen_path() == Path::kSimt ? 1 : 0;
    info->n_splits = sp.n_splits;
    info->split_len = sp.split_len;
    info->context_ctas = (int32_t)context_ctas(g, sp, dev.sm_count);
    info->fused_merge = (fused_merge(g, sp) || split_merge(g, sp)) ? 1 : 0;
    info->kernels = (sp.n_splits && !info->fused_merge) ? 2 : 1;
    info->persistent = persistent(g, sp) ? 1 : 0;
    return GR_OK;
}

int gr_resolve_ancestors(const gr_attn_shape *shape, const int32_t *beam_path, const int32_t *widths,
                         int32_t step, int32_t *anc, gr_stream_t stream) {
    Geometry g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (!beam_path || !anc) return GR_ERR_NULL_ARG;
    if (misaligned(beam_path) || misaligned(anc)) return GR_ERR_MISALIGNED;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    return cuda_status(launch_ancestors(g, beam_path, anc, static_cast<cudaStream_t>(stream)));
}

int gr_validate_beam_path(const gr_attn_shape *shape, const int32_t *beam_path, const int32_t *widths,
                          int32_t step, const int32_t *ctx_len, int32_t *bad_count, gr_stream_t stream) {
    Geometry g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (!beam_path || !ctx_len || !bad_count) return GR_ERR_NULL_ARG;
    if (misaligned(beam_path) || misaligned(ctx_len)) return GR_ERR_MISALIGNED;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    return cuda_status(launch_validate(g, beam_path, ctx_len, bad_count, static_cast<cudaStream_t>(stream)));
}

size_t gr_beam_select_workspace_size(const gr_select_shape *shape) {
    if (!shape || shape->num_requests < 1 || shape->width < 1 || shape->vocab < 1 || shape->next_width < 1 ||
        shape->next_width > select_max_width() || shape->width > select_max_beams() ||
        (long long)shape->width * shape->vocab >= (1LL << 31) ||
        shape->next_width > (long long)shape->width * shape->vocab)
        return 0;
    return select_list_bytes(shape->num_requests, shape->width, shape->vocab, shape->next_width);
}

static int beam_select_impl(const gr_select_shape *shape, const float *logits, const float *beam_scores,
                            int32_t *next_parent, int64_t parent_stride, int32_t *next_token, float *next_score,
                            void *workspace, size_t workspace_bytes, gr_stream_t stream, gr_event_t const *events) {
    if (!shape || !logits || !beam_scores || !next_parent || !next_token || !next_score || !workspace)
        return GR_ERR_NULL_ARG;
    const size_t need = gr_beam_select_workspace_size(shape);
    if (need == 0 || parent_stride < shape->next_width) return GR_ERR_BAD_SHAPE;
    if (misaligned(logits) || misaligned(beam_scores) || misaligned(next_parent) || misaligned(next_token) ||
        misaligned(next_score) || misaligned(workspace))
        return GR_ERR_MISALIGNED;
    if (workspace_bytes < need) return GR_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (events) {
        if (!events[0] || !events[1] || !events[2]) return GR_ERR_NULL_ARG;
        const int e0 = cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(events[0]), s));
        if (e0 != GR_OK) return e0;
    }
    const int e1 = cuda_status(launch_beam_select(
        shape->num_requests, shape->width, shape->vocab, shape->next_width, logits, beam_scores, next_parent,
        (long long)parent_stride, next_token, next_score, workspace, s,
        events ? static_cast<cudaEvent_t>(events[1]) : nullptr));
    if (e1 != GR_OK || !events) return e1;
    return cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(events[2]), s));
}

int gr_beam_select(const gr_select_shape *shape, const float *logits, const float *beam_scores,
                   int32_t *next_parent, int64_t parent_stride, int32_t *next_token, float *next_score,
                   void *workspace, size_t workspace_bytes, gr_stream_t stream) {
    return beam_select_impl(shape, logits, beam_scores, next_parent, parent_stride, next_token, next_score,
                            workspace, workspace_bytes, stream, nullptr);
}

int gr_beam_select_timed(const gr_select_shape *shape, const float *logits, const float *beam_scores,
                         int32_t *next_parent, int64_t parent_stride, int32_t *next_token, float *next_score,
                         void *workspace, size_t workspace_bytes, gr_stream_t stream, gr_event_t const *events) {
    if (!events) return GR_ERR_NULL_ARG;
    return beam_select_impl(shape, logits, beam_scores, next_parent, parent_stride, next_token, next_score,
                            workspace, workspace_bytes, stream, events);
}

size_t gr_trie_select_workspace_size(const gr_trie_select_shape *shape) {
    if (!shape || shape->num_requests < 1 || shape->width < 1 || shape->vocab < 1 || shape->next_width < 1 ||
        shape->next_width > select_max_width() || shape->width > select_max_beams() || shape->num_nodes < 1 ||
        shape->num_edges < 0 || (long long)shape->width * shape->vocab >= (1LL << 31))
        return 0;
    return trie_select_bytes(shape->num_requests, shape->width, shape->next_width);
}

int gr_trie_select(const gr_trie_select_shape *shape, const float *logits, const float *beam_scores,
                   const int32_t *beam_node, const int32_t *trie_offsets, const int32_t *trie_tokens,
                   const int32_t *trie_children, int32_t *next_parent, int64_t parent_stride, int32_t *next_token,
                   float *next_score, int32_t *next_node, void *workspace, size_t workspace_bytes,
                   gr_stream_t stream) {
    if (!shape || !logits || !beam_scores || !beam_node || !trie_offsets || !next_parent || !next_token ||
        !next_score || !next_node || !workspace)
        return GR_ERR_NULL_ARG;
    if (shape->num_edges > 0 && (!trie_tokens || !trie_children)) return GR_ERR_NULL_ARG;
    const size_t need = gr_trie_select_workspace_size(shape);
    if (need == 0 || parent_stride < shape->next_width) return GR_ERR_BAD_SHAPE;
    if (misaligned(logits) || misaligned(beam_scores) || misaligned(beam_node) || misaligned(trie_offsets) ||
        (trie_tokens && misaligned(trie_tokens)) || (trie_children && misaligned(trie_children)) ||
        misaligned(next_parent) || misaligned(next_token) || misaligned(next_score) || misaligned(next_node) ||
        misaligned(workspace))
        return GR_ERR_MISALIGNED;
    if (workspace_bytes < need) return GR_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    return cuda_status(launch_trie_select(shape->num_requests, shape->width, shape->vocab, shape->next_width,
                                          shape->num_nodes, shape->num_edges, logits, beam_scores, beam_node,
                                          trie_offsets, trie_tokens, trie_children, next_parent,
                                          (long long)parent_stride, next_token, next_score, next_node, workspace,
                                          static_cast<cudaStream_t>(stream)));
}

int gr_beam_reorder(const gr_attn_shape *shape, const void *beam_k, const void *beam_v, const int32_t *beam_path,
                    const int32_t *widths, int32_t step, void *out_k, void *out_v, int32_t *out_path,
                    gr_stream_t stream) {
    Geometry g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (!beam_k || !beam_v || !beam_path || !out_k || !out_v || !out_path) return GR_ERR_NULL_ARG;
    if (misaligned(beam_k) || misaligned(beam_v) || misaligned(beam_path) || misaligned(out_k) ||
        misaligned(out_v) || misaligned(out_path))
        return GR_ERR_MISALIGNED;
    // out of place only: no output may share a byte with an input, since
    // other CTAs still read the inputs while the outputs are written
    {
        const size_t kv = (size_t)g.R * g.S_max * g.W_max * g.Hkv * g.D * 2;
        const size_t path = (size_t)g.R * g.S_max * g.W_max * sizeof(int32_t);
        const void *in[3] = {beam_k, beam_v, beam_path};
        const size_t in_bytes[3] = {kv, kv, path};
        const void *outs[3] = {out_k, out_v, out_path};
        const size_t out_bytes[3] = {kv, kv, path};
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 3; ++j)
                if (overlaps(outs[i], out_bytes[i], in[j], in_bytes[j])) return GR_ERR_BAD_SHAPE;
    }
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    return cuda_status(launch_reorder(g, static_cast<const uint16_t *>(beam_k), static_cast<const uint16_t *>(beam_v),
                                      beam_path, static_cast<uint16_t *>(out_k), static_cast<uint16_t *>(out_v),
                                      out_path, dev.err_ptr, static_cast<cudaStream_t>(stream)));
}

int gr_beam_reorder_inplace(const gr_attn_shape *shape, void *beam_k, void *beam_v, int32_t *beam_path,
                            const int32_t *widths, int32_t step, gr_stream_t stream) {
    Geometry g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (!beam_k || !beam_v || !beam_path) return GR_ERR_NULL_ARG;
    if (misaligned(beam_k) || misaligned(beam_v) || misaligned(beam_path)) return GR_ERR_MISALIGNED;
    // the K and V tiles are reordered by different CTAs and the path is read
    // by all of them: the three buffers must not share a byte
    {
        const size_t kv = (size_t)g.R * g.S_max * g.W_max * g.Hkv * g.D * 2;
        const size_t path = (size_t)g.R * g.S_max * g.W_max * sizeof(int32_t);
        if (overlaps(beam_k, kv, beam_v, kv) || overlaps(beam_k, kv, beam_path, path) ||
            overlaps(beam_v, kv, beam_path, path))
            return GR_ERR_BAD_SHAPE;
    }
    size_t smem = 0;
    if (inplace_tile_chunks(g, &smem) == 0) return GR_ERR_UNSUPPORTED;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    return cuda_status(launch_reorder_inplace(g, static_cast<uint16_t *>(beam_k), static_cast<uint16_t *>(beam_v),
                                              beam_path, dev.err_ptr, static_cast<cudaStream_t>(stream)));
}

int gr_beam_append(const gr_attn_shape *shape, const int32_t *widths, int32_t step, const void *k_new,
                   const void *v_new, int64_t src_stride, void *beam_k, void *beam_v, gr_stream_t stream) {
    Geometry g;
    int rc = make_geometry(shape, widths, step, &g);
    if (rc != GR_OK) return rc;
    if (!k_new || !v_new || !beam_k || !beam_v) return GR_ERR_NULL_ARG;
    const long long row = (long long)g.Hkv * g.D;
    if (src_stride < row) return GR_ERR_BAD_SHAPE;
    if (misaligned(k_new) || misaligned(v_new) || misaligned(beam_k) || misaligned(beam_v) || src_stride % 8 != 0)
        return GR_ERR_MISALIGNED;
    {
        const size_t kv = (size_t)g.R * g.S_max * g.W_max * g.Hkv * g.D * 2;
        const size_t src = ((size_t)(g.R * (long long)g.W_s - 1) * src_stride + row) * 2;
        if (overlaps(beam_k, kv, beam_v, kv) || overlaps(k_new, src, beam_k, kv) || overlaps(k_new, src, beam_v, kv) ||
            overlaps(v_new, src, beam_k, kv) || overlaps(v_new, src, beam_v, kv))
            return GR_ERR_BAD_SHAPE;
    }
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    return cuda_status(launch_append(g.R, g.W_s, g.S_max, g.W_max, g.Hkv, g.D, step,
                                     static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                                     (long long)src_stride, static_cast<uint16_t *>(beam_k),
                                     static_cast<uint16_t *>(beam_v), dev.sm_count, static_cast<cudaStream_t>(stream)));
}

int gr_get_device_error(void) {
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc != GR_OK) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GR_ERR_CUDA;
    }
    int code = 0;
    if (cudaMemcpyFromSymbol(&code, g_device_error, sizeof code) != cudaSuccess) {
        cudaGetLastError();
        return GR_ERR_CUDA;
    }
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return GR_ERR_CUDA;
    }
    if (code == kDevErrTimeout) return GR_ERR_DEVICE_TIMEOUT;
    if (code == kDevErrBadParent) return GR_ERR_BAD_BEAM_PATH;
    return GR_OK;
}

}  // extern "C"
