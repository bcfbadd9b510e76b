// gr_ctx_tc.cu -- shared (context) stage on the fifth-generation tensor cores.
//
// The shared stage is the one dense contraction of this attention: every
// query row (active beam x query head) of a request / kv-head pair attends to
// the same ContextKV, so the W*G rows of the pair form one dense M dimension
// and the context is streamed once per 256 rows instead of once per beam
// (GR-Inference blog, "kernel design": tensor-core MMA with split-KV over the
// long ContextKV; SID-GR README, section 9: the context part is processed per
// request and beam tile).  Online softmax over 128-key blocks follows the
// FlashAttention-style blocking the xGR review describes ("xAttention").
//
// One CTA = one (request, kv head, pair of 128-row tiles, key split):
//   warp 8      TMA producer: Q tiles once, then K/V blocks through a
//               4-slot shared-memory ring (128-byte swizzle).
//   warp 9      tensor-core issuer (one lane): S_t = Q_t K^T into TMEM,
//               O_t += P_t V with P read back from TMEM; owns the TMEM.
//   warps 0-3   softmax of tile 0, warps 4-7 softmax of tile 1: one thread
//               per row (TMEM lane), online max/sum, P (bf16) written over
//               the S columns; the O rescale is conditional (only when a
//               row's maximum grows by more than 2^8) and done in TMEM.
// The two tiles ping-pong, so one tile's softmax overlaps the other tile's
// MMAs.  Each split writes a normalised partial (O / l, LSE) per row; the
// per-beam stage and the LSE merge run in gr_beam_merge.cu.
//
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
// Every mbarrier wait is bounded: on expiry the CTA records a device error,
// drains its in-flight copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gr_common.cuh"
#include "gr_ptx.cuh"
#include "gr_tc_common.cuh"

namespace gr {

namespace {

using tc::kBM;
using tc::kBN;
using tc::fma_bf16x2;
using tc::kv_coords;
using tc::wait_lane;
using tc::wait_warp;
constexpr int kStages = 4;         // K/V ring slots
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBeamWarp = 10;               // warps 10 and 11: per-beam stage
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
// A block whose p = 2^(s*c - m) sum past this (so some p may be past it) has
// its row rescaled; below it every p is bounded by it, far from the fp32 and
// bf16 ranges, so the running maximum may lag the true one by up to 16 (log2)
constexpr float kSumLimit = 65536.0f;
constexpr int kFusedMaxTokens = 8;          // chain tokens the fused epilogue holds (steps < 8)
constexpr int kPrefetchBlocks = 1;          // K/V blocks of the next wave's CTA prefetched into L2

// barrier slots
constexpr int kBarKvFull = 0;               // [kStages]
constexpr int kBarKvEmpty = kStages;        // [kStages]
constexpr int kBarQFull = 2 * kStages;
constexpr int kBarSFull = 2 * kStages + 1;  // [2]
constexpr int kBarPFull = 2 * kStages + 3;  // [2]
constexpr int kBarODone = 2 * kStages + 5;  // [2]
constexpr int kBarFin = 2 * kStages + 7;
constexpr int kBarVTail = 2 * kStages + 8;     // the tail block's V rows past ctx_len are zeroed
constexpr int kBarBeam = 2 * kStages + 9;      // chain slots and scores are in shared memory
constexpr int kBarMerge = 2 * kStages + 10;    // [2] split merge: another split's partial tile has landed
constexpr int kNumBars = 2 * kStages + 12;

template <int D>
struct Cfg {
    static constexpr int kHalves = D / 64;              // 64-element (128-byte) swizzle columns
    static constexpr int kHalfBytes = kBM * 128;        // one 128-row x 64-element half
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kQOff = 0;                     // Q0, Q1
    static constexpr int kKvOff = 2 * kTileBytes;       // ring
    static constexpr int kBarOff = kKvOff + kStages * kTileBytes;
    // fused epilogue: per row and chain token, the token's score (base-2
    // units) and BeamKV slot; per row a flag for a broken chain
    static constexpr int kBeamX = kBarOff + kNumBars * 8 + 16;                  // float [kFusedMaxTokens][256]
    static constexpr int kBeamSlot = kBeamX + kFusedMaxTokens * 2 * kBM * 4;    // int   [kFusedMaxTokens][256]
    static constexpr int kBeamBad = kBeamSlot + kFusedMaxTokens * 2 * kBM * 4;  // int   [256]
    static constexpr int kUsed = kBeamBad + 2 * kBM * 4;
    // >= 116 KB keeps one CTA per SM, so the 512-column TMEM allocation never waits
    static constexpr int kSmem = (kUsed + 1024 > 118 * 1024 ? kUsed + 1024 : 118 * 1024);
    static constexpr int kOCol = 256;
};

struct TcParams {
    CtxArgs a;
    int bpt;    // beams per tile
    int tiles;  // tiles per (request, kv head)
    int sms;    // CTAs resident at once (one per SM)
};

// A tile's fp32 rows in shared memory as a TMA tensor copy lays them out
// with 128-byte swizzle: D/32 column chunks of 128 rows x 128 bytes, the
// 16-byte granule c of row m at m*128 + ((c ^ (m & 7)) << 4).  Used for the
// split partials (stored and loaded by TMA, so that a whole tile moves in
// one copy instead of one uncoalesced row per thread).
__device__ __forceinline__ uint32_t f32_granule(uint32_t stg, int k, int m_local, int c) {
    return stg + (uint32_t)(k * (kBM * 128) + m_local * 128 + ((c ^ (m_local & 7)) << 4));
}
__device__ __forceinline__ void st_f32x4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ float4 ld_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// One query row of the per-beam stage: its chain is walked by beam_prologue.
struct BeamRow {
    bool valid;      // a row of this call (inside the tile and the step's width)
    long long row;   // global row index (r, beam, query head)
    int beam;        // a_s: the row's beam at the current step
    int ridx;        // the row's slot in the shared-memory tables
    uint32_t q_smem; // the row's query in the swizzled Q tile
    int swz;         // 128-byte swizzle phase of that row
};

// Per-beam (unshared) stage for NR rows at a time, run by the beam warps
// while the context loop runs: walk BeamPath back from each row's beam
// (a_s = b, a_{t-1} = BeamPath[r, t, a_t]), score each chain token against
// the query (base-2 units), and keep slot and score in shared memory for the
// epilogue.  The NR rows advance together, and a token's parent index and K
// row are fetched together, so a token costs one memory round trip for all
// NR rows; the chain's V rows are prefetched into L2 for the epilogue.
template <int D, int NR>
__device__ __forceinline__ void beam_prologue(const CtxArgs &a, int r, int kvh, const BeamRow (&br)[NR],
                                              bool q_in_smem, float *s_x, int *s_slot, int *s_bad) {
    const Geometry &g = a.g;
    int slot[NR], bad[NR];
    bool on[NR];
#pragma unroll
    for (int k = 0; k < NR; ++k) {
        slot[k] = br[k].beam;
        bad[k] = 0;
        on[k] = br[k].valid;
    }
    // query chunk ch of row k: from the swizzled Q tile when it was loaded, else from global memory
    auto q_chunk = [&](int k, int ch) -> uint4 {
        uint4 v;
        if (q_in_smem) {
            const uint32_t addr =
                br[k].q_smem + (uint32_t)(ch >> 3) * (kBM * 128) + (uint32_t)(((ch & 7) ^ br[k].swz) * 16);
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(addr));
        } else {
            v = __ldg(reinterpret_cast<const uint4 *>(a.q + br[k].row * D) + ch);
        }
        return v;
    };
    for (int t = g.step; t >= 0; --t) {
        int par[NR];
        uint4 kv[NR][D / 8];
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            par[k] = 0;
            if (!on[k]) continue;
            if (t > 0) par[k] = __ldg(a.beam_path + ((long long)r * g.S_max + t) * g.W_max + slot[k]);
            const long long kv_off = ((((long long)r * g.S_max + t) * g.W_max + slot[k]) * g.Hkv + kvh) * D;
            const uint4 *kr = reinterpret_cast<const uint4 *>(a.beam_k + kv_off);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.beam_v + kv_off));
            if (D > 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.beam_v + kv_off + 64));
#pragma unroll
            for (int ch = 0; ch < D / 8; ++ch) kv[k][ch] = __ldg(kr + ch);
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            if (!on[k]) continue;
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
            for (int ch = 0; ch < D / 8; ++ch) {
                const uint4 qv = q_chunk(k, ch);
                const uint4 kc = kv[k][ch];
                fma_bf16x2(d0, d1, qv.x, kc.x);
                fma_bf16x2(d2, d3, qv.y, kc.y);
                fma_bf16x2(d0, d1, qv.z, kc.z);
                fma_bf16x2(d2, d3, qv.w, kc.w);
            }
            s_x[t * 2 * kBM + br[k].ridx] = ((d0 + d1) + (d2 + d3)) * g.scale_log2;
            s_slot[t * 2 * kBM + br[k].ridx] = slot[k];
            if (t > 0) {
                if (par[k] < 0 || par[k] >= width_of(g, r, t - 1)) {
                    bad[k] = 1;   // a parent out of range: nothing past it is read
                    on[k] = false;
                } else {
                    slot[k] = par[k];
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < NR; ++k)
        if (br[k].valid) s_bad[br[k].ridx] = bad[k];
}

// Merge for the row this thread owns (fused epilogue, single key split): the
// context partial (O in TMEM, running max m in base-2 units, sum l) and the
// chain tokens scored by beam_prologue are combined by log-sum-exp (the
// merging stage); the fp32 LSE is written, and the final bf16 row goes into
// `stage` (the tile's Q tile: row m_local, 128-byte swizzled as TMA lays it
// out) for the tile's TMA store.  The chain's V rows were prefetched into L2
// by the beam warps; they are loaded two tokens at a time.  tcgen05.ld is
// warp-collective, so every lane takes part in the O loads.  beam_ok is false
// when the beam warps gave up (the call already reports a timeout): the row
// is then written as NaN without reading the chain tables.
//
// kPartial (split 0 of a call with several key splits): the merged row is
// not final, since the other splits' context partials are still to come; it
// goes as split 0's normalised fp32 partial into `stage`, the tile's fp32
// staging (see f32_granule), and its LSE to *lse_part, so that the split
// merge finds the chain folded into it.
template <int D, bool kPartial>
__device__ __forceinline__ void beam_epilogue(const CtxArgs &a, int r, int kvh, long long row, bool row_ok,
                                              bool have_ctx, float m_ctx, float l_ctx, uint32_t tO,
                                              const float *s_x, const int *s_slot, const int *s_bad, int ridx,
                                              bool beam_ok, uint32_t stage, int m_local, float *lse_part = nullptr) {
    const Geometry &g = a.g;
    auto stage_chunk = [&](int hh, int c) -> uint32_t {
        return stage + (uint32_t)(hh * (kBM * 128) + m_local * 128 + ((c ^ (m_local & 7)) << 4));
    };
    const bool bad = row_ok && (!beam_ok || s_bad[ridx] != 0);
    if (!have_ctx) {
        m_ctx = -INFINITY;
        l_ctx = 0.f;
    }
    float m_tot = m_ctx;
    if (row_ok && !bad)
        for (int t = 0; t <= g.step; ++t) m_tot = fmaxf(m_tot, s_x[t * 2 * kBM + ridx]);
    const float w_ctx = ptx::ex2(m_ctx - m_tot);   // no context: exp2(-inf) = 0
    float L = l_ctx * w_ctx;
    if (row_ok && !bad)
        for (int t = 0; t <= g.step; ++t) L += ptx::ex2(s_x[t * 2 * kBM + ridx] - m_tot);
    const float inv = row_ok && !bad ? 1.f / L : 0.f;
#pragma unroll 1
    for (int hh = 0; hh < D / 64; ++hh) {
        float acc[64];
        if (have_ctx) {
            ptx::tmem_ld32(tO + 64 * hh, reinterpret_cast<uint32_t *>(&acc[0]));
            ptx::tmem_ld32(tO + 64 * hh + 32, reinterpret_cast<uint32_t *>(&acc[32]));
            ptx::tmem_wait_ld();
        } else {
#pragma unroll
            for (int d = 0; d < 64; ++d) acc[d] = 0.f;
        }
        if (!row_ok) continue;
        if (bad) {
            // NaN marks a row whose chain is broken
            if (kPartial) {
                const float nan = __int_as_float(0x7fc00000);
#pragma unroll
                for (int c = 0; c < 16; ++c) st_f32x4(f32_granule(stage, 2 * hh + (c >> 3), m_local, c & 7), nan, nan, nan, nan);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(stage_chunk(hh, c)), "r"(0x7fc07fc0u)
                                 : "memory");
            }
            continue;
        }
        const float wc = w_ctx * inv;
#pragma unroll
        for (int d = 0; d < 64; ++d) acc[d] *= wc;
        // chain tokens two at a time: both V row halves are in flight together
        for (int t0 = 0; t0 <= g.step; t0 += 2) {
            const bool two = t0 < g.step;
            uint4 va[8], vb[8];
            const float pa = ptx::ex2(s_x[t0 * 2 * kBM + ridx] - m_tot) * inv;
            const float pb = two ? ptx::ex2(s_x[(t0 + 1) * 2 * kBM + ridx] - m_tot) * inv : 0.f;
            const uint4 *ra = reinterpret_cast<const uint4 *>(
                a.beam_v + ((((long long)r * g.S_max + t0) * g.W_max + s_slot[t0 * 2 * kBM + ridx]) * g.Hkv + kvh) * D +
                64 * hh);
#pragma unroll
            for (int c = 0; c < 8; ++c) va[c] = __ldg(ra + c);
            if (two) {
                const uint4 *rb = reinterpret_cast<const uint4 *>(
                    a.beam_v +
                    ((((long long)r * g.S_max + t0 + 1) * g.W_max + s_slot[(t0 + 1) * 2 * kBM + ridx]) * g.Hkv + kvh) *
                        D +
                    64 * hh);
#pragma unroll
                for (int c = 0; c < 8; ++c) vb[c] = __ldg(rb + c);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) vb[c] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t ua[4] = {va[c].x, va[c].y, va[c].z, va[c].w};
                const uint32_t ub[4] = {vb[c].x, vb[c].y, vb[c].z, vb[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float &lo = acc[8 * c + 2 * e], &hi = acc[8 * c + 2 * e + 1];
                    lo = fmaf(pb, __uint_as_float(ub[e] << 16), fmaf(pa, __uint_as_float(ua[e] << 16), lo));
                    hi = fmaf(pb, __uint_as_float(ub[e] & 0xffff0000u), fmaf(pa, __uint_as_float(ua[e] & 0xffff0000u), hi));
                }
            }
        }
        if (kPartial) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
                st_f32x4(f32_granule(stage, 2 * hh + (c >> 3), m_local, c & 7), acc[4 * c + 0], acc[4 * c + 1],
                         acc[4 * c + 2], acc[4 * c + 3]);
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stage_chunk(hh, c)),
                             "r"(pack_bf16x2(acc[8 * c + 0], acc[8 * c + 1])),
                             "r"(pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3])),
                             "r"(pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5])),
                             "r"(pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]))
                             : "memory");
        }
    }
    if (!row_ok) return;
    float *lse_out = kPartial ? lse_part : a.lse + row;
    if (bad) {
        *lse_out = __int_as_float(0x7fc00000);
        if (beam_ok) raise_device_error(a.err, kDevErrBadParent);
        return;
    }
    *lse_out = (m_tot + log2f(L)) * kLn2;
}

// The split merge of one tile, run by its 128 softmax threads in the last
// CTA of a (request, kv head, tile pair) to finish its key split (the
// merging stage): every split has stored its normalised partial tile (O / l
// in fp32; split 0's includes the chain tokens) and its LSEs (natural log).
// The thread of row m_local weighs the splits by exp(lse_i - M) / sum, M the
// largest: each split's tile is brought into the staging area `stg` by TMA
// (one copy per split, from L2), in split order, and every thread reads its
// row back.  The
// final bf16 rows go to the tile's Q tile (`out_stage`, free once the MMAs
// are done) and leave by TMA stores; the fp32 LSE is written per row.  Every
// named barrier is reached by all 128 threads whatever happens, so a wait
// that gives up only records the error.  A NaN partial (a broken chain)
// makes the row NaN.
constexpr int kMaxMergeSplits = 16;   // splits the in-kernel merge takes

template <int D>
__device__ __forceinline__ void merge_tile(const CtxArgs &a, const CUtensorMap *tm_part, const CUtensorMap *tm_out,
                                           int r, int kvh, int tile, int bpt, int t, int m_local, bool row_ok,
                                           long long row, int sp_own, float lse_own, uint32_t stg, uint32_t mbar,
                                           uint32_t out_stage, volatile int *abort_flag) {
    const Geometry &g = a.g;
    const int n = a.sp.n_splits;
    const long long n_rows = (long long)g.R * g.W_s * g.Hq;
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    // the splits' LSEs (the own one is in a register, the others in L2): a
    // first pass for their maximum M, a second for the sum of the weights;
    // each weight is formed again where it is used
    auto lse_of = [&](int sp) -> float {
        if (!row_ok) return -INFINITY;
        return sp == sp_own ? lse_own : __ldcg(a.part_lse + sp * n_rows + row);
    };
    float M = -INFINITY;
#pragma unroll 1
    for (int sp = 0; sp < n; ++sp) M = fmaxf(M, lse_of(sp));
    float wsum = 0.f;
#pragma unroll 1
    for (int sp = 0; sp < n; ++sp) wsum += exp2f((lse_of(sp) - M) * kLog2e);   // an empty split: 0; NaN stays NaN
    float acc[D];
#pragma unroll
    for (int d = 0; d < D; ++d) acc[d] = 0.f;
    // every split's tile (this CTA's own included, so that the sum runs in
    // split order whichever CTA arrives last and the rows are the same in
    // every call) comes back by TMA; the tiles were published before this
    // CTA's acquire, which is ordered before the async-proxy loads here
    ptx::fence_proxy_async_global();
    int round = 0;
#pragma unroll 1
    for (int sp = 0; sp < n; ++sp) {
        ptx::named_bar_sync(1 + t, 4 * 32);   // the tile's own store has read `stg`, or the previous tile has been read
        if (quarter == 0 && lane == 0) {
            // a box is the tile's bpt * G rows (all of them count, past W_s too)
            ptx::mbar_arrive_expect_tx(mbar, (uint32_t)((D / 32) * bpt * g.G * 128));
#pragma unroll
            for (int k = 0; k < D / 32; ++k)
                ptx::tma_load_4d(stg + (uint32_t)(k * kBM * 128), tm_part, mbar, 32 * k, kvh * g.G, tile * bpt,
                                 sp * g.R + r);
        }
        if (!wait_warp(mbar, round & 1, abort_flag)) {
            *abort_flag = 1;
            if (lane == 0) raise_device_error(a.err, kDevErrTimeout);
        }
        ++round;
        const float ws = exp2f((lse_of(sp) - M) * kLog2e);
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = ld_f32x4(f32_granule(stg, k, m_local, c));
                acc[32 * k + 4 * c + 0] = fmaf(ws, v.x, acc[32 * k + 4 * c + 0]);
                acc[32 * k + 4 * c + 1] = fmaf(ws, v.y, acc[32 * k + 4 * c + 1]);
                acc[32 * k + 4 * c + 2] = fmaf(ws, v.z, acc[32 * k + 4 * c + 2]);
                acc[32 * k + 4 * c + 3] = fmaf(ws, v.w, acc[32 * k + 4 * c + 3]);
            }
    }
    const float inv = 1.f / wsum;
    if (row_ok) {
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float *o = acc + 64 * hh + 8 * c;
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 out_stage + (uint32_t)(hh * (kBM * 128) + m_local * 128 + ((c ^ (m_local & 7)) << 4))),
                             "r"(pack_bf16x2(o[0] * inv, o[1] * inv)), "r"(pack_bf16x2(o[2] * inv, o[3] * inv)),
                             "r"(pack_bf16x2(o[4] * inv, o[5] * inv)), "r"(pack_bf16x2(o[6] * inv, o[7] * inv))
                             : "memory");
            }
        a.lse[row] = M + logf(wsum);
    }
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(1 + t, 4 * 32);
    if (quarter == 0 && lane == 0) {
        for (int h = 0; h < D / 64; ++h)
            ptx::tma_store_4d(tm_out, out_stage + (uint32_t)(h * kBM * 128), h * 64, kvh * g.G, tile * bpt, r);
        ptx::bulk_commit();
        ptx::bulk_wait_all();   // the rows are written before the CTA (and its shared memory) ends
    }
}

// Requests ranked by context length, longest first (ties by index): the grid's
// y index counts (rank, kv head), so the CTAs of the longest requests are
// dispatched first and the short ones fill the tail of the last wave (a
// longest-processing-time order; it matters when context lengths differ).
// Each warp ranks the requests on its own, lane c taking request c, so no
// block barrier is needed.  Past 32 requests the order stays by index.
constexpr int kMaxRankedRequests = 32;

__device__ __forceinline__ int request_at_rank(const CtxArgs &a, int rank) {
    const Geometry &g = a.g;
    if (g.R <= 1 || g.R > kMaxRankedRequests) return rank;
    auto blocks = [&](int r) {
        int len = a.ctx_len[r];
        len = len < 0 ? 0 : (len > g.Lc_max ? g.Lc_max : len);
        return (len + tc::kBN - 1) / tc::kBN;
    };
    const int c = threadIdx.x & 31;
    int rk = -1;
    if (c < g.R) {
        const int bc = blocks(c);
        rk = 0;
        for (int o = 0; o < g.R; ++o) {
            const int bo = blocks(o);
            rk += (bo > bc || (bo == bc && o < c)) ? 1 : 0;
        }
    }
    const unsigned m = __ballot_sync(kFullMask, rk == rank);
    return m ? __ffs(m) - 1 : rank;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    ctx_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                  const __grid_constant__ CUtensorMap tm_part, const __grid_constant__ TcParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar0 = sbase + C::kBarOff;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kBarOff + kNumBars * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kBarOff + kNumBars * 8 + 4);

    const Geometry &g = p.a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x;
    const int kvh = blockIdx.y % g.Hkv, r = request_at_rank(p.a, blockIdx.y / g.Hkv), sp = blockIdx.z;
    const int tile0 = 2 * pair;
    const bool t1_active = (tile0 + 1) < p.tiles;
    const int rows_per_tile = p.bpt * g.G;

    // with per-request widths, a CTA whose tiles lie past its request's width has no rows
    if (g.req_widths && tile0 * p.bpt >= width_of(g, r, g.step)) return;
    int len = p.a.ctx_len[r];
    len = len < 0 ? 0 : (len > g.Lc_max ? g.Lc_max : len);
    const int kbeg = sp * p.a.sp.split_len;
    const int kend = min(kbeg + p.a.sp.split_len, len);
    const int nb = kend > kbeg ? (kend - kbeg + kBN - 1) / kBN : 0;

    // The producer initialises the barriers and starts the loads that the first
    // S needs (the Q tiles and K of block 0) while warp 9 allocates TMEM.
    if (warp == kProducerWarp && lane == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(bar(kBarKvFull + i), 1);
            ptx::mbar_init(bar(kBarKvEmpty + i), 1);
        }
        ptx::mbar_init(bar(kBarQFull), 1);
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(kBarSFull + t), 1);
            ptx::mbar_init(bar(kBarPFull + t), 4);   // one arrival per softmax warp
            ptx::mbar_init(bar(kBarODone + t), 1);
        }
        ptx::mbar_init(bar(kBarFin), 1);
        ptx::mbar_init(bar(kBarVTail), 1);
        ptx::mbar_init(bar(kBarBeam), 2);   // one arrival per beam warp
        ptx::mbar_init(bar(kBarMerge + 0), 1);
        ptx::mbar_init(bar(kBarMerge + 1), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == kProducerWarp && nb > 0) {
        __syncwarp();
        // rows of a tile past bpt*G are never loaded: keep them zero
        if (rows_per_tile < kBM) {
            const int tail = (kBM - rows_per_tile) * 128;
            for (int t = 0; t < 2; ++t)
                for (int h = 0; h < C::kHalves; ++h)
                    for (int off = lane * 16; off < tail; off += 32 * 16)
                        *reinterpret_cast<uint4 *>(smem + C::kQOff + t * C::kTileBytes + h * C::kHalfBytes +
                                                   rows_per_tile * 128 + off) = make_uint4(0, 0, 0, 0);
            ptx::fence_proxy_async_smem();
            __syncwarp();
        }
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_q);
            ptx::prefetch_tmap(&tm_k);
            ptx::prefetch_tmap(&tm_v);
            const int nt = t1_active ? 2 : 1;
            ptx::mbar_arrive_expect_tx(bar(kBarQFull), (uint32_t)(nt * C::kHalves * rows_per_tile * 128));
            for (int t = 0; t < nt; ++t)
                for (int h = 0; h < C::kHalves; ++h)
                    ptx::tma_load_4d(sbase + C::kQOff + t * C::kTileBytes + h * C::kHalfBytes, &tm_q, bar(kBarQFull),
                                     h * 64, kvh * g.G, (tile0 + t) * p.bpt, r);
            // load 0 (K of block 0) into ring slot 0, which starts out free
            ptx::mbar_arrive_expect_tx(bar(kBarKvFull + 0), (uint32_t)C::kTileBytes);
            int c1, c3;
            kv_coords(p.a, r, kbeg, c1, c3);
            for (int h = 0; h < C::kHalves; ++h)
                ptx::tma_load_4d(sbase + C::kKvOff + h * C::kHalfBytes, &tm_k, bar(kBarKvFull + 0), h * 64, c1, kvh,
                                 c3);
        }
        __syncwarp();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        if (lane == 0) raise_device_error(p.a.err, kDevErrTimeout);
    };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // The CTA one wave on (linear index + SMs) takes an SM as CTAs of this
        // wave finish: its Q tiles and first K/V blocks are prefetched into L2
        // once this CTA's last load is out, so its first S does not wait on
        // DRAM.
        const long long total = (long long)gridDim.x * gridDim.y * gridDim.z;
        const long long succ =
            (long long)blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z) + p.sms;
        int s_r = -1, s_kvh = 0, s_tile0 = 0, s_kbeg = 0, s_len = 0;
        if (p.sms > 0 && succ < total) {   // warp-uniform
            const int sx = (int)(succ % gridDim.x);
            const int sy = (int)((succ / gridDim.x) % gridDim.y);
            const int sz = (int)(succ / ((long long)gridDim.x * gridDim.y));
            s_r = request_at_rank(p.a, sy / g.Hkv);   // warp-collective
            s_kvh = sy % g.Hkv;
            s_tile0 = 2 * sx;
            s_kbeg = sz * p.a.sp.split_len;
            int sl = p.a.ctx_len[s_r];
            sl = sl < 0 ? 0 : (sl > g.Lc_max ? g.Lc_max : sl);
            s_len = min(s_kbeg + p.a.sp.split_len, sl) - s_kbeg;
        }
        int issued = 1;   // the Q tiles and load 0 went out before the CTA-wide barrier
        bool ok = true;
        if (nb > 0) {
            for (int n = 1; n < 2 * nb; ++n) {
                const int s = n % kStages;
                if (!wait_warp(bar(kBarKvEmpty + s), ((n / kStages) & 1) ^ 1, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar(kBarKvFull + s), (uint32_t)C::kTileBytes);
                    const CUtensorMap *tm = (n & 1) ? &tm_v : &tm_k;
                    int c1, c3;
                    kv_coords(p.a, r, kbeg + (n >> 1) * kBN, c1, c3);
                    for (int h = 0; h < C::kHalves; ++h)
                        ptx::tma_load_4d(sbase + C::kKvOff + s * C::kTileBytes + h * C::kHalfBytes, tm,
                                         bar(kBarKvFull + s), h * 64, c1, kvh, c3);
                }
                __syncwarp();
                issued = n + 1;
                const int valid = min(kBN, kend - (kbeg + (n >> 1) * kBN));
                if ((n & 1) && valid < kBN) {
                    // the last block of the range: context positions past ctx_len hold
                    // anything, so once the V block lands its rows past the end are
                    // zeroed (P is 0 there, but 0 * NaN would not be)
                    if (!wait_warp(bar(kBarKvFull + s), (n / kStages) & 1, abort_flag)) {
                        fail();
                        ok = false;
                        break;
                    }
                    const int bytes = (kBN - valid) * 128;
                    for (int h = 0; h < C::kHalves; ++h)
                        for (int off = lane * 16; off < bytes; off += 32 * 16)
                            *reinterpret_cast<uint4 *>(smem + C::kKvOff + s * C::kTileBytes + h * C::kHalfBytes +
                                                       valid * 128 + off) = make_uint4(0, 0, 0, 0);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(kBarVTail));
                }
            }
            if (!ok) {
                // drain: every copy in flight lands before the CTA leaves
                wait_warp(bar(kBarQFull), 0, nullptr);
                for (int n = issued - kStages < 0 ? 0 : issued - kStages; n < issued; ++n)
                    wait_warp(bar(kBarKvFull + n % kStages), (n / kStages) & 1, nullptr);
            } else if (s_r >= 0 && lane == 0) {
                const int nt = (s_tile0 + 1 < p.tiles) ? 2 : 1;
                for (int t = 0; t < nt; ++t)
                    for (int h = 0; h < C::kHalves; ++h)
                        ptx::tma_prefetch_4d(&tm_q, h * 64, s_kvh * g.G, (s_tile0 + t) * p.bpt, s_r);
                for (int b = 0; b < kPrefetchBlocks && b * kBN < s_len; ++b) {
                    int c1, c3;
                    kv_coords(p.a, s_r, s_kbeg + b * kBN, c1, c3);
                    for (int h = 0; h < C::kHalves; ++h) {
                        ptx::tma_prefetch_4d(&tm_k, h * 64, c1, s_kvh, c3);
                        ptx::tma_prefetch_4d(&tm_v, h * 64, c1, s_kvh, c3);
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // One lane issues; lanes 1-31 go straight to the final barrier, so the
        // issuing thread never reconverges its warp between MMA groups.
        if (nb > 0 && lane == 0) {
            constexpr uint32_t kIdescQK = ptx::idesc_bf16(kBM, kBN, 0);
            constexpr uint32_t kIdescPV = ptx::idesc_bf16(kBM, D, 1);
            const int ntiles = t1_active ? 2 : 1;
            // Every descriptor is formed once, so each MMA costs only an add and
            // the instruction itself.  A k-step of 16 elements moves a K-major
            // 128B-swizzled operand by 32 bytes inside the swizzle atom (and by a
            // whole 64-column half after 4 steps), and the N-major V operand by 16
            // rows = 2048 bytes; in descriptor units (16 bytes) these are small
            // constants added to the address field.  Q tiles and ring slots are
            // equally spaced, so a slot's descriptor is the first one's plus a
            // multiple of the slot size.
            const uint64_t dq0 = ptx::smem_desc(sbase + C::kQOff, 16, 1024);
            const uint64_t dk0 = ptx::smem_desc(sbase + C::kKvOff, 16, 1024);
            const uint64_t dv0 = ptx::smem_desc(sbase + C::kKvOff, C::kHalfBytes, 1024);
            constexpr uint64_t kSlot = C::kTileBytes >> 4;
            auto qk_step = [](int kk) -> uint64_t { return (uint64_t)((kk >> 2) * (C::kHalfBytes >> 4) + (kk & 3) * 2); };
            auto issue_s = [&](int t, int s) {
                ptx::tc_fence_after();
                const uint64_t a0 = dq0 + (uint64_t)t * kSlot, b0 = dk0 + (uint64_t)s * kSlot;
                const uint32_t d = tmem + t * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) ptx::mma_ss(d, a0 + qk_step(kk), b0 + qk_step(kk), kIdescQK, kk > 0);
                ptx::mma_commit(bar(kBarSFull + t));
            };
            auto issue_pv = [&](int t, int s, int i) {
                ptx::tc_fence_after();
                const uint64_t b0 = dv0 + (uint64_t)s * kSlot;
                const uint32_t d = tmem + C::kOCol + t * D, a = tmem + t * kBN;
                const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    ptx::mma_ts(d, a + kk * 8, b0 + (uint64_t)(kk * (2048 >> 4)), kIdescPV, kk > 0 ? 1u : acc0);
            };

            bool ok = wait_lane(bar(kBarQFull), 0, abort_flag) && wait_lane(bar(kBarKvFull + 0), 0, abort_flag);
            if (ok) {
                for (int t = 0; t < ntiles; ++t) issue_s(t, 0);
                ptx::mma_commit(bar(kBarKvEmpty + 0));
            }
            // A thread that has just issued MMAs stalls on its next mbarrier
            // wait until they have drained into the tensor pipe, which then runs
            // dry: every wait here costs pipe time, but back-to-back waits cost
            // little more than one.  So the issuer waits at two points per
            // block: for P_0(i) together with V(i) and K(i+1), and for P_1(i).
            for (int i = 0; ok && i < nb; ++i) {
                const int sv = (2 * i + 1) % kStages;
                const bool has_next = (i + 1) < nb;
                const int sk = (2 * (i + 1)) % kStages;
                if (!(ok = wait_lane(bar(kBarPFull + 0), i & 1, abort_flag))) break;
                {
                    // a tail block's V is usable once the producer has zeroed its rows past the end
                    const int valid = min(kBN, kend - (kbeg + i * kBN));
                    const int nv = 2 * i + 1, nk = 2 * (i + 1);
                    if (!(ok = (valid < kBN) ? wait_lane(bar(kBarVTail), 0, abort_flag)
                                             : wait_lane(bar(kBarKvFull + nv % kStages), (nv / kStages) & 1, abort_flag)))
                        break;
                    if (has_next && !(ok = wait_lane(bar(kBarKvFull + nk % kStages), (nk / kStages) & 1, abort_flag))) break;
                }
                issue_pv(0, sv, i);
                if (i == nb - 1) ptx::mma_commit(bar(kBarODone + 0));
                if (has_next) issue_s(0, sk);
                if (t1_active) {
                    if (!(ok = wait_lane(bar(kBarPFull + 1), i & 1, abort_flag))) break;
                    issue_pv(1, sv, i);
                    if (i == nb - 1) ptx::mma_commit(bar(kBarODone + 1));
                }
                // V(i)'s slot is free once the last PV that reads it is done
                ptx::mma_commit(bar(kBarKvEmpty + sv));
                if (t1_active && has_next) issue_s(1, sk);
                if (has_next) ptx::mma_commit(bar(kBarKvEmpty + sk));
            }
            if (!ok) {
                *abort_flag = 1;
                raise_device_error(p.a.err, kDevErrTimeout);
            }
            // no MMA may still be running when the TMEM is released
            ptx::mma_commit(bar(kBarFin));
            wait_lane(bar(kBarFin), 0, nullptr);
        }
    } else if (warp >= kBeamWarp) {
        // ------------------------------------------------------------ per-beam stage
        // 64 threads, four rows each (rows b and b + 64 of each tile, one at a
        // time: measured faster than two rows in flight, which load the SM's
        // memory pipeline harder while the softmax warps use it), while the
        // context loop runs; then one arrival per warp.
        if (p.a.fused || (p.a.split_merge && sp == 0)) {
            bool okq = nb == 0 || wait_warp(bar(kBarQFull), 0, abort_flag);   // q is read from the Q tile
            if (!okq) {
                fail();
            } else {
                float *s_x = reinterpret_cast<float *>(smem + C::kBeamX);
                int *s_slot = reinterpret_cast<int *>(smem + C::kBeamSlot);
                int *s_bad = reinterpret_cast<int *>(smem + C::kBeamBad);
                const int b = (warp - kBeamWarp) * 32 + lane;
                for (int t = 0; t < 2; ++t) {
                    if (t == 1 && !t1_active) break;
                    for (int k = 0; k < 2; ++k) {
                        const int m_local = b + 64 * k;
                        const int beam = (tile0 + t) * p.bpt + m_local / g.G;
                        BeamRow br[1];
                        br[0].valid = (m_local < rows_per_tile) && (beam < width_of(g, r, g.step));
                        br[0].row = ((long long)r * g.W_s + beam) * g.Hq + kvh * g.G + m_local % g.G;
                        br[0].beam = beam;
                        br[0].ridx = t * kBM + m_local;
                        br[0].q_smem = sbase + C::kQOff + t * C::kTileBytes + (uint32_t)m_local * 128u;
                        br[0].swz = m_local & 7;
                        beam_prologue<D, 1>(p.a, r, kvh, br, nb > 0, s_x, s_slot, s_bad);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarBeam));
        }
    } else {
        // ------------------------------------------------------------ softmax + partial epilogue
        const int t = warp >> 2, quarter = warp & 3;
        const int m_local = quarter * 32 + lane;
        const bool tile_active = (t == 0) || t1_active;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)(t * kBN);
        const uint32_t tO = tmem + lane_off + (uint32_t)(C::kOCol + t * D);
        const float c = g.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        float *s_x = reinterpret_cast<float *>(smem + C::kBeamX);
        int *s_slot = reinterpret_cast<int *>(smem + C::kBeamSlot);
        int *s_bad = reinterpret_cast<int *>(smem + C::kBeamBad);
        const int ridx = t * kBM + m_local;

        // this thread's row: beam b, query head kvh*G + m_local%G
        auto row_beam = [&]() { return (tile0 + t) * p.bpt + m_local / g.G; };
        auto row_valid = [&]() { return (m_local < rows_per_tile) && (row_beam() < width_of(g, r, g.step)); };
        auto row_index = [&]() {
            return ((long long)r * g.W_s + row_beam()) * g.Hq + kvh * g.G + m_local % g.G;
        };
        if (tile_active && nb > 0) {
            for (int i = 0; i < nb; ++i) {
                const int valid = min(kBN, kend - (kbeg + i * kBN));
                if (!(ok = wait_warp(bar(kBarSFull + t), i & 1, abort_flag))) break;
                ptx::tc_fence_after();
                uint32_t sv[kBN];
#pragma unroll
                for (int q4 = 0; q4 < kBN / 32; ++q4)
                    ptx::tmem_ld32(tS + 32 * q4, &sv[32 * q4]);
                ptx::tmem_wait_ld();
                if (valid < kBN) {
#pragma unroll
                    for (int j = 0; j < kBN; ++j)
                        if (j >= valid) sv[j] = __float_as_uint(-INFINITY);
                }
                if (i == 0) {
                    // the first block sets the running maximum: 3-input max over 8 chains
                    float mx8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float mu = fmaxf(__uint_as_float(sv[u]), __uint_as_float(sv[u + 8]));
#pragma unroll
                        for (int k = 2; k < 16; k += 2)
                            mu = ptx::fmax3(mu, __uint_as_float(sv[u + 8 * k]), __uint_as_float(sv[u + 8 * k + 8]));
                        mx8[u] = mu;
                    }
                    m = fmaxf(ptx::fmax3(mx8[0], mx8[1], mx8[2]),
                              fmaxf(ptx::fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * c;
                }
                // p = 2^(s*c - m) against the running maximum m.  The block's own
                // maximum is not computed: every p is at most the block's sum, so a
                // sum of at most kSumLimit bounds every p and the row needs no
                // rescale.  Past it (rare after the first block, or inf/NaN) the
                // block maximum is taken from the scores still in registers, O and
                // l are rescaled in TMEM and the pass is redone once.  Packed
                // scale-and-subtract, exp2 on the MUFU unit, packed row sums, and
                // bf16 pairs stored over the first 64 S columns as P for the PV MMA.
                float blk = 0.f;
#pragma unroll 1
                for (int pass = 0; pass < 2; ++pass) {
                    const float neg_m = -m;
                    float sa[2] = {0.f, 0.f}, sb[2] = {0.f, 0.f};
#pragma unroll
                    for (int qtr = 0; qtr < 4; ++qtr) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = 32 * qtr + 2 * j;
                            const float s0 = __uint_as_float(sv[col]), s1 = __uint_as_float(sv[col + 1]);
                            float x0, x1, p0, p1;
                            ptx::ffma2(x0, x1, s0, s1, c, c, neg_m, neg_m);
                            p0 = ptx::ex2(x0);
                            p1 = ptx::ex2(x1);
                            ptx::fadd2(sa[j & 1], sb[j & 1], sa[j & 1], sb[j & 1], p0, p1);
                            pk[j] = pack_bf16x2(p0, p1);
                        }
                        ptx::tmem_st16(tS + 16 * qtr, pk);
                    }
                    blk = (sa[0] + sa[1]) + (sb[0] + sb[1]);
                    const bool need = pass == 0 && !(blk <= kSumLimit);
                    if (!__any_sync(kFullMask, need)) break;
                    float mx8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float mu = fmaxf(__uint_as_float(sv[u]), __uint_as_float(sv[u + 8]));
#pragma unroll
                        for (int k = 2; k < 16; k += 2)
                            mu = ptx::fmax3(mu, __uint_as_float(sv[u + 8 * k]), __uint_as_float(sv[u + 8 * k + 8]));
                        mx8[u] = mu;
                    }
                    const float m_blk = fmaxf(ptx::fmax3(mx8[0], mx8[1], mx8[2]),
                                              fmaxf(ptx::fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * c;
                    // O (and l) carry the old maximum: rescale them in TMEM, then redo
                    const float f = need ? ptx::ex2(m - m_blk) : 1.f;
#pragma unroll 1
                    for (int q4 = 0; q4 < D / 16; ++q4) {
                        uint32_t ov[16];
                        ptx::tmem_ld16(tO + 16 * q4, ov);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
                        ptx::tmem_st16(tO + 16 * q4, ov);
                    }
                    l *= f;
                    if (need) m = m_blk;
                }
                l += blk;
                // P is in TMEM: each thread's stores complete and are fenced, the
                // warp synchronises, and one lane signals for the warp
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kBarPFull + t));
            }
            if (ok) ok = wait_warp(bar(kBarODone + t), 0, abort_flag);
            if (!ok) fail();
            ptx::tc_fence_after();
        }
        const bool row_ok = row_valid();
        const long long row = row_index();
        if (tile_active && p.a.fused) {
            // the beam warps have filled the chain tables
            const bool beam_ok = wait_warp(bar(kBarBeam), 0, abort_flag);
            if (!beam_ok) fail();
            // the final rows leave through this tile's Q tile (free: every S of
            // the tile has completed, the beam warps are done with q) by TMA
            const uint32_t stage = sbase + C::kQOff + t * C::kTileBytes;
            beam_epilogue<D, false>(p.a, r, kvh, row, row_ok, ok && nb > 0, m, l, tO, s_x, s_slot, s_bad, ridx,
                                    beam_ok, stage, m_local);
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1 + t, 4 * 32);
            if (quarter == 0 && lane == 0) {
                for (int h = 0; h < C::kHalves; ++h)
                    ptx::tma_store_4d(&tm_out, stage + h * C::kHalfBytes, h * 64, kvh * g.G, (tile0 + t) * p.bpt, r);
                ptx::bulk_commit();
                ptx::bulk_wait_all();   // the rows are written before the CTA (and its shared memory) ends
            }
        } else if (p.a.split_merge) {
            // this split's normalised partial goes to the tile's fp32 staging
            // (ring slots 2t and 2t+1, free once the MMAs are done) and leaves by
            // TMA; split 0 folds the chain tokens into it
            const long long n_rows = (long long)g.R * g.W_s * g.Hq;
            const uint32_t stg = sbase + C::kKvOff + (uint32_t)(2 * t * C::kTileBytes);
            float lse_own = -INFINITY;
            // the ring is free once every MMA is done: tile 1's last PV may still
            // read a V block when tile 0's own MMAs have finished
            if (tile_active && t == 0 && t1_active && nb > 0 && ok && !wait_warp(bar(kBarODone + 1), 0, abort_flag)) {
                ok = false;
                fail();
            }
            if (tile_active) {
                const bool have = ok && nb > 0;
                if (sp == 0) {
                    const bool beam_ok = wait_warp(bar(kBarBeam), 0, abort_flag);
                    if (!beam_ok) fail();
                    beam_epilogue<D, true>(p.a, r, kvh, row, row_ok, have, m, l, tO, s_x, s_slot, s_bad, ridx,
                                           beam_ok, stg, m_local, &lse_own);
                } else {
                    const float inv = (have && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t ov[32];
                        if (have) {
                            ptx::tmem_ld32(tO + 32 * q4, ov);
                            ptx::tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) ov[j] = 0u;
                        }
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            st_f32x4(f32_granule(stg, q4, m_local, c), __uint_as_float(ov[4 * c]) * inv,
                                     __uint_as_float(ov[4 * c + 1]) * inv, __uint_as_float(ov[4 * c + 2]) * inv,
                                     __uint_as_float(ov[4 * c + 3]) * inv);
                    }
                    lse_own = (have && l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
                }
                if (row_ok) p.a.part_lse[(long long)sp * n_rows + row] = lse_own;
                ptx::fence_proxy_async_smem();
                ptx::named_bar_sync(1 + t, 4 * 32);
                if (quarter == 0 && lane == 0) {
                    for (int k = 0; k < D / 32; ++k)
                        ptx::tma_store_4d(&tm_part, stg + (uint32_t)(k * kBM * 128), 32 * k, kvh * g.G,
                                          (tile0 + t) * p.bpt, sp * g.R + r);
                    ptx::bulk_commit();
                    ptx::bulk_wait_all();
                    ptx::fence_proxy_async_global();
                }
            }
            // arrive on the (request, kv head, tile pair) counter once this CTA's
            // partial tiles and LSEs are visible device-wide; the last split to
            // arrive merges every split's partials into the final rows
            volatile int *s_last = reinterpret_cast<volatile int *>(smem + C::kBarOff + kNumBars * 8 + 8);
            __threadfence();
            ptx::named_bar_sync(3, 8 * 32);
            if (warp == 0 && lane == 0) {
                const int item = (r * g.Hkv + kvh) * (int)gridDim.x + pair;
                const int before = atomicAdd(p.a.counters + item, 1);
                *s_last = (before == p.a.sp.n_splits - 1) ? 1 : 0;
                __threadfence();
            }
            ptx::named_bar_sync(3, 8 * 32);
            if (*s_last && tile_active) {
                __threadfence();
                merge_tile<D>(p.a, &tm_part, &tm_out, r, kvh, tile0 + t, p.bpt, t, m_local, row_ok, row, sp, lse_own,
                              stg, bar(kBarMerge + t), sbase + C::kQOff + (uint32_t)(t * C::kTileBytes), abort_flag);
            }
        } else if (tile_active) {
            const long long n_rows = (long long)g.R * g.W_s * g.Hq;
            float *po = p.a.part_o + ((long long)sp * n_rows + row) * D;
            const bool have = ok && nb > 0;
            const float inv = (have && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
            for (int q4 = 0; q4 < D / 32; ++q4) {
                uint32_t ov[32];
                if (have) {
                    ptx::tmem_ld32(tO + 32 * q4, ov);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = 0u;
                }
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(po + 32 * q4 + j) =
                            make_float4(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv,
                                        __uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
                }
            }
            if (row_ok)
                p.a.part_lse[(long long)sp * n_rows + row] = (have && l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
        }
    }

    // every role is done: the MMA issuer's lanes arrive one by one (its idle
    // lanes early, the issuing lane once the last MMA has completed), then the
    // allocating warp, converged again, releases the TMEM
    ptx::tc_fence_before();
    ptx::block_bar_sync_threads();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------- host side

template <int D>
cudaError_t launch_d(const CtxArgs &a, int bpt, int tiles, int sm_count, cudaStream_t s) {
    using C = Cfg<D>;
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev < 64 && !attr_set[dev]) {
            e = cudaFuncSetAttribute(ctx_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const Geometry &g = a.g;
    CUtensorMap tq, tk, tv, to;
    const uint64_t qd[4] = {(uint64_t)D, (uint64_t)g.Hq, (uint64_t)g.W_s, (uint64_t)g.R};
    const uint64_t qs[3] = {(uint64_t)D * 2, (uint64_t)g.Hq * D * 2, (uint64_t)g.W_s * g.Hq * D * 2};
    const uint32_t qb[4] = {64, (uint32_t)g.G, (uint32_t)bpt, 1};
    // dense [R, Hkv, Lc_max, D] or a paged pool [num_pages, Hkv, page_size, D]
    const uint64_t rows = a.page_size ? (uint64_t)a.page_size : (uint64_t)g.Lc_max;
    const uint64_t outer = a.page_size ? (uint64_t)a.num_pages : (uint64_t)g.R;
    const uint64_t kd[4] = {(uint64_t)D, rows, (uint64_t)g.Hkv, outer};
    const uint64_t ks[3] = {(uint64_t)D * 2, rows * D * 2, (uint64_t)g.Hkv * rows * D * 2};
    const uint32_t kb[4] = {64, (uint32_t)kBN, 1, 1};
    if (!encode_4d(&tq, a.q, qd, qs, qb) || !encode_4d(&tk, a.ctx_k, kd, ks, kb) ||
        !encode_4d(&tv, a.ctx_v, kd, ks, kb))
        return cudaErrorInvalidValue;
    TcParams p;
    p.a = a;
    p.bpt = bpt;
    p.tiles = tiles;
    p.sms = sm_count;
    dim3 grid((tiles + 1) / 2, g.R * g.Hkv, a.sp.n_splits);
    // fused path and split merge: the output rows leave by TMA stores with the
    // Q tiles' geometry
    if (a.fused || a.split_merge) {
        if (!encode_4d(&to, a.out, qd, qs, qb)) return cudaErrorInvalidValue;
    } else {
        to = tq;   // unused
    }
    // split merge: the fp32 partials [n_splits * R, W_s, Hq, D] move as tiles
    // of 32-float column chunks
    CUtensorMap tp;
    if (a.split_merge) {
        const uint64_t pd[4] = {(uint64_t)D, (uint64_t)g.Hq, (uint64_t)g.W_s, (uint64_t)a.sp.n_splits * g.R};
        const uint64_t ps[3] = {(uint64_t)D * 4, (uint64_t)g.Hq * D * 4, (uint64_t)g.W_s * g.Hq * D * 4};
        const uint32_t pb[4] = {32, (uint32_t)g.G, (uint32_t)bpt, 1};
        if (!encode_4d(&tp, a.part_o, pd, ps, pb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) return cudaErrorInvalidValue;
    } else {
        tp = tq;   // unused
    }
    ctx_tc_kernel<D><<<grid, kThreads, C::kSmem, s>>>(tq, tk, tv, to, tp, p);
    return cudaGetLastError();
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

bool encode_4d(CUtensorMap *m, const void *base, const uint64_t dims[4], const uint64_t strides_bytes[3],
               const uint32_t box[4], CUtensorMapDataType dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint32_t elem[4] = {1, 1, 1, 1};
    const CUresult rc = fn(m, dtype, 4, const_cast<void *>(base), dims, strides_bytes,
                           box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

int tc_beams_per_tile(int G) { return kBM / G; }
int tc_fused_max_steps(int) { return kFusedMaxTokens; }
int tc_merge_max_splits() { return kMaxMergeSplits; }

cudaError_t launch_ctx_tc(const CtxArgs &a, int sm_count, cudaStream_t s) {
    const int bpt = tc_beams_per_tile(a.g.G);
    const int tiles = (a.g.W_s + bpt - 1) / bpt;
    if (a.g.D == 128) return launch_d<128>(a, bpt, tiles, sm_count, s);
    return launch_d<64>(a, bpt, tiles, sm_count, s);
}

}  // namespace gr
