// gr_ctx_pk.cu -- the whole decode attention (shared stage on the tensor
// cores, per-beam stage, log-sum-exp merge) as one persistent kernel over
// 128-row tiles.
//
// The shared stage is the one dense contraction of this attention: the W*G
// query rows (active beam x query head) of a request / kv-head pair form one
// dense M dimension against the pair's ContextKV (GR-Inference blog, "kernel
// design": tensor-core MMA over the long ContextKV; SID-GR README, section 9:
// the context part is processed per request and beam tile), with online
// softmax over 128-key blocks (xGR review, "xAttention", FlashAttention-style
// blocking).  Each row's own chain of decoded tokens is reached along
// BeamPath and merged by log-sum-exp in the epilogue (the unshared and
// merging stages).
//
// Work item = (request, kv head, 128-row tile); the grid holds at most one
// CTA per SM and each CTA walks the items blockIdx.x, + gridDim.x, ...
// Consecutive key blocks overlap, and so do consecutive items up to their O
// (the next item's loads and S run while the epilogue drains the last one):
//   TMEM    S_0 [0,128) S_1 [128,256): S of consecutive key blocks (global
//           block n uses S_{n&1}), so S(n+1) is computed while the softmax
//           of block n runs; O [256,256+D): the item's context partial;
//           C [256+D,256+2D): the partial of the rows' own chains, written by
//           the epilogue warps while the context loop runs.
//   SMEM    the item's Q tile (reloaded once its last S is done and its
//           chains are scored); a 3-slot K ring and a 3-slot V ring that
//           run on across items, so a K block is in flight for about two
//           key blocks before its S and a V block for more before its PV.
// Roles (11 warps):
//   warps 0-3   softmax, one thread per row (TMEM lane): online max / sum,
//               P (bf16) over the first 64 columns of S_{n&1}; the O
//               rescale is rare (kSumLimit) and waits for the previous PV.
//   warps 4-7   epilogue, one thread per row: while the item's context
//               loop runs, walks the row's chain, scores its tokens and
//               accumulates their V rows into C (a softmax of its own, with
//               the chain's maximum and sum kept in registers); once O is
//               complete, merges the two partials by log-sum-exp from TMEM
//               and writes the bf16 row (the CTA's last item through its
//               freed Q tile and a TMA store) and its LSE.
//   warp 8      TMA producer of the Q tiles and the K ring.
//   warp 9      MMA issuer (one lane).
//   warp 10     TMA producer of the V ring (zeroes V rows past ctx_len).
// Every mbarrier wait is bounded: on expiry the CTA records a device error,
// each role finishes its loop without waiting, in-flight copies and MMAs are
// drained, the TMEM is freed and the CTA returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gr_common.cuh"
#include "gr_ptx.cuh"
#include "gr_tc_common.cuh"

namespace gr {

namespace {

using tc::fma_bf16x2;
using tc::kBM;
using tc::kBN;
using tc::kv_coords;
using tc::wait_lane;
using tc::wait_warp;

constexpr int kKStages = 3;         // K ring slots
constexpr int kVStages = 3;         // V ring slots
constexpr int kEpiWarp0 = 4;        // warps 4-7 (softmax: 0-3)
constexpr int kKProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;
constexpr int kThreads = 11 * 32;
constexpr int kTmemCols = 512;
constexpr int kMaxTokens = 8;       // chain tokens the epilogue holds (steps < 8)
// A block whose p = 2^(s*c - m) sum past this (so some p may be past it) has
// its row rescaled; below it every p is bounded by it, far from the fp32 and
// bf16 ranges, so the running maximum may lag the true one by up to 16 (log2)
constexpr float kSumLimit = 65536.0f;

// barrier slots
constexpr int kBarKFull = 0;         // [kKStages]
constexpr int kBarKEmpty = 3;        // [kKStages]
constexpr int kBarVFull = 6;         // [kVStages]
constexpr int kBarVEmpty = 9;        // [kVStages]
constexpr int kBarVZero = 12;        // [kVStages] a slot's V rows past ctx_len are zeroed
constexpr int kBarQFull = 15;        // the item's Q tile has landed
constexpr int kBarQFreeS = 16;       // the issuer is done with an item's Q tile (one phase per item)
constexpr int kBarQFreeE = 17;       // the epilogue has scored an item's chains (4 warps)
constexpr int kBarSFull = 18;        // [2] S_b computed
constexpr int kBarPFull = 20;        // [2] P over S_b written (4 softmax warps)
constexpr int kBarOFull = 22;        // O holds the item's context partial
constexpr int kBarOEmpty = 23;       // O read by the epilogue (4 warps)
constexpr int kBarStats = 24;        // the item's row max / sum written (4 softmax warps)
constexpr int kBarStatsFree = 25;    // the epilogue has read them (4 warps)
constexpr int kBarPvDone = 26;       // one phase per PV
constexpr int kBarFin = 27;
constexpr int kNumBars = 28;

template <int D>
struct PkCfg {
    static constexpr int kHalves = D / 64;              // 64-element (128-byte) swizzle columns
    static constexpr int kHalfBytes = kBM * 128;        // one 128-row x 64-element half
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    static constexpr int kMisc = kBarOff + kNumBars * 8;     // TMEM base, abort flag
    static constexpr int kStats = kMisc + 16;                // float [m, l][128]
    static constexpr int kUsed = kStats + 2 * kBM * 4;
    static constexpr int kSmem = kUsed + 1024;
    static constexpr int kSCol = 0;                     // S_b at kSCol + b * kBN
    static constexpr int kOCol = 2 * kBN;               // context partial O
    static constexpr int kCCol = 2 * kBN + D;           // chain partial C
};

struct PkParams {
    CtxArgs a;
    int bpt;     // beams per tile
    int tiles;   // tiles per (request, kv head)
    int items;   // R * Hkv * tiles
};

// One work item of this CTA.
struct Item {
    int r, kvh, tile;
    int nb;        // context key blocks (0: no context)
    int tail;      // valid keys of the last block (kBN when it is full)
    bool active;   // the tile has rows of this call (per-request widths)
};

__device__ __forceinline__ Item item_of(const PkParams &p, int k) {
    const Geometry &g = p.a.g;
    Item it;
    it.tile = k % p.tiles;
    const int rk = k / p.tiles;
    it.kvh = rk % g.Hkv;
    it.r = rk / g.Hkv;
    int len = p.a.ctx_len[it.r];
    len = len < 0 ? 0 : (len > g.Lc_max ? g.Lc_max : len);
    it.nb = (len + kBN - 1) / kBN;
    it.tail = len - (it.nb - 1) * kBN;
    it.active = it.tile * p.bpt < width_of(g, it.r, g.step);
    return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    ctx_pk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                  const __grid_constant__ PkParams p) {
    using C = PkCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar0 = sbase + C::kBarOff;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMisc + 4);

    const Geometry &g = p.a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_per_tile = p.bpt * g.G;
    // items of this CTA: k = blockIdx.x + j * gridDim.x, j = 0 .. n_mine - 1
    const int n_mine = p.items > (int)blockIdx.x ? (p.items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto item_k = [&](int j) { return (int)blockIdx.x + j * (int)gridDim.x; };

    if (warp == kKProducerWarp) {
        if (lane == 0) {
            for (int i = 0; i < kKStages; ++i) {
                ptx::mbar_init(bar(kBarKFull + i), 1);
                ptx::mbar_init(bar(kBarKEmpty + i), 1);
            }
            for (int i = 0; i < kVStages; ++i) {
                ptx::mbar_init(bar(kBarVFull + i), 1);
                ptx::mbar_init(bar(kBarVEmpty + i), 1);
                ptx::mbar_init(bar(kBarVZero + i), 1);
            }
            ptx::mbar_init(bar(kBarQFull), 1);
            ptx::mbar_init(bar(kBarQFreeS), 1);
            ptx::mbar_init(bar(kBarQFreeE), 4);
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(bar(kBarSFull + b), 1);
                ptx::mbar_init(bar(kBarPFull + b), 4);
            }
            ptx::mbar_init(bar(kBarOFull), 1);
            ptx::mbar_init(bar(kBarOEmpty), 4);
            ptx::mbar_init(bar(kBarStats), 4);
            ptx::mbar_init(bar(kBarStatsFree), 4);
            ptx::mbar_init(bar(kBarPvDone), 1);
            ptx::mbar_init(bar(kBarFin), 1);
            *abort_flag = 0;
            ptx::fence_mbar_init();
        }
        // rows of a tile past bpt*G are never loaded: keep them zero
        if (rows_per_tile < kBM) {
            const int tail = (kBM - rows_per_tile) * 128;
            for (int h = 0; h < C::kHalves; ++h)
                for (int off = lane * 16; off < tail; off += 32 * 16)
                    *reinterpret_cast<uint4 *>(smem + C::kQOff + h * C::kHalfBytes + rows_per_tile * 128 + off) =
                        make_uint4(0, 0, 0, 0);
        }
        ptx::fence_proxy_async_smem();
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

    if (warp == kKProducerWarp) {
        // ------------------------------------------------------------ Q and K producer
        bool ok = true;
        int u = 0;        // active items so far (one Q load each)
        int n = 0;        // K loads so far (K of global block n)
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_q);
            ptx::prefetch_tmap(&tm_k);
        }
        for (int j = 0; ok && j < n_mine; ++j) {
            const Item it = item_of(p, item_k(j));
            if (!it.active) continue;
            // the Q tile is free once the previous item's chains are scored and
            // the issuer is done with it (its last S has completed)
            if (u > 0 && !(ok = wait_warp(bar(kBarQFreeE), (uint32_t)((u - 1) & 1), abort_flag))) break;
            if (u > 0 && !(ok = wait_warp(bar(kBarQFreeS), (uint32_t)((u - 1) & 1), abort_flag))) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(kBarQFull), (uint32_t)(C::kHalves * rows_per_tile * 128));
                for (int h = 0; h < C::kHalves; ++h)
                    ptx::tma_load_4d(sbase + C::kQOff + h * C::kHalfBytes, &tm_q, bar(kBarQFull), h * 64, it.kvh * g.G,
                                     it.tile * p.bpt, it.r);
            }
            __syncwarp();
            ++u;
            for (int i = 0; ok && i < it.nb; ++i, ++n) {
                const int s = n % kKStages;
                if (!(ok = wait_warp(bar(kBarKEmpty + s), (uint32_t)(((n / kKStages) & 1) ^ 1), abort_flag))) break;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar(kBarKFull + s), (uint32_t)C::kTileBytes);
                    int c1, c3;
                    kv_coords(p.a, it.r, i * kBN, c1, c3);
                    for (int h = 0; h < C::kHalves; ++h)
                        ptx::tma_load_4d(sbase + C::kKOff + s * C::kTileBytes + h * C::kHalfBytes, &tm_k,
                                         bar(kBarKFull + s), h * 64, c1, it.kvh, c3);
                }
                __syncwarp();
            }
        }
        if (!ok) {
            fail();
            // drain: every copy in flight lands before the CTA leaves
            if (u > 0) wait_warp(bar(kBarQFull), (uint32_t)((u - 1) & 1), nullptr);
            for (int m = n - kKStages < 0 ? 0 : n - kKStages; m < n; ++m)
                wait_warp(bar(kBarKFull + m % kKStages), (uint32_t)((m / kKStages) & 1), nullptr);
        }
    } else if (warp == kVProducerWarp) {
        // ------------------------------------------------------------ V producer
        bool ok = true;
        int n = 0;        // V loads so far
        if (lane == 0) ptx::prefetch_tmap(&tm_v);
        for (int j = 0; ok && j < n_mine; ++j) {
            const Item it = item_of(p, item_k(j));
            if (!it.active) continue;
            for (int i = 0; ok && i < it.nb; ++i, ++n) {
                const int s = n % kVStages;
                if (!(ok = wait_warp(bar(kBarVEmpty + s), (uint32_t)(((n / kVStages) & 1) ^ 1), abort_flag))) break;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar(kBarVFull + s), (uint32_t)C::kTileBytes);
                    int c1, c3;
                    kv_coords(p.a, it.r, i * kBN, c1, c3);
                    for (int h = 0; h < C::kHalves; ++h)
                        ptx::tma_load_4d(sbase + C::kVOff + s * C::kTileBytes + h * C::kHalfBytes, &tm_v,
                                         bar(kBarVFull + s), h * 64, c1, it.kvh, c3);
                }
                __syncwarp();
                if (i == it.nb - 1 && it.tail < kBN) {
                    // the last block: context positions past ctx_len hold anything, so
                    // once the V block lands its rows past the end are zeroed (P is 0
                    // there, but 0 * NaN would not be)
                    if (!(ok = wait_warp(bar(kBarVFull + s), (uint32_t)((n / kVStages) & 1), abort_flag))) {
                        ++n;
                        break;
                    }
                    const int bytes = (kBN - it.tail) * 128;
                    for (int h = 0; h < C::kHalves; ++h)
                        for (int off = lane * 16; off < bytes; off += 32 * 16)
                            *reinterpret_cast<uint4 *>(smem + C::kVOff + s * C::kTileBytes + h * C::kHalfBytes +
                                                       it.tail * 128 + off) = make_uint4(0, 0, 0, 0);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(kBarVZero + s));
                }
            }
        }
        if (!ok) {
            fail();
            for (int m = n - kVStages < 0 ? 0 : n - kVStages; m < n; ++m)
                wait_warp(bar(kBarVFull + m % kVStages), (uint32_t)((m / kVStages) & 1), nullptr);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // One lane issues; lanes 1-31 go straight to the final barrier.
        if (lane == 0) {
            constexpr uint32_t kIdescQK = ptx::idesc_bf16(kBM, kBN, 0);
            constexpr uint32_t kIdescPV = ptx::idesc_bf16(kBM, D, 1);
            // Every descriptor is formed once (as in the tile-pair kernel): a
            // k-step of 16 elements moves a K-major 128B-swizzled operand by 32
            // bytes inside the swizzle atom (a whole 64-column half after 4
            // steps), and the N-major V operand by 16 rows = 2048 bytes.
            const uint64_t dq = ptx::smem_desc(sbase + C::kQOff, 16, 1024);
            const uint64_t dk0 = ptx::smem_desc(sbase + C::kKOff, 16, 1024);
            const uint64_t dv0 = ptx::smem_desc(sbase + C::kVOff, C::kHalfBytes, 1024);
            constexpr uint64_t kSlot = C::kTileBytes >> 4;
            auto qk_step = [](int kk) -> uint64_t { return (uint64_t)((kk >> 2) * (C::kHalfBytes >> 4) + (kk & 3) * 2); };
            bool ok = true;
            int sn = 0;   // S issued so far (global block index of the next S)
            // S(sn): the item's first S waits for its Q tile, and its last one
            // frees the Q tile for the next item's load
            auto issue_s = [&](bool first, bool last, int u_q) -> bool {
                if (first && !wait_lane(bar(kBarQFull), (uint32_t)(u_q & 1), abort_flag)) return false;
                const int slot = sn % kKStages;
                if (!wait_lane(bar(kBarKFull + slot), (uint32_t)((sn / kKStages) & 1), abort_flag)) return false;
                ptx::tc_fence_after();
                const uint64_t b0 = dk0 + (uint64_t)slot * kSlot;
                const uint32_t d = tmem + C::kSCol + (uint32_t)(sn & 1) * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) ptx::mma_ss(d, dq + qk_step(kk), b0 + qk_step(kk), kIdescQK, kk > 0);
                ptx::mma_commit(bar(kBarSFull + (sn & 1)));
                ptx::mma_commit(bar(kBarKEmpty + slot));
                if (last) ptx::mma_commit(bar(kBarQFreeS));
                ++sn;
                return true;
            };

            int n = 0;          // global block of the next PV
            int u = 0;          // active items so far (Q phases)
            int zpar = 0;       // bit s: parity of the next zeroing of V slot s
            int oc = 0;         // items with context so far (one O phase each)
            for (int j = 0; ok && j < n_mine; ++j) {
                const Item it = item_of(p, item_k(j));
                if (!it.active) continue;
                if (it.nb == 0) {
                    // no context: nothing to issue, O is not touched.  Its Q phase is
                    // still awaited and released in turn (a commit, so that it completes
                    // after the previous item's last S), keeping both in order.
                    if (!(ok = wait_lane(bar(kBarQFull), (uint32_t)(u & 1), abort_flag))) break;
                    ptx::mma_commit(bar(kBarQFreeS));
                    ++u;
                    continue;
                }
                for (int i = 0; i < it.nb; ++i, ++n) {
                    // S(n) and, within the item, S(n + 1) -- which goes into the S
                    // buffer that PV(n - 1) has read -- before P(n) is awaited
                    if (sn == n && !(ok = issue_s(i == 0, i == it.nb - 1, u))) break;
                    if (sn == n + 1 && i + 1 < it.nb && !(ok = issue_s(false, i + 1 == it.nb - 1, u))) break;
                    if (!(ok = wait_lane(bar(kBarPFull + (n & 1)), (uint32_t)((n >> 1) & 1), abort_flag))) break;
                    // the item's first PV overwrites O: the epilogue must have read the
                    // previous item's
                    if (i == 0 && oc > 0 && !(ok = wait_lane(bar(kBarOEmpty), (uint32_t)((oc - 1) & 1), abort_flag)))
                        break;
                    const int slot = n % kVStages;
                    const bool ragged = (i == it.nb - 1) && it.tail < kBN;
                    // a ragged last block's V is usable once the producer has zeroed its rows past the end
                    if (!(ok = ragged ? wait_lane(bar(kBarVZero + slot), (uint32_t)((zpar >> slot) & 1), abort_flag)
                                      : wait_lane(bar(kBarVFull + slot), (uint32_t)((n / kVStages) & 1), abort_flag)))
                        break;
                    if (ragged) zpar ^= 1 << slot;
                    ptx::tc_fence_after();
                    const uint64_t b0 = dv0 + (uint64_t)slot * kSlot;
                    const uint32_t d = tmem + C::kOCol, a = tmem + C::kSCol + (uint32_t)(n & 1) * kBN;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        ptx::mma_ts(d, a + kk * 8, b0 + (uint64_t)(kk * (2048 >> 4)), kIdescPV, (kk > 0 || i > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(kBarVEmpty + slot));
                    ptx::mma_commit(bar(kBarPvDone));
                    if (i == it.nb - 1) ptx::mma_commit(bar(kBarOFull));
                }
                ++oc;
                ++u;
            }
            if (!ok) fail();
            // no MMA may still be running when the TMEM is released
            ptx::mma_commit(bar(kBarFin));
            wait_lane(bar(kBarFin), 0, nullptr);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ softmax
        const int m_local = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float c = g.scale_log2;
        float *s_stats = reinterpret_cast<float *>(smem + C::kStats);
        const uint32_t tO = tmem + lane_off + (uint32_t)C::kOCol;
        bool ok = true;
        int n = 0;
        int sc = 0;   // items with context so far (one stats phase each)
        for (int j = 0; ok && j < n_mine; ++j) {
            const Item it = item_of(p, item_k(j));
            if (!it.active) continue;
            if (it.nb == 0) continue;   // no context: no blocks, no row statistics
            float m = -INFINITY, l = 0.f;
            for (int i = 0; i < it.nb; ++i, ++n) {
                const int valid = (i == it.nb - 1) ? it.tail : kBN;
                const uint32_t tS = tmem + lane_off + (uint32_t)(C::kSCol + (n & 1) * kBN);
                if (!(ok = wait_warp(bar(kBarSFull + (n & 1)), (uint32_t)((n >> 1) & 1), abort_flag))) break;
                ptx::tc_fence_after();
                uint32_t sv[kBN];
#pragma unroll
                for (int q4 = 0; q4 < kBN / 32; ++q4) ptx::tmem_ld32(tS + 32 * q4, &sv[32 * q4]);
                ptx::tmem_wait_ld();
                if (valid < kBN) {
#pragma unroll
                    for (int jj = 0; jj < kBN; ++jj)
                        if (jj >= valid) sv[jj] = __float_as_uint(-INFINITY);
                }
                auto row_max = [&]() -> float {
                    float mx8[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float mu = fmaxf(__uint_as_float(sv[q]), __uint_as_float(sv[q + 8]));
#pragma unroll
                        for (int k2 = 2; k2 < 16; k2 += 2)
                            mu = ptx::fmax3(mu, __uint_as_float(sv[q + 8 * k2]), __uint_as_float(sv[q + 8 * k2 + 8]));
                        mx8[q] = mu;
                    }
                    return fmaxf(ptx::fmax3(mx8[0], mx8[1], mx8[2]),
                                 fmaxf(ptx::fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                };
                if (i == 0) m = row_max() * c;   // the first block sets the running maximum
                // p = 2^(s*c - m) against the running maximum m; a block sum of at
                // most kSumLimit bounds every p and needs no rescale.  Past it (rare
                // after the first block, or inf/NaN) the exact block maximum is
                // taken, O and l are rescaled (after the previous PV into O has
                // completed) and the pass is redone once.
                float blk = 0.f;
#pragma unroll 1
                for (int pass = 0; pass < 2; ++pass) {
                    const float neg_m = -m;
                    float sa[2] = {0.f, 0.f}, sb[2] = {0.f, 0.f};
#pragma unroll
                    for (int qtr = 0; qtr < 4; ++qtr) {
                        uint32_t pk[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int col = 32 * qtr + 2 * jj;
                            float x0, x1;
                            ptx::ffma2(x0, x1, __uint_as_float(sv[col]), __uint_as_float(sv[col + 1]), c, c, neg_m, neg_m);
                            const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                            ptx::fadd2(sa[jj & 1], sb[jj & 1], sa[jj & 1], sb[jj & 1], p0, p1);
                            pk[jj] = pack_bf16x2(p0, p1);
                        }
                        ptx::tmem_st16(tS + 16 * qtr, pk);
                    }
                    blk = (sa[0] + sa[1]) + (sb[0] + sb[1]);
                    const bool need = pass == 0 && !(blk <= kSumLimit);
                    if (!__any_sync(kFullMask, need)) break;
                    const float m_blk = row_max() * c;
                    const float f = need ? ptx::ex2(m - m_blk) : 1.f;
                    if (i > 0) {
                        // O_b carries the old maximum: once the previous PV into it is done,
                        // rescale it in TMEM.  S(n) was issued behind PV(n - 2), so the phase
                        // before PV(n - 1)'s is complete and the parity wait is exact.
                        if (!(ok = wait_warp(bar(kBarPvDone), (uint32_t)((n - 1) & 1), abort_flag))) break;
                        ptx::tc_fence_after();
#pragma unroll 1
                        for (int q8 = 0; q8 < D / 8; ++q8) {
                            uint32_t ov[8];
                            ptx::tmem_ld8(tO + 8 * q8, ov);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) ov[jj] = __float_as_uint(__uint_as_float(ov[jj]) * f);
                            ptx::tmem_st8(tO + 8 * q8, ov);
                        }
                    }
                    l *= f;
                    if (need) m = m_blk;
                }
                if (!ok) break;
                l += blk;
                // P is in TMEM: each thread's stores complete and are fenced, the
                // warp synchronises, and one lane signals for the warp
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kBarPFull + (n & 1)));
            }
            if (!ok) break;
            // the item's row max and sum for the epilogue, once it has read the previous item's
            if (sc > 0 && !(ok = wait_warp(bar(kBarStatsFree), (uint32_t)((sc - 1) & 1), abort_flag))) break;
            s_stats[m_local] = m;
            s_stats[kBM + m_local] = l;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarStats));
            ++sc;
        }
        if (!ok) fail();
    } else if (warp < kKProducerWarp) {
        // ------------------------------------------------------------ epilogue
        // Every wait here is bounded and its failure only marks the call.
        const int quarter = warp - kEpiWarp0;
        const int m_local = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + (uint32_t)C::kOCol;
        const uint32_t tC = tmem + lane_off + (uint32_t)C::kCCol;
        const float *s_stats = reinterpret_cast<const float *>(smem + C::kStats);
        const uint32_t q_row = sbase + C::kQOff + (uint32_t)m_local * 128u;
        const int swz = m_local & 7;
        // the CTA's last active item writes its rows through the Q tile (free once
        // its last S has completed, with no further Q to load) and TMA stores;
        // earlier items store their rows directly
        int j_last = n_mine - 1;
        while (j_last >= 0 && !item_of(p, item_k(j_last)).active) --j_last;
        int u = 0;
        int sc = 0;     // items with context so far (stats and O phases)
        for (int j = 0; j < n_mine; ++j) {
            const Item it = item_of(p, item_k(j));
            if (!it.active) continue;
            const bool staged = j == j_last;
            const int beam = it.tile * p.bpt + m_local / g.G;
            const bool row_ok = m_local < rows_per_tile && beam < width_of(g, it.r, g.step);
            const long long row = ((long long)it.r * g.W_s + beam) * g.Hq + it.kvh * g.G + m_local % g.G;
            bool ok = wait_warp(bar(kBarQFull), (uint32_t)(u & 1), abort_flag);
            // The per-beam stage, while the item's context loop runs: walk BeamPath
            // back from the row's beam (a_s = b, a_{t-1} = BeamPath[r, t, a_t]),
            // fetching each token's parent index and K row in one round trip, and
            // score the token against the row's query (base-2 units).  A parent
            // outside [0, W_{t-1}) is not followed: the row is flagged and nothing
            // past it is read.  The V rows are prefetched into L2 for the chain partial.
            float x[kMaxTokens];
            int slot_of[kMaxTokens];
            bool chain_ok = true;
            {
                int slot = beam;
#pragma unroll
                for (int tt = kMaxTokens - 1; tt >= 0; --tt) {
                    x[tt] = -INFINITY;
                    slot_of[tt] = 0;
                    if (tt > g.step || !ok || !row_ok || !chain_ok) continue;
                    int par = 0;
                    if (tt > 0) par = __ldg(p.a.beam_path + ((long long)it.r * g.S_max + tt) * g.W_max + slot);
                    const long long kv_off = ((((long long)it.r * g.S_max + tt) * g.W_max + slot) * g.Hkv + it.kvh) * D;
                    const uint4 *kr = reinterpret_cast<const uint4 *>(p.a.beam_k + kv_off);
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.a.beam_v + kv_off));
                    if (D > 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.a.beam_v + kv_off + 64));
                    uint4 kv[D / 8];
#pragma unroll
                    for (int ch = 0; ch < D / 8; ++ch) kv[ch] = __ldg(kr + ch);
                    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
                    for (int ch = 0; ch < D / 8; ++ch) {
                        uint4 qv;
                        const uint32_t addr = q_row + (uint32_t)(ch >> 3) * (kBM * 128) + (uint32_t)(((ch & 7) ^ swz) * 16);
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(qv.x), "=r"(qv.y), "=r"(qv.z), "=r"(qv.w)
                                     : "r"(addr));
                        fma_bf16x2(d0, d1, qv.x, kv[ch].x);
                        fma_bf16x2(d2, d3, qv.y, kv[ch].y);
                        fma_bf16x2(d0, d1, qv.z, kv[ch].z);
                        fma_bf16x2(d2, d3, qv.w, kv[ch].w);
                    }
                    x[tt] = ((d0 + d1) + (d2 + d3)) * g.scale_log2;
                    slot_of[tt] = slot;
                    if (tt > 0) {
                        if (par < 0 || par >= width_of(g, it.r, tt - 1)) chain_ok = false;
                        else slot = par;
                    }
                }
            }
            // the Q tile may be reloaded for the next item
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarQFreeE));
            // The chain's own partial, still while the context loop runs: its
            // maximum m_c, weights w_t = 2^(x_t - m_c) and sum l_c in registers,
            // and C = sum_t w_t v_t in TMEM, one token's V row at a time.  TMEM is
            // read and written by the whole warp; rows without a chain add zeros.
            const bool chain = row_ok && ok && chain_ok;
            float m_c = -INFINITY;
#pragma unroll
            for (int tt = 0; tt < kMaxTokens; ++tt) m_c = fmaxf(m_c, x[tt]);   // unused levels hold -inf
            float w[kMaxTokens];
            float l_c = 0.f;
#pragma unroll
            for (int tt = 0; tt < kMaxTokens; ++tt) {
                w[tt] = chain ? ptx::ex2(x[tt] - m_c) : 0.f;
                l_c += w[tt];
            }
#pragma unroll 1
            for (int tt = 0; tt <= g.step; ++tt) {
                // this token's weight and slot, picked from the register tables
                float wt = w[0];
                int st = slot_of[0];
#pragma unroll
                for (int k = 1; k < kMaxTokens; ++k) {
                    wt = tt == k ? w[k] : wt;
                    st = tt == k ? slot_of[k] : st;
                }
                const uint4 *rv = reinterpret_cast<const uint4 *>(
                    p.a.beam_v + ((((long long)it.r * g.S_max + tt) * g.W_max + st) * g.Hkv + it.kvh) * D);
                uint4 v[D / 8];
#pragma unroll
                for (int ch = 0; ch < D / 8; ++ch) v[ch] = chain ? __ldg(rv + ch) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t acc[32];
                    if (tt > 0) {
                        ptx::tmem_ld32(tC + 32 * q, acc);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint4 &vc = v[4 * q + (e >> 2)];
                        const uint32_t vw = (e & 3) == 0 ? vc.x : (e & 3) == 1 ? vc.y : (e & 3) == 2 ? vc.z : vc.w;
                        acc[2 * e] = __float_as_uint(fmaf(wt, __uint_as_float(vw << 16), __uint_as_float(acc[2 * e])));
                        acc[2 * e + 1] =
                            __float_as_uint(fmaf(wt, __uint_as_float(vw & 0xffff0000u), __uint_as_float(acc[2 * e + 1])));
                    }
                    ptx::tmem_st32(tC + 32 * q, acc);
                }
                ptx::tmem_wait_st();
            }
            // the context partial (items with context only)
            float m_ctx = -INFINITY, l_ctx = 0.f;
            bool have_ctx = false;
            if (it.nb > 0) {
                ok = wait_warp(bar(kBarStats), (uint32_t)(sc & 1), abort_flag) && ok;
                ok = wait_warp(bar(kBarOFull), (uint32_t)(sc & 1), abort_flag) && ok;
                ++sc;
                have_ctx = ok;
                if (have_ctx) {
                    m_ctx = s_stats[m_local];
                    l_ctx = s_stats[kBM + m_local];
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kBarStatsFree));
            }
            if (!ok) fail();
            ptx::tc_fence_after();
            // log-sum-exp merge of the context partial (O, m_ctx, l_ctx) and the
            // chain partial (C, m_c, l_c)
            const bool bad = row_ok && (!ok || !chain_ok);
            const bool good = row_ok && !bad;
            const float m_tot = fmaxf(m_ctx, m_c);
            const float w_ctx = good ? ptx::ex2(m_ctx - m_tot) : 0.f;   // no context: exp2(-inf) = 0
            const float w_ch = good ? ptx::ex2(m_c - m_tot) : 0.f;
            const float L = l_ctx * w_ctx + l_c * w_ch;
            const float inv = good ? 1.f / L : 0.f;
            const float wc = w_ctx * inv, wh = w_ch * inv;
            uint16_t *orow = p.a.out + row * D;
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32], cc[32];
                if (have_ctx) ptx::tmem_ld32(tO + 32 * q, o);
                ptx::tmem_ld32(tC + 32 * q, cc);
                ptx::tmem_wait_ld();
                if (q == D / 32 - 1 && it.nb > 0) {
                    // O is read: the next item with context may accumulate into it
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(kBarOEmpty));
                }
                if (!row_ok) continue;
                uint32_t pk[16];
                if (bad) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = 0x7fc07fc0u;   // NaN marks a row whose chain is broken
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float a0 = have_ctx ? __uint_as_float(o[2 * e]) * wc : 0.f;
                        const float a1 = have_ctx ? __uint_as_float(o[2 * e + 1]) * wc : 0.f;
                        pk[e] = pack_bf16x2(fmaf(__uint_as_float(cc[2 * e]), wh, a0),
                                            fmaf(__uint_as_float(cc[2 * e + 1]), wh, a1));
                    }
                }
                if (staged) {
                    // columns 32q.. of the row: half q/2, 16-byte chunks 4(q&1).. of its
                    // 128-byte swizzled line, as the output tensor map lays a box out
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int chunk = 4 * (q & 1) + k;
                        const uint32_t addr = q_row + (uint32_t)(q >> 1) * (kBM * 128) + (uint32_t)((chunk ^ swz) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * k]),
                                     "r"(pk[4 * k + 1]), "r"(pk[4 * k + 2]), "r"(pk[4 * k + 3])
                                     : "memory");
                    }
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * q);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
            if (staged) {
                // the tile's rows leave by TMA (rows past W_s or past the tile's
                // beams are outside the box or the tensor and are not written)
                ptx::fence_proxy_async_smem();
                ptx::named_bar_sync(1, 4 * 32);
                if (quarter == 0 && lane == 0) {
                    for (int h = 0; h < C::kHalves; ++h)
                        ptx::tma_store_4d(&tm_out, sbase + C::kQOff + h * C::kHalfBytes, h * 64, it.kvh * g.G,
                                          it.tile * p.bpt, it.r);
                    ptx::bulk_commit();
                    ptx::bulk_wait_all();   // the rows are written before the CTA (and its shared memory) ends
                }
            }
            if (row_ok) {
                if (bad) {
                    p.a.lse[row] = __int_as_float(0x7fc00000);
                    if (ok) raise_device_error(p.a.err, kDevErrBadParent);
                } else {
                    p.a.lse[row] = (m_tot + log2f(L)) * kLn2;
                }
            }
            ++u;
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

template <int D>
cudaError_t launch_pk_d(const CtxArgs &a, int bpt, int tiles, int sm_count, cudaStream_t s) {
    using C = PkCfg<D>;
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev < 64 && !attr_set[dev]) {
            e = cudaFuncSetAttribute(ctx_pk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const Geometry &g = a.g;
    CUtensorMap tq, tk, tv, to;
    const uint64_t qd[4] = {(uint64_t)D, (uint64_t)g.Hq, (uint64_t)g.W_s, (uint64_t)g.R};
    const uint64_t qs[3] = {(uint64_t)D * 2, (uint64_t)g.Hq * D * 2, (uint64_t)g.W_s * g.Hq * D * 2};
    const uint32_t qb[4] = {64, (uint32_t)g.G, (uint32_t)bpt, 1};
    const uint64_t rows = a.page_size ? (uint64_t)a.page_size : (uint64_t)g.Lc_max;
    const uint64_t outer = a.page_size ? (uint64_t)a.num_pages : (uint64_t)g.R;
    const uint64_t kd[4] = {(uint64_t)D, rows, (uint64_t)g.Hkv, outer};
    const uint64_t ks[3] = {(uint64_t)D * 2, rows * D * 2, (uint64_t)g.Hkv * rows * D * 2};
    const uint32_t kb[4] = {64, (uint32_t)kBN, 1, 1};
    if (!encode_4d(&tq, a.q, qd, qs, qb) || !encode_4d(&to, a.out, qd, qs, qb)) return cudaErrorInvalidValue;
    if (g.Lc_max > 0) {
        if (!encode_4d(&tk, a.ctx_k, kd, ks, kb) || !encode_4d(&tv, a.ctx_v, kd, ks, kb)) return cudaErrorInvalidValue;
    } else {
        tk = tq;   // no context: never read
        tv = tq;
    }
    PkParams p;
    p.a = a;
    p.bpt = bpt;
    p.tiles = tiles;
    p.items = g.R * g.Hkv * tiles;
    const int grid = p.items < sm_count ? p.items : sm_count;
    ctx_pk_kernel<D><<<grid, kThreads, C::kSmem, s>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace

int pk_max_steps() { return kMaxTokens; }

cudaError_t launch_ctx_pk(const CtxArgs &a, int sm_count, cudaStream_t s) {
    const int bpt = kBM / a.g.G;
    const int tiles = (a.g.W_s + bpt - 1) / bpt;
    if (a.g.D == 128) return launch_pk_d<128>(a, bpt, tiles, sm_count, s);
    return launch_pk_d<64>(a, bpt, tiles, sm_count, s);
}

}  // namespace gr
