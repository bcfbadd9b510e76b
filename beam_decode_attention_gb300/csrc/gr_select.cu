// gr_select.cu -- beam selection after a decode forward: log_softmax over
// every active beam's logits, plus the beam's cumulative score, and the W'
// best candidates of each request (SID-GR README, section 10 "TODO and
// Roadmap": log_softmax + topK + beam selection on the device; xGR review,
// "xBeam": one size-BW selection over all beams' candidates).
//
//   score[r, b, v] = S[r, b] + (z[r, b, v] - (m_b + ln sum_v exp(z[r, b, v] - m_b)))
//
// in fp32; candidates are ordered by score descending, then by the flat
// index b * V + v ascending, and the first W' of each request give the next
// BeamPath row (parents), the tokens and the new cumulative scores.
//
// Kernel 1 (select_rows_kernel), one CTA per beam row at a time, several CTAs
// per SM, grid-strided over the rows; every row is read from HBM once:
//   the first logits of the row (held in registers) set a threshold, about
//                 twice the share of the row's L best (L = min(W', V)) that
//                 a prefix of that length holds, by a histogram of their
//                 ordered bit patterns and a refinement inside its boundary bin;
//                 or, once the request has a bound on its W'-th score (below),
//                 a threshold guessed from the bound and the row's estimated
//                 log-normaliser;
//   the stream    gives the row's maximum and sum of exponentials and keeps
//                 every logit at or above the threshold in shared memory;
//   the select    turns the kept logits into scores and finds the row's L-th
//                 score among them; when the kept set provably holds every
//                 logit that can reach that score (at least L kept, within
//                 the slots, and the threshold's predecessor scoring below
//                 it), the kept candidates that can still be selected are
//                 sorted by (score desc, v asc) and written to the workspace.
//   A row whose kept set is not provably complete (a skewed prefix, ties,
//   peaked or degenerate logits) takes an exact radix select on the scores
//   over the whole row instead (more passes, same result).
// Each row also publishes lower bounds on its request's W'-th score key
// (valid when L = W'):
//   its L-th score key (atomicMax per request): that row alone holds W'
//                 candidates at or above it;
//   its k-th score key into slot b mod m of m per-request slots (atomicMax,
//                 k = ceil(W' / m)): m distinct rows then hold m * k >= W'
//                 candidates at or above the smallest slot, once every slot
//                 is set.
// A row that finds the bound above every score its threshold can have left
// out keeps the candidates at or above the bound without selecting its own
// L-th (most rows after each request's first ones).
// Kernel 2 (select_merge_kernel), one CTA per request: a tighter bound from
// the first keys of every list; each sorted list's prefix at or above it; the
// W'-th largest score over those prefixes by a radix select in shared
// memory; the candidates above it plus the tied ones in flat-index order;
// and a final sort by (score desc, flat index asc).
#include <cstdint>
#include <mutex>

#include "gr_common.cuh"
#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kRowThreads = 256;
constexpr int kRowBlocksPerSm = 4;    // row CTAs resident per SM
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kCap = 4096;            // candidate slots per row in shared memory
constexpr int kSide = kHistBins / 2;  // 8-byte entries the histogram's space holds
constexpr int kMergeThreads = 1024;
constexpr int kMaxSel = 1024;         // GR_SELECT_MAX_WIDTH
constexpr int kBoundSlots = 32;       // per-request slots of rows' k-th score keys
constexpr float kGuessMargin = 0.5f;  // slack of the guessed threshold (logit units)

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)

// 2^x on the MUFU unit (ex2.approx)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Order-preserving map of an fp32 value to uint32 (-0 taken as +0).
__device__ __forceinline__ uint32_t ord_key(float x) {
    if (x == 0.f) x = 0.f;
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct RowArgs {
    const float *logits;
    const float *beam_scores;
    unsigned long long *lists;   // [R * W_s][L] (score key << 32 | ~v), sorted descending
    int *plen;                   // [R * W_s] entries written to each list (<= L)
    unsigned *tau_lb;            // [R] lower bound on each request's W'-th score key (null: none)
    unsigned *tau_slot;          // [R][nslot] rows' slot_k-th score keys, by beam mod nslot
    int nslot, slot_k;           // nslot * slot_k >= W'
    int rows, W, V, L;
};

// The fp32 score of logit z in a row with log-normaliser c and beam score S:
// fl(S + fl(z - c)); monotone (non-decreasing) in z.
__device__ __forceinline__ float score_of(float z, float c, float S) { return S + (z - c); }

// Visit z = row[v] for v in [0, V): 16-byte loads where the row allows, in
// groups of eight per thread so that several loads are in flight.
template <typename F>
__device__ __forceinline__ void for_row(const float *row, int V, F &&f) {
    const int head = min(V, (int)(((16 - (reinterpret_cast<uintptr_t>(row) & 15)) & 15) >> 2));
    for (int v = threadIdx.x; v < head; v += blockDim.x) f(__ldg(row + v), v);
    const float4 *row4 = reinterpret_cast<const float4 *>(row + head);
    const int n4 = (V - head) >> 2;
    constexpr int kU = 8;
    int i = threadIdx.x;
    for (; i + (kU - 1) * (int)blockDim.x < n4; i += kU * blockDim.x) {
        float4 x[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) x[u] = __ldg(row4 + i + u * blockDim.x);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int v = head + 4 * (i + u * blockDim.x);
            f(x[u].x, v);
            f(x[u].y, v + 1);
            f(x[u].z, v + 2);
            f(x[u].w, v + 3);
        }
    }
    for (; i < n4; i += blockDim.x) {
        const float4 x = __ldg(row4 + i);
        const int v = head + 4 * i;
        f(x.x, v);
        f(x.y, v + 1);
        f(x.z, v + 2);
        f(x.w, v + 3);
    }
    for (int v = head + 4 * n4 + threadIdx.x; v < V; v += blockDim.x) f(__ldg(row + v), v);
}

// Online (max, sum of exp) pair; -inf logits add nothing.
struct MaxSum {
    float m, s;
};
__device__ __forceinline__ MaxSum ms_add(MaxSum a, float z) {
    if (z == -INFINITY) return a;
    if (z > a.m) {
        a.s = a.s * __expf(a.m - z) + 1.f;   // a.m = -inf: 0 * ... = 0
        a.m = z;
    } else {
        a.s += __expf(z - a.m);
    }
    return a;
}
__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b) {
    if (b.m == -INFINITY) return a;
    if (a.m == -INFINITY) return b;
    const float m = fmaxf(a.m, b.m);
    return {m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}

// Exclusive prefix sum over the block in thread order (all threads take part);
// `red` holds one int per warp; returns the block total in *total.
__device__ __forceinline__ int block_excl_scan(int x, int *red, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) red[warp] = inc;
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < nw; ++w) {
        if (w < warp) base += red[w];
        tot += red[w];
    }
    *total = tot;
    return base + inc - x;
}

// Given a histogram (kHistBins counts, highest key bin last), the bin holding
// the need-th largest element and the count of elements in higher bins.
// Each thread owns kHistBins / blockDim consecutive bins.
__device__ __forceinline__ void find_bin(const int *hist, int need, int *red, int *s_bin, int *s_above) {
    const int per = kHistBins / blockDim.x;
    const int hi = kHistBins - 1 - threadIdx.x * per;   // this thread's bins: hi, hi-1, ..., hi-per+1
    int mine = 0;
    for (int k = 0; k < per; ++k) mine += hist[hi - k];
    int total;
    const int above = block_excl_scan(mine, red, &total);   // elements in higher bins than this thread's
    if (above < need && above + mine >= need) {
        int acc = above;
        for (int k = 0; k < per; ++k) {
            const int c = hist[hi - k];
            if (acc + c >= need) {
                *s_bin = hi - k;
                *s_above = acc;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

// Descending bitonic sort of n (a power of two) 64-bit values in shared memory.
__device__ __forceinline__ void bitonic_desc(unsigned long long *a, int n) {
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const unsigned long long x = a[i], y = a[p];
                    if (((i & k) == 0) ? (x < y) : (x > y)) {
                        a[i] = y;
                        a[p] = x;
                    }
                }
            }
            __syncthreads();
        }
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
    const uint32_t lo = __shfl_xor_sync(kFullMask, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(kFullMask, (uint32_t)(v >> 32), m);
    return ((unsigned long long)hi << 32) | lo;
}

// The same descending bitonic sort with the elements in registers: thread t
// holds elements t + q * blockDim (q < n / blockDim, or one element for
// t < n when n <= blockDim), exchanges at strides below 32 are warp shuffles
// (no barrier) and larger strides go through shared memory.  n is a power of
// two, 64 <= n <= 4 * blockDim, blockDim a multiple of 32.
__device__ __forceinline__ void bitonic_desc_shfl(unsigned long long *a, int n) {
    constexpr int kMaxPer = 4;
    const int bd = blockDim.x, t = threadIdx.x, lane = t & 31;
    const int per = n > bd ? n / bd : 1;
    const bool active = t < n;   // n >= 64 is a multiple of 32: whole warps are in or out
    unsigned long long x[kMaxPer];
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q) x[q] = (q < per && active) ? a[t + q * bd] : 0ull;
    for (int k = 2; k <= n; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            if (jj >= 32) {
                __syncthreads();   // the previous stage's reads are done
#pragma unroll
                for (int q = 0; q < kMaxPer; ++q)
                    if (q < per && active) a[t + q * bd] = x[q];
                __syncthreads();
#pragma unroll
                for (int q = 0; q < kMaxPer; ++q) {
                    if (!(q < per && active)) continue;
                    const int i = t + q * bd, pi = i ^ jj;
                    const unsigned long long o = a[pi];
                    const bool take_max = ((i & k) == 0) == (i < pi);
                    x[q] = take_max ? (o > x[q] ? o : x[q]) : (o < x[q] ? o : x[q]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < kMaxPer; ++q) {
                    if (q >= per) continue;   // uniform across the block
                    const int i = t + q * bd;
                    const unsigned long long o = shfl_xor_u64(x[q], jj);
                    const bool take_max = ((i & k) == 0) == ((lane & jj) == 0);
                    x[q] = take_max ? (o > x[q] ? o : x[q]) : (o < x[q] ? o : x[q]);
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q)
        if (q < per && active) a[t + q * bd] = x[q];
    __syncthreads();
}

// The same descending bitonic sort with EPT consecutive elements per thread
// (thread t holds elements t * EPT .. t * EPT + EPT - 1, threads t < n / EPT):
// the strides below EPT are compare-exchanges inside a thread, those below
// 32 * EPT warp shuffles with lane t ^ (stride / EPT), and only the larger
// ones (n > 32 * EPT) go through shared memory and a block barrier, where
// element e of thread t sits at a[e * T + t] (T = n / EPT) so that a warp's
// accesses fall on consecutive words.  All threads of the block call it; n
// is a power of two with 32 * EPT <= n <= EPT * blockDim.  Not inlined: in
// the row kernel (64 registers a thread) inlining it cost spills elsewhere.
template <int EPT>
__device__ __noinline__ void bitonic_desc_blocked(unsigned long long *a, int n) {
    const int t = threadIdx.x, lane = t & 31, T = n / EPT;
    const bool active = t < T;   // whole warps (T is a multiple of 32)
    unsigned long long x[EPT];
    if (active) {
        const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(a + t * EPT);
#pragma unroll
        for (int q = 0; q < EPT / 2; ++q) {
            const ulonglong2 v = src[q];
            x[2 * q] = v.x;
            x[2 * q + 1] = v.y;
        }
    }
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j >= EPT; j >>= 1) {
            const int m = j / EPT;   // partner thread t ^ m
            if (m < 32) {
                if (active) {
                    const bool lower = (lane & m) == 0;
#pragma unroll
                    for (int e = 0; e < EPT; ++e) {
                        const unsigned long long o = shfl_xor_u64(x[e], m);
                        const bool take_max = (((t * EPT + e) & k) == 0) == lower;
                        x[e] = take_max ? (o > x[e] ? o : x[e]) : (o < x[e] ? o : x[e]);
                    }
                }
            } else {
                __syncthreads();   // the previous exchange's reads (and the initial loads) are done
                if (active) {
#pragma unroll
                    for (int e = 0; e < EPT; ++e) a[e * T + t] = x[e];
                }
                __syncthreads();
                if (active) {
                    const bool lower = (t & m) == 0;
#pragma unroll
                    for (int e = 0; e < EPT; ++e) {
                        const unsigned long long o = a[e * T + (t ^ m)];
                        const bool take_max = (((t * EPT + e) & k) == 0) == lower;
                        x[e] = take_max ? (o > x[e] ? o : x[e]) : (o < x[e] ? o : x[e]);
                    }
                }
            }
        }
        // the strides below EPT, inside each thread (compile-time indices)
        if (active) {
#pragma unroll
            for (int jj = EPT / 2; jj > 0; jj >>= 1) {
                if (jj >= k) continue;
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    if ((e ^ jj) <= e) continue;
                    const bool desc = ((t * EPT + e) & k) == 0;
                    const unsigned long long lo = x[e], hi = x[e ^ jj];
                    const bool sw = desc ? lo < hi : lo > hi;
                    x[e] = sw ? hi : lo;
                    x[e ^ jj] = sw ? lo : hi;
                }
            }
        }
    }
    __syncthreads();
    if (active) {
        ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(a + t * EPT);
#pragma unroll
        for (int q = 0; q < EPT / 2; ++q) dst[q] = make_ulonglong2(x[2 * q], x[2 * q + 1]);
    }
    __syncthreads();
}

// Descending sort of n (a power of two) values: in registers where the
// shuffle form takes n, else the shared-memory network.
__device__ __forceinline__ void sort_desc(unsigned long long *a, int n) {
    if (n >= 64 && n <= 4 * (int)blockDim.x) bitonic_desc_shfl(a, n);
    else bitonic_desc(a, n);
}

// The same with four consecutive elements per thread where n allows.
__device__ __forceinline__ void sort_desc_blocked(unsigned long long *a, int n) {
    if (n >= 128 && n <= 4 * (int)blockDim.x) bitonic_desc_blocked<4>(a, n);
    else sort_desc(a, n);
}

__device__ __forceinline__ unsigned long long pack(uint32_t key, uint32_t low) {
    return ((unsigned long long)key << 32) | low;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the one ahead of it has finished, and
// waits here until that grid has completed and its writes are visible (a
// no-op when launched without it); a kernel lets the next one start early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Keeps the entries e of a[0, n) with keep(e), transformed by xf(e), at the
// front of a, in their order (chunk by chunk, a block-wide scan each);
// returns the count (every thread).
template <typename Keep, typename Xf>
__device__ __forceinline__ int compact(unsigned long long *arr, int n, int *red, Keep &&keep, Xf &&xf) {
    int kept = 0;
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const unsigned long long e = i < n ? arr[i] : 0ull;
        const int f = (i < n && keep(e)) ? 1 : 0;
        int tot;
        const int pos = block_excl_scan(f, red, &tot);   // synchronises before any write below
        if (f) arr[kept + pos] = xf(e);
        kept += tot;
        __syncthreads();
    }
    return kept;
}

__device__ __noinline__ void find_bin_call(const int *hist, int need, int *red, int *s_bin, int *s_above);

// The need-th largest key among cand[0, n) (high 32 bits), by a radix select
// in shared memory (12 + 12 + 8 bits); every thread gets it.  kCalls: the bin
// searches as calls (the per-row kernel's form, see find_bin_call).
template <bool kCalls = false>
__device__ __forceinline__ uint32_t radix_kth(const unsigned long long *cand, int n, int need, int *hist, int *red,
                                              int *s_bin, int *s_above) {
    uint32_t prefix = 0, mask = 0;
    const int shifts[3] = {20, 8, 0}, widths[3] = {12, 12, 8};
#pragma unroll
    for (int rd = 0; rd < 3; ++rd) {
        for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const int sh = shifts[rd];
        const uint32_t bm = (1u << widths[rd]) - 1u;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t k = (uint32_t)(cand[i] >> 32);
            if ((k & mask) == prefix) atomicAdd(&hist[kHistBins - 1 - (int)(bm - ((k >> sh) & bm))], 1);
        }
        __syncthreads();
        if (kCalls) find_bin_call(hist, need, red, s_bin, s_above);
        else find_bin(hist, need, red, s_bin, s_above);
        need -= *s_above;
        prefix |= (bm - (uint32_t)(kHistBins - 1 - *s_bin)) << sh;
        mask |= bm << sh;
        __syncthreads();
    }
    return prefix;
}

// Out-of-line copies for the per-row kernel (64 registers a thread): as calls
// they leave the row's stream its registers, and that kernel measured 5 %
// faster so; the merge kernel keeps them inlined (it measured slower as calls).
__device__ __noinline__ void find_bin_call(const int *hist, int need, int *red, int *s_bin, int *s_above) {
    find_bin(hist, need, red, s_bin, s_above);
}
__device__ __noinline__ uint32_t radix_kth_call(const unsigned long long *cand, int n, int need, int *hist, int *red,
                                               int *s_bin, int *s_above) {
    return radix_kth<true>(cand, n, need, hist, red, s_bin, s_above);
}

// The exact candidate set of a row without a usable threshold: the L-th
// largest score key of the whole row by a radix select over the row itself
// (three more reads of it), then every larger score plus the tied ones in
// ascending v, into cand; returns their count (at most L).
__device__ __forceinline__ int exact_candidates(const float *z, int V, int L, float c, float S,
                                                unsigned long long *cand, int *hist, int *red, int *s_bin,
                                                int *s_above, int *s_cnt) {
    uint32_t prefix = 0, mask = 0;
    int need = L;
    const int shifts[3] = {20, 8, 0}, widths[3] = {12, 12, 8};
#pragma unroll
    for (int rd = 0; rd < 3; ++rd) {
        for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const int sh = shifts[rd];
        const uint32_t bm = (1u << widths[rd]) - 1u;
        for_row(z, V, [&](float x, int) {
            const uint32_t k = ord_key(score_of(x, c, S));
            // bins are placed at the top of the histogram so find_bin's
            // highest-first walk works for 8-bit rounds too
            if ((k & mask) == prefix) atomicAdd(&hist[kHistBins - 1 - (int)(bm - ((k >> sh) & bm))], 1);
        });
        __syncthreads();
        find_bin_call(hist, need, red, s_bin, s_above);
        const uint32_t digit = bm - (uint32_t)(kHistBins - 1 - *s_bin);
        need -= *s_above;
        prefix |= digit << sh;
        mask |= bm << sh;
        __syncthreads();
    }
    const uint32_t kstar = prefix;
    if (threadIdx.x == 0) *s_cnt = 0;
    __syncthreads();
    // larger keys (fewer than L) in any order; ties in ascending v, chunk by
    // chunk so that the order is kept
    int taken = 0;
    for (int base = 0; base < V; base += blockDim.x) {
        const int v = base + threadIdx.x;
        const float x = v < V ? __ldg(z + v) : -INFINITY;
        const uint32_t k = v < V ? ord_key(score_of(x, c, S)) : 0u;
        if (v < V && k > kstar) {
            const int slot = atomicAdd(s_cnt, 1);
            if (slot < kCap) cand[slot] = pack(k, ~(uint32_t)v);
        }
        const int tie = (v < V && k == kstar) ? 1 : 0;
        int tot;
        const int rank = block_excl_scan(tie, red, &tot);
        if (tie && taken + rank < need) {
            const int slot = atomicAdd(s_cnt, 1);
            if (slot < kCap) cand[slot] = pack(k, ~(uint32_t)v);
        }
        taken += tot;
        if (taken >= need) {
            // the remaining larger keys still have to be gathered
            for (int v2 = base + blockDim.x + threadIdx.x; v2 < V; v2 += blockDim.x) {
                const uint32_t k2 = ord_key(score_of(__ldg(z + v2), c, S));
                if (k2 > kstar) {
                    const int slot = atomicAdd(s_cnt, 1);
                    if (slot < kCap) cand[slot] = pack(k2, ~(uint32_t)v2);
                }
            }
            break;
        }
    }
    __syncthreads();
    return min(*s_cnt, kCap);
}

// The row's log-normaliser and candidates in one read of the row.
//   1. The first kFirst * blockDim logits (in registers) set the threshold:
//      the exact need_s-th largest of them (a 12-bit histogram, then a
//      12-bit refinement inside the boundary bin), need_s about twice the
//      share of the row's L best that a prefix of this size holds (L when
//      the prefix is the whole row).
//   2. The rest of the row streams from HBM once: running maximum and sum of
//      exponentials (chunk maximum first, one rescale per chunk at most),
//      and every logit at or above the threshold is kept as (logit key, ~v).
//   3. With the log-normaliser c known, the candidates' logit keys become
//      score keys and the row's L-th largest score key kl is found among
//      them.  The set is exact when it holds at least L entries, fits its
//      slots, and kl is above the score of the largest float below the
//      threshold (a logit outside the set can then neither beat nor tie
//      kl, the score being monotone in the logit).  Otherwise the row takes
//      exact_candidates (more reads of the row, same result).
// Then, as before: only candidates at or above max(kl, the request's
// published bound) are kept, sorted by (score desc, v asc) and written; the
// row publishes kl.  Several CTAs share an SM, so one row's select and sort
// overlap another row's stream.
constexpr int kFirst = 16;   // logits per thread in the threshold prefix
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kWarpCap = kCap / kRowWarps;   // candidate slots of each warp's region

// Warp-wide: the lanes' `cnt` candidates get consecutive slots of this warp's
// region (one shared-memory atomic per warp); returns the lane's first slot
// (unbounded: slots past kWarpCap are not stored, the count records them).
__device__ __forceinline__ int warp_slots(int cnt, int *wcnt) {
    const int lane = threadIdx.x & 31;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(kFullMask, incl, 31);
    int base = 0;
    if (lane == 31 && total > 0) base = atomicAdd(wcnt, total);
    base = __shfl_sync(kFullMask, base, 31);
    return base + incl - cnt;
}

// Warp 0 reads the request's bound so far: the largest published L-th key,
// and the smallest slot once every slot is set (0: none).
__device__ __forceinline__ void read_bound(const RowArgs &a, int row, unsigned *out) {
    const int lane = threadIdx.x & 31;
    const int req = row / a.W;
    uint32_t v = lane < a.nslot ? *reinterpret_cast<volatile unsigned *>(a.tau_slot + req * a.nslot + lane) : ~0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFullMask, v, o));
    if (lane == 0) {
        const uint32_t l = *reinterpret_cast<volatile unsigned *>(a.tau_lb + req);
        *out = max(a.nslot > 0 ? v : 0u, l);
    }
}

__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSm) select_rows_kernel(RowArgs a) {
    extern __shared__ unsigned long long sel_smem[];
    unsigned long long *cand = sel_smem;                          // [kCap]
    int *hist = reinterpret_cast<int *>(cand + kCap);             // [kHistBins]
    int *red = hist + kHistBins;                                  // [32]
    __shared__ MaxSum s_ms[kRowThreads / 32];
    __shared__ int s_bin, s_above, s_cnt;
    __shared__ int s_wcnt[kRowWarps];   // candidates of each warp's region
    __shared__ float s_c;
    __shared__ unsigned s_lb;
    __shared__ int s_npre;
    __shared__ float s_cpre, s_corr;   // the prefix's log-normaliser; c - c_pre of the last row with a bound
    const int warp = threadIdx.x >> 5;
    unsigned long long *wreg = cand + warp * kWarpCap;   // this warp's region
    if (threadIdx.x == 0) s_corr = 0.f;

    for (int row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const float *z = a.logits + (long long)row * a.V;
        const float S = a.beam_scores[row];
        const int F = min(a.V, kFirst * (int)blockDim.x);

        // 1. the threshold from the prefix [0, F)
        float xf[kFirst];
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < kFirst; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            xf[k] = v < F ? __ldg(z + v) : -INFINITY;
            mt = fmaxf(mt, xf[k]);
        }
        for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
        if (threadIdx.x < kRowWarps) s_wcnt[threadIdx.x] = 0;
        if (threadIdx.x == 0) s_npre = 0;
        if (a.tau_lb && warp == 0) read_bound(a, row, &s_lb);
        __syncthreads();
        // the prefix's exponentials, against the thread's maximum so far
        float acc = 0.f;
        if (mt != -INFINITY) {
            const float off = -mt * kLog2e;
#pragma unroll
            for (int k = 0; k < kFirst; ++k) acc += ex2_approx(fmaf(xf[k], kLog2e, off));
        }
        // With a bound on the request's W'-th score, the threshold is guessed
        // from it: a logit reaches the bound when z >= bound - S + c, and the
        // row's log-normaliser c is estimated as the prefix's c_pre plus the
        // difference c - c_pre this CTA saw on its last row that had a bound
        // (0 before: c >= c_pre, so that guess is always safe), less a
        // margin.  The guess is taken when the prefix predicts at most kCap / 2
        // candidates for the row, otherwise the histogram's threshold; either
        // way the completeness check after the stream decides with the row's
        // own c (a guess set too high fails it, and the row takes the exact
        // path).
        float tau = -INFINITY;
        bool by_bound = false;
        const uint32_t lb0 = a.tau_lb ? s_lb : 0u;
        if (lb0 != 0u && a.V > F) {
            MaxSum ms{mt, acc};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                MaxSum other{__shfl_xor_sync(kFullMask, ms.m, o), __shfl_xor_sync(kFullMask, ms.s, o)};
                ms = ms_merge(ms, other);
            }
            if ((threadIdx.x & 31) == 0) s_ms[warp] = ms;
            __syncthreads();
            if (threadIdx.x == 0) {
                MaxSum t = s_ms[0];
                for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = ms_merge(t, s_ms[w]);
                s_cpre = t.m + __logf(t.s);
                s_c = s_cpre + s_corr;
            }
            __syncthreads();
            const float lbs = key_float(lb0), ce = s_c;
            const float tb = (lbs - S + ce) - (kGuessMargin + 1e-3f * (fabsf(lbs) + fabsf(S) + fabsf(ce)));
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < kFirst; ++k) cnt += (threadIdx.x + k * (int)blockDim.x < F && xf[k] >= tb) ? 1 : 0;
            cnt = __reduce_add_sync(kFullMask, cnt);
            if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(&s_npre, cnt);
            __syncthreads();
            by_bound = isfinite(tb) && (long long)s_npre * a.V <= (long long)(kCap / 2) * F;
            tau = tb;
        }
        if (!by_bound) {
#pragma unroll
            for (int k = 0; k < kFirst; ++k)
                if (threadIdx.x + k * (int)blockDim.x < F) atomicAdd(&hist[ord_key(xf[k]) >> (32 - kHistBits)], 1);
            __syncthreads();
            const int need_s = a.V <= F ? a.L : min(F, 2 * (int)(((long long)F * a.L + a.V - 1) / a.V) + 16);
            find_bin_call(hist, need_s, red, &s_bin, &s_above);
            const uint32_t b_hi = (uint32_t)s_bin;
            const int need_lo = need_s - s_above;
            __syncthreads();
            for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kFirst; ++k) {
                const uint32_t key = ord_key(xf[k]);
                if (threadIdx.x + k * (int)blockDim.x < F && (key >> 20) == b_hi) atomicAdd(&hist[(key >> 8) & 0xfffu], 1);
            }
            __syncthreads();
            find_bin_call(hist, need_lo, red, &s_bin, &s_above);
            const uint32_t tau_key = (b_hi << 20) | ((uint32_t)s_bin << 8);
            // keys at or below 0x7fffff hold -inf and NaN patterns: no threshold there
            tau = tau_key <= 0x7fffffu ? -INFINITY : key_float(tau_key);
        }
        {
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < kFirst; ++k) cnt += (threadIdx.x + k * (int)blockDim.x < F && xf[k] >= tau) ? 1 : 0;
            int slot = warp_slots(cnt, &s_wcnt[warp]);
#pragma unroll
            for (int k = 0; k < kFirst; ++k) {
                const int v = threadIdx.x + k * blockDim.x;
                if (v < F && xf[k] >= tau) {
                    if (slot < kWarpCap) wreg[slot] = pack(ord_key(xf[k]), ~(uint32_t)v);
                    ++slot;
                }
            }
        }

        // 2. the rest of the row, once: 16-byte loads where the row allows
        {
            const float *zr = z + F;
            const int Vr = a.V - F;
            const int head = min(Vr, (int)(((16 - (reinterpret_cast<uintptr_t>(zr) & 15)) & 15) >> 2));
            const int n4 = (Vr - head) >> 2, tail = head + 4 * n4;
            auto one = [&](float x, int v) {   // a logit outside the 16-byte body
                if (x > mt) {
                    acc = (mt == -INFINITY ? 0.f : acc * ex2_approx((mt - x) * kLog2e)) + 1.f;
                    mt = x;
                } else if (x != -INFINITY) {
                    acc += ex2_approx((x - mt) * kLog2e);
                }
                if (x >= tau) {
                    const int slot = atomicAdd(&s_wcnt[warp], 1);
                    if (slot < kWarpCap) wreg[slot] = pack(ord_key(x), ~(uint32_t)v);
                }
            };
            for (int v = threadIdx.x; v < head; v += blockDim.x) one(__ldg(zr + v), F + v);
            for (int v = tail + threadIdx.x; v < Vr; v += blockDim.x) one(__ldg(zr + v), F + v);
            const float4 *row4 = reinterpret_cast<const float4 *>(zr + head);
            // kU 16-byte loads per thread per step, and the next step's loads
            // issued before this step's logits are used (2 * kU in flight)
            constexpr int kU = 4;
            const int step = kU * blockDim.x;
            auto load = [&](float4 (&x)[kU], int c0) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = c0 + threadIdx.x + u * blockDim.x;
                    x[u] = i < n4 ? __ldg(row4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
            };
            auto use = [&](const float4 (&x)[kU], int c0) {
                float cm = -INFINITY;
#pragma unroll
                for (int u = 0; u < kU; ++u) cm = fmaxf(cm, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)));
                if (cm > mt) {
                    acc = mt == -INFINITY ? 0.f : acc * ex2_approx((mt - cm) * kLog2e);
                    mt = cm;
                }
                if (mt != -INFINITY) {
                    const float off = -mt * kLog2e;
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        acc += (ex2_approx(fmaf(x[u].x, kLog2e, off)) + ex2_approx(fmaf(x[u].y, kLog2e, off))) +
                               (ex2_approx(fmaf(x[u].z, kLog2e, off)) + ex2_approx(fmaf(x[u].w, kLog2e, off)));
                }
                // only lanes whose step holds a candidate take this path (about a
                // quarter of them): one atomic on the warp's own counter per lane,
                // then the lane's candidates in order (the -inf fill past the
                // body is never a candidate, even when the threshold is -inf)
                if (cm >= tau) {
                    int cnt = 0;
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        if (c0 + (int)threadIdx.x + u * (int)blockDim.x < n4)
                            cnt += (x[u].x >= tau) + (x[u].y >= tau) + (x[u].z >= tau) + (x[u].w >= tau);
                    if (cnt > 0) {
                        int slot = atomicAdd(&s_wcnt[warp], cnt);
#pragma unroll
                        for (int u = 0; u < kU; ++u) {
                            const int i4 = c0 + threadIdx.x + u * blockDim.x;
                            const int v = F + head + 4 * i4;
                            const float q[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (i4 < n4 && q[e] >= tau) {
                                    if (slot < kWarpCap) wreg[slot] = pack(ord_key(q[e]), ~(uint32_t)(v + e));
                                    ++slot;
                                }
                        }
                    }
                }
            };
            float4 xa[kU], xb[kU];
            load(xa, 0);
            for (int c0 = 0; c0 < n4; c0 += 2 * step) {
                load(xb, c0 + step);
                use(xa, c0);
                if (c0 + step >= n4) break;
                load(xa, c0 + 2 * step);
                use(xb, c0 + step);
            }
        }
        MaxSum ms{mt, acc};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            MaxSum other{__shfl_xor_sync(kFullMask, ms.m, o), __shfl_xor_sync(kFullMask, ms.s, o)};
            ms = ms_merge(ms, other);
        }
        if ((threadIdx.x & 31) == 0) s_ms[threadIdx.x >> 5] = ms;
        __syncthreads();
        if (threadIdx.x == 0) {
            MaxSum t = s_ms[0];
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = ms_merge(t, s_ms[w]);
            s_c = t.m + __logf(t.s);   // log-normaliser c_b
            // the prefix's share of the normaliser, for the next row's guess
            if (lb0 != 0u && a.V > F && isfinite(s_c - s_cpre)) s_corr = s_c - s_cpre;
        }
        __syncthreads();
        const float c = s_c;
        // the warps' regions become one array: every warp reads its entries
        // into registers, and after a barrier writes them at its offset
        int n = 0, off = 0;
        bool overflow = false;
        for (int w = 0; w < kRowWarps; ++w) {
            const int cw = s_wcnt[w];
            overflow |= cw > kWarpCap;
            if (w < warp) off += min(cw, kWarpCap);
            n += min(cw, kWarpCap);
        }
        {
            constexpr int kPer = kWarpCap / 32;
            const int lane = threadIdx.x & 31, cw = min(s_wcnt[warp], kWarpCap);
            unsigned long long ent[kPer];
#pragma unroll
            for (int j = 0; j < kPer; ++j) ent[j] = lane + 32 * j < cw ? wreg[lane + 32 * j] : 0ull;
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kPer; ++j)
                if (lane + 32 * j < cw) cand[off + lane + 32 * j] = ent[j];
            __syncthreads();
        }
        if (overflow) n = kCap + 1;

        // the request's bound so far: the largest published L-th key, and the
        // smallest slot once every slot is set (0: none)
        uint32_t lb = 0u;
        if (a.tau_lb) {
            if (warp == 0) read_bound(a, row, &s_lb);
            __syncthreads();
            lb = s_lb;
        }

        // 3. score keys; the bound settles the row when every logit below the
        // threshold scores below it (then the kept set holds every candidate
        // at or above the bound); otherwise the row's L-th, and whether the
        // set is exact
        uint32_t kl = 0u;
        bool settled = lb != 0u && n <= kCap;
        if (settled && tau != -INFINITY) settled = lb > ord_key(score_of(nextafterf(tau, -INFINITY), c, S));
        bool exact = settled || (n >= a.L && n <= kCap);
        if (exact) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const unsigned long long e = cand[i];
                cand[i] = pack(ord_key(score_of(key_float((uint32_t)(e >> 32)), c, S)), (uint32_t)e);
            }
            __syncthreads();
        }
        if (exact && !settled) {
            kl = radix_kth_call(cand, n, a.L, hist, red, &s_bin, &s_above);
            if (tau != -INFINITY) {
                const float below = nextafterf(tau, -INFINITY);
                exact = kl > ord_key(score_of(below, c, S));
            }
        }
        if (!exact) {
            n = exact_candidates(z, a.V, a.L, c, S, cand, hist, red, &s_bin, &s_above, &s_cnt);
            kl = radix_kth_call(cand, n, a.L, hist, red, &s_bin, &s_above);
        }
        // Only candidates at or above the larger of kl and the request's
        // bound can be selected (kl bounds the request's W'-th score from
        // below when L = W'): keep those (the row's best, at most L of them,
        // plus ties), sort and write them.
        const uint32_t keep = kl > lb ? kl : lb;
        // The kept entries go to the histogram's space (free from here on) in
        // any order, one shared atomic per warp and step: the sort below
        // orders them.  Past its kSide entries the candidate array is
        // compacted in place instead, by a block scan.
        unsigned long long *side = reinterpret_cast<unsigned long long *>(hist);
        if (threadIdx.x == 0) s_cnt = 0;
        __syncthreads();
        for (int base = 0; base < n; base += blockDim.x) {
            const int i = base + threadIdx.x;
            const bool f = i < n && (uint32_t)(cand[i] >> 32) >= keep;
            const unsigned m = __ballot_sync(kFullMask, f);
            if (m) {
                const int lane = threadIdx.x & 31;
                int b0 = 0;
                if (lane == 0) b0 = atomicAdd(&s_cnt, __popc(m));
                b0 = __shfl_sync(kFullMask, b0, 0);
                const int pos = b0 + __popc(m & ((1u << lane) - 1u));
                if (f && pos < kSide) side[pos] = cand[i];
            }
        }
        __syncthreads();
        int kept = s_cnt;
        unsigned long long *srt = side;
        if (kept > kSide) {
            srt = cand;
            kept = 0;
            for (int base = 0; base < n; base += blockDim.x) {
                const int i = base + threadIdx.x;
                const unsigned long long e = i < n ? cand[i] : 0ull;
                const int f = (i < n && (uint32_t)(e >> 32) >= keep) ? 1 : 0;
                int tot;
                const int pos = block_excl_scan(f, red, &tot);   // synchronises before any write below
                if (f) cand[kept + pos] = e;
                kept += tot;
                __syncthreads();
            }
        }
        int np2 = 1;
        while (np2 < kept) np2 <<= 1;
        for (int i = kept + threadIdx.x; i < np2; i += blockDim.x) srt[i] = 0ull;
        __syncthreads();
        sort_desc_blocked(srt, np2);
        const int cnt = min(kept, a.L);
        unsigned long long *out = a.lists + (long long)row * a.L;
        for (int j = threadIdx.x; j < cnt; j += blockDim.x) out[j] = srt[j];
        if (threadIdx.x == 0) {
            a.plen[row] = cnt;
            if (a.tau_lb) {
                // the row holds slot_k candidates at or above its slot_k-th
                const int req = row / a.W, beam = row - req * a.W;
                if (kept >= a.slot_k)
                    atomicMax(a.tau_slot + req * a.nslot + beam % a.nslot, (unsigned)(srt[a.slot_k - 1] >> 32));
                if (keep != 0u) atomicMax(a.tau_lb + req, keep);
            }
        }
        __syncthreads();
    }
}

// Descending bitonic sort of a warp's 256 entries, eight per lane (entry
// 8 * lane + j in e[j]): the exchanges below 8 inside a lane, the rest by
// warp shuffles.  All 32 lanes take part.
__device__ __forceinline__ void warp_sort256_desc(unsigned long long (&e)[8], int lane) {
#pragma unroll
    for (int k = 2; k <= 256; k <<= 1) {
#pragma unroll
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            if (jj >= 8) {
                const int m = jj >> 3;
                const bool lower = (lane & m) == 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = 8 * lane + j;
                    const bool desc = (i & k) == 0;
                    const unsigned long long o = shfl_xor_u64(e[j], m);
                    const bool take_max = desc == lower;
                    e[j] = take_max ? (o > e[j] ? o : e[j]) : (o < e[j] ? o : e[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int pj = j ^ jj;
                    if (pj > j) {
                        const int i = 8 * lane + j;
                        const bool desc = (i & k) == 0;
                        const unsigned long long lo = e[j], hi = e[pj];
                        const bool sw = desc ? (lo < hi) : (lo > hi);
                        e[j] = sw ? hi : lo;
                        e[pj] = sw ? lo : hi;
                    }
                }
            }
        }
    }
}

// A list tail of n <= 256 entries sorted descending in place by one warp
// (out of line: the merge kernel's rare overflow path).
__device__ __noinline__ void sort_tail_in_place(unsigned long long *t, int n, int lane) {
    unsigned long long e8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e8[j] = 8 * lane + j < n ? t[8 * lane + j] : 0ull;
    warp_sort256_desc(e8, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (8 * lane + j < n) t[8 * lane + j] = e8[j];
}

struct MergeSelArgs {
    const unsigned long long *lists;
    const unsigned *tau_lb;
    const int *plen;   // [R * W_s] entries of each row list
    int W, V, L, next_width;
    int32_t *next_parent;
    long long parent_stride;
    int32_t *next_token;
    float *next_score;
    // item-constrained selection only (null otherwise): the trie and each
    // beam's node, to give every kept beam its child node
    const int32_t *beam_node, *trie_offsets, *trie_tokens, *trie_children;
    int32_t *next_node;
    int num_nodes, num_edges;
    // a list entry's low word is ~u, and its flat index b * flat_mul + u orders
    // equal scores: u = v (flat_mul = V), or, for item-constrained rows, the
    // edge index (flat_mul = num_edges; edges are sorted by token within a
    // node, so the order is the same), which also names the child node
    unsigned flat_mul;
    int edge_coded;
    // > 0 (item-constrained rows): a list that holds every candidate of its
    // row has its first head_sorted entries in order and the rest in none.
    // Set only when head_sorted equals the merge's head keys per list and
    // those fit its shared memory (the prefixes are then read from them).
    int head_sorted;
};

// The merge's head keys per list (their next_width-th largest bounds the
// request's next_width-th score) and whether they fit its shared memory.
__host__ __device__ inline int merge_head_keys(int W, int next_width) {
    const int k = (8 * next_width + W - 1) / W;
    return k < 1 ? 1 : (k > 32 ? 32 : k);
}

// dynamic shared memory of the merge kernel: list offsets, per-list counts
// above and tied with the threshold, the histogram and the selection
constexpr int kMaxBeams = 4096;   // GR_SELECT_MAX_BEAMS
constexpr int kEntCap = 4096;     // entries the merge holds in shared memory at once
constexpr int kMergeSmem = (3 * (kMaxBeams + 1) + kHistBins) * 4 + (kMaxSel + kEntCap) * 8;

// One CTA per request.  Each row list holds the row's best candidates down to
// the bound that row saw; only entries at or above the final lower bound can
// be selected.  The entries of all lists are walked as one flat range (list
// offsets in shared memory), so every thread keeps several independent loads
// in flight.  The W'-th largest key is found by a radix select (12 + 12 + 8
// bits), then every key above it is taken and the tied ones in flat-index
// order (lists in b order, each list in v order: the lists are sorted), and
// the W' are sorted by (score desc, flat asc).
__global__ void __launch_bounds__(kMergeThreads, 1) select_merge_kernel(MergeSelArgs a) {
    grid_dep_wait();   // the row lists, lengths and bounds of the kernel(s) before
    extern __shared__ unsigned long long msm[];
    unsigned long long *sel = msm;                           // [kMaxSel] (8-byte entries first)
    unsigned long long *ent = sel + kMaxSel;                 // [kEntCap] the candidates at or above the bound
    int *offs = reinterpret_cast<int *>(ent + kEntCap);      // [W + 1]
    int *gtc = offs + (kMaxBeams + 1);                       // [W + 1] entries above tau, then offsets
    int *eqc = gtc + (kMaxBeams + 1);                        // [W + 1] entries tied with tau, then offsets
    int *hist = eqc + (kMaxBeams + 1);                       // [kHistBins]
    __shared__ int red[32];
    __shared__ int s_bin, s_above;
    const int r = blockIdx.x;
    const unsigned long long *lists = a.lists + (long long)r * a.W * a.L;
    const int *plen = a.plen + (long long)r * a.W;
    uint32_t lb = a.tau_lb ? a.tau_lb[r] : 0u;
    const int per = (a.W + blockDim.x - 1) / blockDim.x;
    const int b0 = min(a.W, (int)threadIdx.x * per), b1 = min(a.W, b0 + per);
    // A tighter bound: the next_width-th largest key among the first kh keys
    // of every list (real candidates, so at least next_width entries reach it),
    // to its top 24 bits: a radix select of two 12-bit passes, the key's low 8
    // bits left zero (a lower bound still, looser by at most one 256-ulp bin).
    const int kh = merge_head_keys(a.W, a.next_width);
    // the keys go where offs, gtc and eqc will be (not yet in use)
    const unsigned *heads = reinterpret_cast<const unsigned *>(offs);
    const bool have_heads = a.W * kh <= 3 * (kMaxBeams + 1);
    {
        unsigned *heads_w = reinterpret_cast<unsigned *>(offs);
        const int cap = 3 * (kMaxBeams + 1);
        int nh = 0;
        if (a.W * kh <= cap) {
            for (int t = threadIdx.x; t < a.W * kh; t += blockDim.x) {
                const int b = t / kh, j = t % kh;
                heads_w[t] = j < plen[b] ? (unsigned)(lists[(long long)b * a.L + j] >> 32) : 0u;
            }
            nh = a.W * kh;
        }
        __syncthreads();
        if (nh >= a.next_width) {
            uint32_t prefix = 0, mask = 0;
            int need = a.next_width;
            const int shifts[2] = {20, 8}, widths[2] = {12, 12};
#pragma unroll
            for (int rd = 0; rd < 2; ++rd) {
                for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
                __syncthreads();
                const int sh = shifts[rd];
                const uint32_t bm = (1u << widths[rd]) - 1u;
                for (int i = threadIdx.x; i < nh; i += blockDim.x) {
                    const uint32_t k = heads[i];
                    if ((k & mask) == prefix) atomicAdd(&hist[kHistBins - 1 - (int)(bm - ((k >> sh) & bm))], 1);
                }
                __syncthreads();
                find_bin(hist, need, red, &s_bin, &s_above);
                need -= s_above;
                prefix |= (bm - (uint32_t)(kHistBins - 1 - s_bin)) << sh;
                mask |= bm << sh;
                __syncthreads();
            }
            lb = prefix > lb ? prefix : lb;
        }
    }
    // per list, the sorted prefix at or above the bound: from the head keys
    // when the prefix ends among them (most lists), else by a binary search
    // past them; then the list offsets (lists [b0, b1) of this thread are
    // consecutive, at most 4 of them).  The head keys share memory with the
    // offsets: every thread reads them before the scan's barriers, and the
    // offsets are written after it.
    int pl[4] = {0, 0, 0, 0};
    int mine = 0;
    unsigned pend = 0u;   // lists (bit q) whose tail past the head keys is in no order and may reach the bound
    auto search = [&](int b, int lo) {   // first index at or past lo whose key < lb (sorted list)
        const unsigned long long *lst = lists + (long long)b * a.L;
        int hi = plen[b];
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((uint32_t)(lst[mid] >> 32) >= lb) lo = mid + 1;
            else hi = mid;
        }
        return lo;
    };
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = b0 + q;
        if (b >= b1) break;
        const int len = plen[b];
        int lo = 0;
        if (have_heads) {
            const int hn = min(kh, len);
            while (lo < hn && heads[b * kh + lo] >= lb) ++lo;
            if (lo < hn || len <= kh) {
                pl[q] = lo;
                mine += lo;
                continue;
            }
            if (a.head_sorted) {
                pl[q] = kh;
                mine += kh;
                pend |= 1u << q;
                continue;
            }
        }
        pl[q] = search(b, lo);
        mine += pl[q];
    }
    int total;
    auto write_offsets = [&]() {
        int off = block_excl_scan(mine, red, &total);
        __syncthreads();   // every head key has been read
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int b = b0 + q;
            if (b >= b1) break;
            offs[b] = off;
            off += pl[q];
            gtc[b] = 0;
            eqc[b] = 0;
        }
        if (threadIdx.x == 0) offs[a.W] = total;
        __syncthreads();
    };
    write_offsets();
    // Lists whose head keys all reach the bound and whose tails are in no
    // order (item-constrained rows; about one per request): their tail
    // entries at or above the bound go after the prefixes, filtered by a warp
    // per list.  If the candidates then overflow the shared memory, the
    // tails are sorted in place instead and taken into the prefixes.
    int ntail = 0;
    if (a.head_sorted) {
        int *pend_list = hist;   // free until the selection below
        if (threadIdx.x == 0) {
            s_bin = 0;
            s_above = 0;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (pend >> q & 1u) pend_list[atomicAdd(&s_bin, 1)] = b0 + q;
        __syncthreads();
        const int npend = s_bin;
        const int wq = threadIdx.x >> 5, ln = threadIdx.x & 31, nwq = blockDim.x >> 5;
        for (int pi = wq; pi < npend; pi += nwq) {
            const int b = pend_list[pi];
            const unsigned long long *lst = lists + (long long)b * a.L;
            const int len = plen[b];
            for (int j = kh + ln; j < len; j += 32) {
                const unsigned long long v = lst[j];
                if ((uint32_t)(v >> 32) >= lb) {
                    const int pos = atomicAdd(&s_above, 1);
                    if (total + pos < kEntCap) {
                        const uint32_t flat = (uint32_t)b * a.flat_mul + ~(uint32_t)v;
                        ent[total + pos] = ((v >> 32) << 32) | (uint32_t)~flat;
                    }
                }
            }
        }
        __syncthreads();
        ntail = s_above;
        if (npend > 0 && total + ntail > kEntCap) {
            for (int pi = wq; pi < npend; pi += nwq) {   // warp-uniform
                const int b = pend_list[pi];
                // the workspace's list: a warp row's tail holds at most 256 - kh
                // entries; a wide row's list is in order already, and sorting the
                // first 256 entries of its tail keeps it so
                sort_tail_in_place(const_cast<unsigned long long *>(lists) + (long long)b * a.L + kh, plen[b] - kh, ln);
            }
            __syncthreads();   // the sorted tails are visible to the block
            mine = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int b = b0 + q;
                if (b >= b1) break;
                if (pend >> q & 1u) pl[q] = search(b, kh);
                mine += pl[q];
            }
            write_offsets();
            ntail = 0;
        }
    }
    // entry e of the flat range: list b (offs[b] <= e < offs[b+1]) and index j
    auto locate = [&](int e, int &b, int &j) {
        int lo = 0, hi = a.W;   // the last b with offs[b] <= e
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (offs[mid] <= e) lo = mid;
            else hi = mid;
        }
        b = lo;
        j = e - offs[lo];
    };
    // the W' selected entries, sorted by (score desc, flat asc), into the outputs
    auto emit = [&](const unsigned long long *src, int n_sel) {
        for (int j = threadIdx.x; j < a.next_width; j += blockDim.x) {
            int32_t pb = -1, tv = -1, nd = -1;
            float sc = -INFINITY;
            if (j < n_sel) {
                const unsigned long long e = src[j];
                const uint32_t flat = ~(uint32_t)e;
                pb = (int32_t)(flat / a.flat_mul);
                const uint32_t u = flat % a.flat_mul;
                sc = key_float((uint32_t)(e >> 32));
                tv = (int32_t)u;
                if (a.edge_coded) {
                    // the edge itself: its token and child node
                    tv = a.trie_tokens[u];
                    if (a.next_node) nd = a.trie_children[u];
                } else if (a.next_node) {
                    // the edge of the parent's node that carries the token; the node
                    // and its edge range are checked as the rows kernel checks them,
                    // and a search that lands past the range or on another token (a
                    // node whose tokens are not increasing) gives no child
                    const int n = a.beam_node[(long long)r * a.W + pb];
                    if (n >= 0 && n < a.num_nodes) {
                        const int e0 = a.trie_offsets[n], e1 = a.trie_offsets[n + 1];
                        if (e0 >= 0 && e1 <= a.num_edges && e0 <= e1) {
                            int lo = e0, hi = e1;
                            while (lo < hi) {
                                const int mid = (lo + hi) >> 1;
                                if (a.trie_tokens[mid] < tv) lo = mid + 1;
                                else hi = mid;
                            }
                            if (lo < e1 && a.trie_tokens[lo] == tv) nd = a.trie_children[lo];
                        }
                    }
                }
            }
            a.next_parent[(long long)r * a.parent_stride + j] = pb;
            a.next_token[(long long)r * a.next_width + j] = tv;
            a.next_score[(long long)r * a.next_width + j] = sc;
            if (a.next_node) a.next_node[(long long)r * a.next_width + j] = nd;
        }
    };
    if (total + ntail <= kEntCap) {
        // Every candidate at or above the bound fits in shared memory: read each
        // once as (score key, ~flat index) and sort them in registers (up to
        // kMaxSel of them; past that only those at or above the n_sel-th
        // largest key); the first n_sel are the selection, ties in flat-index
        // order.
        for (int e = threadIdx.x; e < total; e += blockDim.x) {
            int b, j;
            locate(e, b, j);
            const unsigned long long v = lists[(long long)b * a.L + j];
            const uint32_t flat = (uint32_t)b * a.flat_mul + ~(uint32_t)v;
            ent[e] = ((v >> 32) << 32) | (uint32_t)~flat;
        }
        __syncthreads();
        total += ntail;   // the filtered tails follow the prefixes
        const int n_sel = min(a.next_width, total);
        int n = total;
        if (n > kMaxSel && n_sel > 0) {
            // more than a sort takes cheaply: the n_sel-th largest key first, and
            // only the entries at or above it (ties included) are sorted
            const uint32_t tau = radix_kth(ent, total, n_sel, hist, red, &s_bin, &s_above);
            n = compact(ent, total, red, [&](unsigned long long e) { return (uint32_t)(e >> 32) >= tau; },
                        [](unsigned long long e) { return e; });
        }
        int np2 = 1;
        while (np2 < n) np2 <<= 1;
        for (int i = n + threadIdx.x; i < np2; i += blockDim.x) ent[i] = 0ull;
        __syncthreads();
        // sorted by (score desc, flat asc): the first n_sel are the selection
        sort_desc_blocked(ent, np2);
        emit(ent, n_sel);
        return;
    }
    constexpr int kIn = 4;   // loads in flight per thread
    // radix select of the n_sel-th largest key (n_sel < next_width only when
    // the request has fewer candidates: the rest of the slots are padding)
    const int n_sel = min(a.next_width, total);
    uint32_t prefix = 0, mask = 0;
    int need = n_sel;
    const int shifts[3] = {20, 8, 0}, widths[3] = {12, 12, 8};
    if (n_sel > 0) {
#pragma unroll
    for (int rd = 0; rd < 3; ++rd) {
        for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const int sh = shifts[rd];
        const uint32_t bm = (1u << widths[rd]) - 1u;
        for (int e0 = threadIdx.x; e0 < total; e0 += kIn * blockDim.x) {
            uint32_t k[kIn];
#pragma unroll
            for (int u = 0; u < kIn; ++u) {
                const int e = e0 + u * blockDim.x;
                k[u] = 0u;
                if (e < total) {
                    int b, j;
                    locate(e, b, j);
                    k[u] = (uint32_t)(lists[(long long)b * a.L + j] >> 32);
                }
            }
#pragma unroll
            for (int u = 0; u < kIn; ++u)
                if (e0 + u * blockDim.x < total && k[u] >= lb && (k[u] & mask) == prefix)
                    atomicAdd(&hist[kHistBins - 1 - (int)(bm - ((k[u] >> sh) & bm))], 1);
        }
        __syncthreads();
        find_bin(hist, need, red, &s_bin, &s_above);
        need -= s_above;
        prefix |= (bm - (uint32_t)(kHistBins - 1 - s_bin)) << sh;
        mask |= bm << sh;
        __syncthreads();
    }
    }
    const uint32_t tau = prefix;   // need = how many entries equal to tau are taken
    // per list: entries above tau and tied with it (runs at the list's front)
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
        int b, j;
        locate(e, b, j);
        const uint32_t k = (uint32_t)(lists[(long long)b * a.L + j] >> 32);
        if (k > tau) atomicAdd(&gtc[b], 1);
        else if (k == tau) atomicAdd(&eqc[b], 1);
    }
    __syncthreads();
    int gt = 0, eq = 0;
    for (int b = b0; b < b1; ++b) {
        gt += gtc[b];
        eq += eqc[b];
    }
    int n_gt, n_eq;
    int pos_gt = block_excl_scan(gt, red, &n_gt);
    int pos_eq = block_excl_scan(eq, red, &n_eq);
    // the counts become offsets (in b order); entry W holds the totals, so a
    // list's count is the next offset minus its own
    for (int b = b0; b < b1; ++b) {
        const int g = gtc[b], q = eqc[b];
        gtc[b] = pos_gt;
        eqc[b] = pos_eq;
        pos_gt += g;
        pos_eq += q;
    }
    if (threadIdx.x == 0) {
        gtc[a.W] = n_gt;
        eqc[a.W] = n_eq;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
        int b, j;
        locate(e, b, j);
        const int og = gtc[b], g = gtc[b + 1] - og;
        const int oe = eqc[b], q = eqc[b + 1] - oe;
        if (j >= g + q) continue;
        const unsigned long long ent = lists[(long long)b * a.L + j];
        const uint32_t flat = (uint32_t)b * a.flat_mul + ~(uint32_t)ent;
        const unsigned long long item = ((ent >> 32) << 32) | (uint32_t)~flat;
        if (j < g) sel[og + j] = item;
        else if (oe + (j - g) < need) sel[n_gt + oe + (j - g)] = item;
    }
    __syncthreads();
    int np2 = 1;
    while (np2 < a.next_width) np2 <<= 1;
    for (int i = n_sel + threadIdx.x; i < np2; i += blockDim.x) sel[i] = 0ull;
    __syncthreads();
    sort_desc_blocked(sel, np2);
    emit(sel, n_sel);
}

// ---------------------------------------------------------------- item-constrained rows
//
// One CTA per beam row.  The row's legal tokens are the edges of its trie
// node (CSR); their logits are gathered (pass A: maximum and sum of
// exponentials over the legal tokens only, the log-normaliser of the masked
// log_softmax), then scored in chunks of kTrieChunk edges that are sorted
// together with the best entries so far, keeping the best min(W', degree)
// by (score desc, token asc).  A node index or edge range outside the trie,
// or an edge token outside [0, V), is skipped (nothing is read out of range).

constexpr int kTrieThreads = 256;
constexpr int kTrieChunk = 1024;

struct TrieRowArgs {
    const float *logits;
    const float *beam_scores;
    const int32_t *beam_node, *offsets, *tokens;
    unsigned long long *lists;   // [R * W_s][W'] sorted descending
    int *plen;
    unsigned *tau_lb;
    int *big_count;              // rows whose node has more edges than a warp holds
    int *big_rows;               // [R * W_s] those rows, in any order
    int rows, W, V, next_width, num_nodes, num_edges;
    int edge_coded;              // list entries carry the edge index instead of the token
    int head_sorted;             // > 0: a row keeping every candidate orders only its best head_sorted
};

// A row's trie node and its edge range [p0, p1) (empty for a node index or
// edge range outside the trie).
__device__ __forceinline__ void node_edges(const TrieRowArgs &a, int row, int &p0, int &p1) {
    const int n = a.beam_node[row];
    p0 = 0;
    p1 = 0;
    if (n >= 0 && n < a.num_nodes) {
        p0 = a.offsets[n];
        p1 = a.offsets[n + 1];
        if (p0 < 0 || p1 > a.num_edges || p1 < p0) p0 = p1 = 0;
    }
}

// One warp per beam row whose node has at most kTrieWarpDeg edges (8 per
// lane): the legal logits are gathered in one round trip, the masked
// log-normaliser comes from warp reductions, and the row's candidates
// (score key, ~v) are sorted by a bitonic network in registers (lane l holds
// elements 8l..8l+7; exchanges across lanes are shuffles), so a row costs no
// block barrier.  The best min(W', degree) are written as the block kernel
// writes them.  Rows with more edges are appended to big_rows for
// trie_rows_kernel.
constexpr int kTrieWarpDeg = 256;
constexpr int kTrieWarpRows = 8;   // rows (warps) per CTA

__global__ void __launch_bounds__(kTrieWarpRows * 32) trie_rows_warp_kernel(TrieRowArgs a) {
    // the wide-row kernel may be scheduled now (it waits for this grid): every
    // CTA of this grid is resident at once, so it takes no slot from them
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kTrieWarpRows + (threadIdx.x >> 5);
    if (row >= a.rows) return;   // warp-uniform
    int p0, p1;
    node_edges(a, row, p0, p1);
    const int deg = p1 - p0;
    if (deg > kTrieWarpDeg) {
        if (lane == 0) a.big_rows[atomicAdd(a.big_count, 1)] = row;
        return;
    }
    const float *z = a.logits + (long long)row * a.V;
    const float S = a.beam_scores[row];
    // lane l takes edges 8l .. 8l+7
    int v[8];
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int k = 8 * lane + j;
        v[j] = k < deg ? a.tokens[p0 + k] : -1;
        if (v[j] >= a.V) v[j] = -1;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = v[j] >= 0 ? __ldg(z + v[j]) : -INFINITY;
    MaxSum ms{-INFINITY, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (v[j] >= 0) ms = ms_add(ms, x[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum other{__shfl_xor_sync(kFullMask, ms.m, o), __shfl_xor_sync(kFullMask, ms.s, o)};
        ms = ms_merge(ms, other);
    }
    const float c = ms.m + __logf(ms.s);
    // a skipped edge sorts last and is not kept: key 0 is below every score
    unsigned long long e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        e[j] = v[j] >= 0 ? pack(ord_key(score_of(x[j], c, S)),
                                ~(uint32_t)(a.edge_coded ? p0 + 8 * lane + j : v[j]))
                         : 0ull;
    // the valid candidates (a skipped edge is 0, below every score)
    int valid = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) valid += (e[j] >> 32) != 0ull ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) valid += __shfl_xor_sync(kFullMask, valid, o);
    unsigned long long *out = a.lists + (long long)row * a.next_width;
    if (a.head_sorted > 0 && valid < a.next_width) {   // warp-uniform
        // The row keeps every candidate, and the merge reads in order only
        // its first head_sorted: those in order, the rest in none.  Each
        // lane sorts its eight, then every round takes the warp's largest
        // head (entries are distinct: one lane holds it) and that lane
        // moves up its next.
#pragma unroll
        for (int k = 2; k <= 8; k <<= 1) {
#pragma unroll
            for (int jj = k >> 1; jj > 0; jj >>= 1) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int pj = j ^ jj;
                    if (pj > j) {
                        const bool desc = (j & k) == 0;
                        const unsigned long long lo = e[j], hi = e[pj];
                        const bool sw = desc ? (lo < hi) : (lo > hi);
                        e[j] = sw ? hi : lo;
                        e[pj] = sw ? lo : hi;
                    }
                }
            }
        }
        const int T = min(a.head_sorted, valid);
        unsigned long long top = 0ull;
        for (int rr = 0; rr < T; ++rr) {
            unsigned long long h = e[0];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long x = shfl_xor_u64(h, o);
                h = x > h ? x : h;
            }
            if (lane == rr) top = h;
            const bool win = e[0] == h;
#pragma unroll
            for (int j = 0; j < 7; ++j) e[j] = win ? e[j + 1] : e[j];
            e[7] = win ? 0ull : e[7];
        }
        if (lane < T) out[lane] = top;
        // the rest: each lane's remaining valid entries (first in e[]), after those of the lanes before it
        int mine = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) mine += (e[j] >> 32) != 0ull ? 1 : 0;
        int pre = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(kFullMask, pre, o);
            if (lane >= o) pre += x;
        }
        pre -= mine;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < mine) out[T + pre + j] = e[j];
        if (lane == 0) a.plen[row] = valid;
        return;
    }
    // descending sort of the warp's 256 entries (entry 8 * lane + j in e[j])
    warp_sort256_desc(e, lane);
    const int cnt = min(valid, a.next_width);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (8 * lane + j < cnt) out[8 * lane + j] = e[j];
    if (lane == 0) a.plen[row] = cnt;
    // a row with W' candidates of its own bounds the request's W'-th score
    if (cnt == a.next_width && cnt > 0 && a.tau_lb) {   // warp-uniform
        const int jl = (cnt - 1) & 7;
        unsigned long long pick = e[0];
#pragma unroll
        for (int j = 1; j < 8; ++j)
            if (j == jl) pick = e[j];
        const unsigned long long last = __shfl_sync(kFullMask, pick, (cnt - 1) >> 3);
        if (lane == 0) atomicMax(a.tau_lb + row / a.W, (unsigned)(last >> 32));
    }
}

// The rows whose node has more edges than a warp holds, one CTA at a time per
// row (grid-strided over big_rows).
__global__ void __launch_bounds__(kTrieThreads) trie_rows_kernel(TrieRowArgs a) {
    grid_dep_wait();   // the wide-row list of the warp kernel
    grid_dep_launch();
    __shared__ unsigned long long buf[kMaxSel + kTrieChunk];
    __shared__ MaxSum s_ms[kTrieThreads / 32];
    __shared__ float s_c;
    __shared__ int s_keep;
    const int nbig = *reinterpret_cast<volatile int *>(a.big_count);
    for (int bi = blockIdx.x; bi < nbig; bi += gridDim.x) {
    const int row = a.big_rows[bi];
    const int n = a.beam_node[row];
    int p0 = 0, p1 = 0;
    if (n >= 0 && n < a.num_nodes) {
        p0 = a.offsets[n];
        p1 = a.offsets[n + 1];
        if (p0 < 0 || p1 > a.num_edges || p1 < p0) p0 = p1 = 0;
    }
    const int deg = p1 - p0;
    const float *z = a.logits + (long long)row * a.V;
    const float S = a.beam_scores[row];
    auto legal = [&](int k, int &v) {
        v = a.tokens[p0 + k];
        return v >= 0 && v < a.V;
    };
    // pass A: the log-normaliser over the legal logits
    MaxSum ms{-INFINITY, 0.f};
    for (int k = threadIdx.x; k < deg; k += blockDim.x) {
        int v;
        if (legal(k, v)) ms = ms_add(ms, __ldg(z + v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum other{__shfl_xor_sync(kFullMask, ms.m, o), __shfl_xor_sync(kFullMask, ms.s, o)};
        ms = ms_merge(ms, other);
    }
    if ((threadIdx.x & 31) == 0) s_ms[threadIdx.x >> 5] = ms;
    __syncthreads();
    if (threadIdx.x == 0) {
        MaxSum t = s_ms[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = ms_merge(t, s_ms[w]);
        s_c = t.m + __logf(t.s);
    }
    __syncthreads();
    const float c = s_c;
    // pass B: the best L entries, chunk by chunk
    const int L = min(a.next_width, deg);
    int cnt = 0;
    for (int base = 0; base < deg; base += kTrieChunk) {
        const int m = min(kTrieChunk, deg - base);
        for (int k = threadIdx.x; k < m; k += blockDim.x) {
            int v;
            // a skipped edge sorts last and is not kept: key 0 is below every score
            buf[cnt + k] = legal(base + k, v) ? pack(ord_key(score_of(__ldg(z + v), c, S)),
                                                     ~(uint32_t)(a.edge_coded ? p0 + base + k : v))
                                              : 0ull;
        }
        const int tot = cnt + m;
        int np2 = 1;
        while (np2 < tot) np2 <<= 1;
        for (int i = tot + threadIdx.x; i < np2; i += blockDim.x) buf[i] = 0ull;
        __syncthreads();
        bitonic_desc(buf, np2);
        cnt = min(tot, L);
    }
    // drop skipped edges (key 0) from the kept count
    if (threadIdx.x == 0) {
        int k = cnt;
        while (k > 0 && (buf[k - 1] >> 32) == 0ull) --k;
        s_keep = k;
    }
    __syncthreads();
    cnt = s_keep;
    unsigned long long *out = a.lists + (long long)row * a.next_width;
    for (int j = threadIdx.x; j < cnt; j += blockDim.x) out[j] = buf[j];
    if (threadIdx.x == 0) {
        a.plen[row] = cnt;
        // a row with W' candidates of its own bounds the request's W'-th score
        if (cnt == a.next_width && a.tau_lb) atomicMax(a.tau_lb + row / a.W, (unsigned)(buf[cnt - 1] >> 32));
    }
    __syncthreads();   // buf and the shared scalars are reused by the next row
    }
}

}  // namespace

// workspace: row lists [R * W][L] u64 | lower bounds [R] u32 and bound slots
// [R][kBoundSlots] u32 (16-byte padded) | list lengths [R * W] int32
static size_t list_bytes(int R, int W, int L) { return (size_t)R * W * L * sizeof(unsigned long long); }
static size_t bound_bytes(int R) { return ((size_t)R * (1 + kBoundSlots) * 4 + 15) / 16 * 16; }

// Launches a kernel that may start while the one before it on the stream
// finishes (programmatic stream serialization; the kernel waits in
// grid_dep_wait before reading that kernel's output).  Without `overlap`
// it is an ordinary launch (an event recorded between the two kernels must
// see the first one complete).
template <typename... Params, typename... Args>
static cudaError_t launch_after(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                bool overlap, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

size_t select_list_bytes(int R, int W, int V, int next_width) {
    const int L = next_width < V ? next_width : V;
    return list_bytes(R, W, L) + bound_bytes(R) + (size_t)R * W * sizeof(int);
}

int select_max_width() { return kMaxSel; }
int select_max_beams() { return kMaxBeams; }

cudaError_t launch_beam_select(int R, int W, int V, int next_width, const float *logits,
                               const float *beam_scores, int32_t *next_parent, long long parent_stride,
                               int32_t *next_token, float *next_score, void *workspace, cudaStream_t s,
                               cudaEvent_t between) {
    static std::mutex mu;
    static int sm_count[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (sm_count[dev] == 0) {
            int n = 0;
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(select_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kCap * 8 + kHistBins * 4 + 32 * 4);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(select_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMergeSmem);
            if (e != cudaSuccess) return e;
            sm_count[dev] = n;
        }
    }
    const int L = next_width < V ? next_width : V;
    unsigned char *wsb = static_cast<unsigned char *>(workspace);
    unsigned *tau_lb = reinterpret_cast<unsigned *>(wsb + list_bytes(R, W, L));
    int *counts = reinterpret_cast<int *>(wsb + list_bytes(R, W, L) + bound_bytes(R));
    // the bound is only valid when a row alone holds W' candidates (V >= W')
    const bool bound = L == next_width;
    if (bound) {
        e = cudaMemsetAsync(tau_lb, 0, (size_t)R * (1 + kBoundSlots) * 4, s);
        if (e != cudaSuccess) return e;
    }
    RowArgs ra;
    ra.logits = logits;
    ra.beam_scores = beam_scores;
    ra.lists = reinterpret_cast<unsigned long long *>(wsb);
    ra.tau_lb = bound ? tau_lb : nullptr;
    ra.tau_slot = tau_lb + R;
    ra.nslot = W < kBoundSlots ? W : kBoundSlots;
    ra.slot_k = (next_width + ra.nslot - 1) / ra.nslot;
    ra.plen = counts;
    ra.rows = R * W;
    ra.W = W;
    ra.V = V;
    ra.L = L;
    const int smem = kCap * 8 + kHistBins * 4 + 32 * 4;
    const int slots = sm_count[dev] * kRowBlocksPerSm;
    const int grid = ra.rows < slots ? ra.rows : slots;
    select_rows_kernel<<<grid, kRowThreads, smem, s>>>(ra);
    e = cudaGetLastError();
    if (e == cudaSuccess && between) e = cudaEventRecord(between, s);
    if (e != cudaSuccess) return e;
    MergeSelArgs ma = {};
    ma.lists = ra.lists;
    ma.tau_lb = ra.tau_lb;
    ma.plen = counts;
    ma.W = W;
    ma.V = V;
    ma.L = ra.L;
    ma.next_width = next_width;
    ma.next_parent = next_parent;
    ma.parent_stride = parent_stride;
    ma.next_token = next_token;
    ma.next_score = next_score;
    ma.flat_mul = (unsigned)V;
    ma.edge_coded = 0;
    e = launch_after(select_merge_kernel, dim3(R), dim3(kMergeThreads), kMergeSmem, s, between == nullptr, ma);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// trie workspace: row lists [R * W][W'] u64 | lower bounds [R] u32 and the
// big-row count (16-byte padded) | list lengths [R * W] int32 | big rows [R * W] int32
static size_t trie_bound_bytes(int R) { return ((size_t)(R + 1) * 4 + 15) / 16 * 16; }

size_t trie_select_bytes(int R, int W, int next_width) {
    return list_bytes(R, W, next_width) + trie_bound_bytes(R) + 2 * (size_t)R * W * sizeof(int);
}

cudaError_t launch_trie_select(int R, int W, int V, int next_width, int num_nodes, int num_edges,
                               const float *logits, const float *beam_scores, const int32_t *beam_node,
                               const int32_t *offsets, const int32_t *tokens, const int32_t *children,
                               int32_t *next_parent, long long parent_stride, int32_t *next_token,
                               float *next_score, int32_t *next_node, void *workspace, cudaStream_t s,
                               cudaEvent_t between) {
    static std::mutex mu;
    static int sm_count[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (sm_count[dev] == 0) {
            int nsm = 0;
            e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(select_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmem);
            if (e != cudaSuccess) return e;
            sm_count[dev] = nsm;
        }
    }
    unsigned char *wsb = static_cast<unsigned char *>(workspace);
    unsigned *tau_lb = reinterpret_cast<unsigned *>(wsb + list_bytes(R, W, next_width));
    int *big_count = reinterpret_cast<int *>(tau_lb + R);
    int *plen = reinterpret_cast<int *>(wsb + list_bytes(R, W, next_width) + trie_bound_bytes(R));
    int *big_rows = plen + (size_t)R * W;
    // the bounds and the big-row count start at zero (one copy)
    e = cudaMemsetAsync(tau_lb, 0, (size_t)(R + 1) * 4, s);
    if (e != cudaSuccess) return e;
    TrieRowArgs ta;
    ta.logits = logits;
    ta.beam_scores = beam_scores;
    ta.beam_node = beam_node;
    ta.offsets = offsets;
    ta.tokens = tokens;
    ta.lists = reinterpret_cast<unsigned long long *>(wsb);
    ta.plen = plen;
    ta.tau_lb = tau_lb;
    ta.rows = R * W;
    ta.W = W;
    ta.V = V;
    ta.next_width = next_width;
    ta.num_nodes = num_nodes;
    ta.num_edges = num_edges;
    ta.big_count = big_count;
    ta.big_rows = big_rows;
    // edge-coded entries while every flat index b * num_edges + e fits 32 bits
    ta.edge_coded = (num_edges > 0 && (unsigned long long)W * (unsigned long long)num_edges < (1ull << 32)) ? 1 : 0;
    // rows that keep every candidate order only the merge's head keys when
    // those fit its shared memory and are few (a full sort is cheaper past 8)
    {
        const int kh = merge_head_keys(W, next_width);
        ta.head_sorted = ((long long)W * kh <= 3LL * (kMaxBeams + 1) && kh <= 8) ? kh : 0;
    }
    trie_rows_warp_kernel<<<(R * W + kTrieWarpRows - 1) / kTrieWarpRows, kTrieWarpRows * 32, 0, s>>>(ta);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    {
        const int grid = R * W < 2 * sm_count[dev] ? R * W : 2 * sm_count[dev];
        e = launch_after(trie_rows_kernel, dim3(grid), dim3(kTrieThreads), 0, s, true, ta);
        if (e != cudaSuccess) return e;
    }
    e = cudaGetLastError();
    if (e == cudaSuccess && between) e = cudaEventRecord(between, s);
    if (e != cudaSuccess) return e;
    MergeSelArgs ma = {};
    ma.lists = ta.lists;
    ma.tau_lb = tau_lb;
    ma.plen = plen;
    ma.head_sorted = ta.head_sorted;
    ma.W = W;
    ma.V = V;
    ma.L = next_width;
    ma.next_width = next_width;
    ma.next_parent = next_parent;
    ma.parent_stride = parent_stride;
    ma.next_token = next_token;
    ma.next_score = next_score;
    ma.beam_node = beam_node;
    ma.trie_offsets = offsets;
    ma.trie_tokens = tokens;
    ma.trie_children = children;
    ma.next_node = next_node;
    ma.num_nodes = num_nodes;
    ma.num_edges = num_edges;
    ma.edge_coded = ta.edge_coded;
    ma.flat_mul = ta.edge_coded ? (unsigned)num_edges : (unsigned)V;
    e = launch_after(select_merge_kernel, dim3(R), dim3(kMergeThreads), kMergeSmem, s, between == nullptr, ma);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gr
