// select.cu -- beam candidate selection of one decode step.
//
// "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", section 1.1: every decode
// step selects local candidates from each beam's token distribution, merges them
// with the accumulated scores and keeps a fixed number W of candidate sequences;
// the candidates, their scores and the parent index come out.  Readings: the
// distribution is the softmax of the beam's logits, scores add log-probabilities,
//     score(b, v) = cum[b] + logits[b, v] - logsumexp_u(logits[b, u]),
// the W best (b, v) of a request are kept, best first, equal scores by the
// smaller b * V + v.
//
// Two or three launches on the caller's stream:
//   1. row_select_kernel, one CTA per beam row, two passes over the row.  The first
//      (from HBM) computes the row's logsumexp and the maximum of each of 2048
//      interleaved groups of its logits; those maxima are 2048 distinct logits, so
//      the W-th largest of them (narrowed by a radix selection on an order-preserving
//      integer key) bounds the row's W-th best from below.  The first pass also keeps
//      every float4's maximum, truncated to bf16, in shared memory; the second pass
//      reads back from L2 only the float4s whose stored maximum reaches the bound
//      (rows longer than 131,072 logits stream the whole row again), gathers the
//      logits at or above the bound into shared memory, and a bitonic sort in
//      registers orders them: the beam's W best (value, token) and its logsumexp go
//      to the workspace.  A beam's W best tokens contain its whole share of the
//      request's W best candidates.
//   2. the merge, a radix selection over the W x W local candidates of a request keyed
//      by their scores: merge_part_kernel selects the W best of each of S slices of
//      beams (S = 1 when all W x W fit one CTA's key cache: then it writes the result),
//   3. and for S > 1, merge_final_kernel the W best of the S * W survivors of each
//      request (two levels, so that more than R CTAs share the work).
// HBM-bound: the logits come from HBM once; everything else stays on chip or in L2.
#include "bg_internal.h"
#include "bg_ptx.cuh"

#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

namespace bg {
namespace {

constexpr int kSelThreads = 512;
constexpr int kCap = 2048;          // ck/ci entries: filtered logits, the sort's exchange halves
constexpr int kBins = 4096;         // 12-bit radix digits

// Row selection: kRowLoads float4 loads per thread in flight; 4 * kSelThreads groups
// of logits give the maxima that bound the row's W-th best; the float4 groups holding a
// logit at or above that bound are gathered, at most kGather logits (a row with more
// takes the full radix path).
constexpr int kRowLoads = 8;
constexpr int kGather = 4096;
constexpr int kBoundCap = 448;                         // most group maxima at or above the bound
constexpr int kGatherSmem = kGather * 8;               // gathered logits: value + token
// Rows of at most kMaxStored float4 groups also keep, per group, its maximum truncated to
// bf16 (2 bytes) in shared memory, so that the second pass re-reads only the groups that
// can pass the bound instead of the whole row.
constexpr int kMaxStored = 32768;
constexpr int kRowDynSmemMax = kGatherSmem + kMaxStored * 2;
// The merges keep their candidates' keys in shared memory: level 2 always (S * W <= 16 * 512
// of them), level 1 when its largest slice, ceil(W / S) beams of W candidates, has at most
// kMergeCacheKeys; otherwise level 1 recomputes them in every pass.
constexpr int kMergeCacheKeys = 16384;
constexpr int kMergeSmemMax = kMergeCacheKeys * 4;
static_assert(16 * BG_MAX_BEAM <= kMergeCacheKeys, "level 2's keys always fit");
__host__ __device__ inline bool merge_part_cached(int W, int S)
{
    return static_cast<int64_t>((W + S - 1) / S) * W <= kMergeCacheKeys;
}
static_assert(kGather % 4 == 0, "gathered float4 groups stay 16-byte aligned");
static_assert(4 * kSelThreads >= BG_MAX_BEAM, "there are at least W group maxima");
static_assert(kSelThreads / 32 <= 32, "one warp holds the per-warp totals");
static_assert(kCap >= 2 * kSelThreads, "ck/ci hold the register sort's two exchange halves");
static_assert(kSelThreads >= BG_MAX_BEAM, "a selection sorts W entries at once");

// Order-preserving map fp32 -> uint32: a larger float gets a larger key (-inf lowest).
__device__ __forceinline__ uint32_t f2key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Shared state of a selection; CAP = the entries ck/ci hold.
template <int CAP>
struct SelState {
    uint32_t hist[kBins];
    uint32_t ck[CAP];
    int32_t ci[CAP];
    float red_m[kSelThreads / 32];
    float red_s[kSelThreads / 32];
    uint32_t warp_tot[kSelThreads / 32];
    int n_cand;
    uint32_t digit;        // selected bin of the current level
    uint32_t above;        // keys in higher bins of the current level (plus earlier levels)
};
using SelShared = SelState<kCap>;

struct RowShared : SelState<kCap> {
    int count;             // logits gathered by the second pass
};

// Finds, over hist[0..nbins), the bin d where the count of keys in bins >= d first
// reaches `need` (counting from the top).  Writes sh.digit = d and adds the count of
// keys in bins > d to sh.above.  nbins = kBins or 256; all threads call it.
template <class Sh>
__device__ void find_digit(Sh &sh, int nbins, uint32_t need)
{
    const int tid = threadIdx.x;
    const int per = nbins / kSelThreads > 0 ? nbins / kSelThreads : 1;   // bins per thread (8 or 1)
    const int active = nbins / per;                                      // threads that own bins
    // thread t owns bins [top - per*(t+1) + 1, top - per*t], counted from the top
    uint32_t local = 0;
    if (tid < active)
        for (int k = 0; k < per; ++k) local += sh.hist[nbins - 1 - (tid * per + k)];
    // exclusive scan of `local` over threads (descending bin order)
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh.warp_tot[warp] = incl;
    __syncthreads();
    // totals of the warps before this one: lane w < warp contributes warp w's, summed over the warp
    uint32_t before = lane < warp ? sh.warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    const uint32_t excl = before + incl - local;
    __syncthreads();
    if (tid < active && excl < need && excl + local >= need) {
        uint32_t acc = excl;
        for (int k = 0; k < per; ++k) {
            const int bin = nbins - 1 - (tid * per + k);
            const uint32_t c = sh.hist[bin];
            if (acc + c >= need) {
                sh.digit = static_cast<uint32_t>(bin);
                sh.above += acc;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

// Calls body(i, key(i)) for every element i < n owned by this thread, loading eight
// keys before using any, so that eight loads per thread are in flight.
template <typename KeyFn, typename Body>
__device__ __forceinline__ void for_each_key(int n, KeyFn key, Body body)
{
    constexpr int U = 8;
    int i = threadIdx.x;
    for (; i + (U - 1) * kSelThreads < n; i += U * kSelThreads) {
        uint32_t k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) k[u] = key(i + u * kSelThreads);
#pragma unroll
        for (int u = 0; u < U; ++u) body(i + u * kSelThreads, k[u]);
    }
    for (; i < n; i += kSelThreads) body(i, key(i));
}

// Radix narrowing of the `need` highest keys, given the level-1 histogram of key >> 20
// in sh.hist; visit(body) calls body(i, key) for every element this thread owns (keys
// of 0 may stand for elements that take no part, if need never reaches them).  Returns
// the bottom lo of a radix bin with between need and cap keys >= lo (exact = false), or,
// when the last level's bin still holds too many, the exact key T of the need-th highest
// (exact = true; sh.above = the number of keys > T, sh.hist[sh.digit] = the number of
// keys equal to T).  Leaves sh.hist in use: the caller synchronises before clearing it.
template <class Sh, typename VisitFn>
__device__ uint32_t radix_cut(Sh &sh, uint32_t need, uint32_t cap, VisitFn visit, bool &exact)
{
    const int tid = threadIdx.x;
    if (tid == 0) sh.above = 0;
    __syncthreads();
    exact = false;
    find_digit(sh, kBins, need);
    const uint32_t d1 = sh.digit;
    if (sh.above + sh.hist[d1] <= cap) return d1 << 20;
    // level 2: bits 19..8 of the keys in bin d1
    const uint32_t need1 = need - sh.above;
    __syncthreads();
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
    __syncthreads();
    visit([&](int, uint32_t k) {
        if ((k >> 20) == d1) atomicAdd(&sh.hist[(k >> 8) & 0xfffu], 1u);
    });
    __syncthreads();
    find_digit(sh, kBins, need1);
    const uint32_t d2 = sh.digit;
    if (sh.above + sh.hist[d2] <= cap) return (d1 << 20) | (d2 << 8);
    // level 3: bits 7..0 give the exact key T of the need-th element
    const uint32_t need2 = need - sh.above;
    const uint32_t pre = (d1 << 12) | d2;
    __syncthreads();
    for (int b = tid; b < 256; b += kSelThreads) sh.hist[b] = 0u;
    __syncthreads();
    visit([&](int, uint32_t k) {
        if ((k >> 8) == pre) atomicAdd(&sh.hist[k & 0xffu], 1u);
    });
    __syncthreads();
    find_digit(sh, 256, need2);
    exact = true;
    return (pre << 8) | sh.digit;
}

// Sorts one (key, token) per thread, threads [0, P) for P a power of two with
// 32 <= P <= kSelThreads, so that thread t ends with the t-th best (higher key first, equal
// keys by the smaller token); a bitonic network whose exchanges at distance < 32 are warp
// shuffles and the others go through xk/xt (two halves of 2 * kSelThreads entries,
// alternated so that one barrier per exchange suffices).  All threads call it; threads
// >= P sort their own entries among themselves (pairs never cross a multiple of P).
__device__ __forceinline__ void sort_in_registers(uint32_t &key, int32_t &tok, int P, uint32_t *xk, int32_t *xt)
{
    const int t = threadIdx.x;
    // one 64-bit value per entry, larger = better: the key, then the token inverted (smaller
    // tokens first among equal keys)
    uint64_t v = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~tok);
    int buf = 0;
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            uint64_t o;
            if (j < 32) {
                o = __shfl_xor_sync(0xffffffffu, v, j);
            } else {
                xk[buf * kSelThreads + t] = static_cast<uint32_t>(v >> 32);
                xt[buf * kSelThreads + t] = static_cast<int32_t>(static_cast<uint32_t>(v));
                __syncthreads();
                o = (static_cast<uint64_t>(xk[buf * kSelThreads + (t ^ j)]) << 32) |
                    static_cast<uint32_t>(xt[buf * kSelThreads + (t ^ j)]);
                buf ^= 1;
            }
            const bool keep_better = ((t & j) == 0) == ((t & k) == 0);
            if ((v > o) != keep_better) v = o;
        }
    }
    key = static_cast<uint32_t>(v >> 32);
    tok = static_cast<int32_t>(~static_cast<uint32_t>(v));
}

// Selection of the W highest keys of n elements (key(i) for element i; equal keys by
// smaller i), given the level-1 histogram of key >> 20 in sh.hist.  visit(body) calls
// body(i, key(i)) for every element this thread owns, in any order (the bulk passes);
// key(i) itself serves the rare in-order pass over equal keys.  At most kSelThreads
// candidates are gathered and sorted in registers; leaves the W winners sorted in
// sh.ck/ci[0..W).  n >= W >= 1, W <= kSelThreads.
template <typename KeyFn, typename VisitFn>
__device__ void select_top(SelShared &sh, int n, int W, KeyFn key, VisitFn visit)
{
    const int tid = threadIdx.x;
    bool exact;
    const uint32_t lo = radix_cut(sh, static_cast<uint32_t>(W), static_cast<uint32_t>(kSelThreads), visit, exact);
    __syncthreads();
    if (tid == 0) sh.n_cand = 0;
    __syncthreads();
    // every key >= lo (all fit), or, at the last level, the keys above T ...
    visit([&](int i, uint32_t k) {
        if (exact ? k > lo : k >= lo) {
            const int pos = atomicAdd(&sh.n_cand, 1);
            if (pos < kSelThreads) {   // always (at most kSelThreads qualify); guards shared memory
                sh.ck[pos] = k;
                sh.ci[pos] = i;
            }
        }
    });
    __syncthreads();
    if (exact) {
        // ... then the first W - above keys equal to T in index order
        const uint32_t T = lo;
        const int base = sh.n_cand;
        const int need = W - base;
        int taken = 0;
        const int lane = tid & 31, warp = tid >> 5;
        for (int c0 = 0; c0 < n && taken < need; c0 += kSelThreads) {
            const int i = c0 + tid;
            const bool eq = i < n && key(i) == T;
            const uint32_t bal = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) sh.warp_tot[warp] = __popc(bal);
            __syncthreads();
            int before = taken;
            for (int w = 0; w < warp; ++w) before += static_cast<int>(sh.warp_tot[w]);
            const int pos = before + __popc(bal & ((1u << lane) - 1u));
            if (eq && pos < need) {
                sh.ck[base + pos] = T;
                sh.ci[base + pos] = i;
            }
            int tot = 0;
            for (int w = 0; w < kSelThreads / 32; ++w) tot += static_cast<int>(sh.warp_tot[w]);
            taken += tot;
            __syncthreads();
        }
        if (tid == 0) sh.n_cand = W;
        __syncthreads();
    }
    const int nc = min(sh.n_cand, kSelThreads);
    uint32_t k = 0u;
    int32_t t = 0x7fffffff;
    if (tid < nc) {
        k = sh.ck[tid];
        t = sh.ci[tid];
    }
    __syncthreads();
    int P = 32;
    while (P < nc) P <<= 1;
    sort_in_registers(k, t, P, sh.ck, sh.ci);
    __syncthreads();
    sh.ck[tid] = k;
    sh.ci[tid] = t;
    __syncthreads();
}

// Gathers into sh.ck/ci (key, token) a superset, at most cap >= W entries, of the W best
// of the n entries in bval/btok (key descending, token ascending; entries whose token is
// V or more are padding and never count).  Returns the radix threshold lo of the gathered
// set: it holds every entry with key >= lo, or, when `strict`, every entry with key > lo
// and, of the entries tied at lo, those with the smallest tokens.
template <class Sh>
__device__ uint32_t row_reduce(Sh &sh, const float *bval, const int32_t *btok, int n, int V, int W, int cap,
                               bool &strict)
{
    const int tid = threadIdx.x;
    // an entry's key; 0 (below every logit's key) for the padding past V of a group
    auto bkey = [&](int e) -> uint32_t { return btok[e] < V ? f2key(bval[e]) : 0u; };
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
    __syncthreads();
    for (int e = tid; e < n; e += kSelThreads) atomicAdd(&sh.hist[bkey(e) >> 20], 1u);
    __syncthreads();
    auto visit = [&](auto &&body) {
        for (int e = tid; e < n; e += kSelThreads) body(e, bkey(e));
    };
    bool exact;
    const uint32_t lo = radix_cut(sh, static_cast<uint32_t>(W), static_cast<uint32_t>(cap), visit, exact);
    const uint32_t above = exact ? sh.above : 0u;
    const uint32_t n_eq = exact ? sh.hist[sh.digit] : 0u;
    __syncthreads();
    if (tid == 0) sh.n_cand = 0;
    __syncthreads();
    strict = exact;
    auto append = [&](uint32_t k, int32_t tok) {
        const int pos = atomicAdd(&sh.n_cand, 1);
        if (pos < cap) {   // always (at most cap entries qualify); guards shared memory
            sh.ck[pos] = k;
            sh.ci[pos] = tok;
        }
    };
    if (!exact || above + n_eq <= static_cast<uint32_t>(cap)) {
        // every entry >= lo fits (with exact: all the entries tied at T come along)
        visit([&](int e, uint32_t k) {
            if (k >= lo) append(k, btok[e]);
        });
    } else {
        // More entries tie at T than fit: the entries above T, then of the tied ones those
        // with the smallest tokens, by the same radix narrowing over ~token (distinct keys,
        // all >= 2^31 since tokens < 2^31; entries off T take key 0 and no part).
        visit([&](int e, uint32_t k) {
            if (k > lo) append(k, btok[e]);
        });
        auto visit_tok = [&](auto &&body) {
            for (int e = tid; e < n; e += kSelThreads)
                body(e, bkey(e) == lo ? ~static_cast<uint32_t>(btok[e]) : 0u);
        };
        for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
        __syncthreads();
        visit_tok([&](int, uint32_t k) {
            if (k) atomicAdd(&sh.hist[k >> 20], 1u);
        });
        __syncthreads();
        bool exact_tok;
        const uint32_t lo_tok = radix_cut(sh, static_cast<uint32_t>(W) - above, static_cast<uint32_t>(cap) - above,
                                          visit_tok, exact_tok);
        __syncthreads();
        visit_tok([&](int e, uint32_t k) {
            if (k && k >= lo_tok) append(lo, btok[e]);
        });
    }
    __syncthreads();
    if (tid == 0 && sh.n_cand > cap) sh.n_cand = cap;
    __syncthreads();
    return lo;
}

// Streams the float4 groups [0, n4) of a row, this thread taking every kSelThreads-th:
// consume(f, i0) gets four float4 at a time, groups i0 + u * kSelThreads (u < 4, -inf
// past the row).  kRowLoads loads are in flight before the first is used, and each half
// is reissued for the next batch as soon as it has been consumed.  Batches wholly inside
// the row load without bounds checks; only the last, partial one checks.  Every thread
// runs the same iterations (consume may use warp-wide votes).
template <typename Load, typename Consume>
__device__ __forceinline__ void stream_row(int n4, Load load, Consume consume)
{
    constexpr int U = kRowLoads, H = kRowLoads / 2;
    constexpr int kStep = U * kSelThreads;
    const float4 pad = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const int tid = static_cast<int>(threadIdx.x);
    const int nfull = n4 / kStep;                       // batches with every group in the row
    const bool tail = nfull * kStep < n4;
    auto fetch_tail = [&](int b0, int u) -> float4 {
        const int i = b0 + tid + u * kSelThreads;
        return i < n4 ? load(i) : pad;
    };
    float4 f[U];
    if (nfull > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) f[u] = load(tid + u * kSelThreads);
    } else {
#pragma unroll
        for (int u = 0; u < U; ++u) f[u] = fetch_tail(0, u);
    }
    for (int b = 0; b < nfull; ++b) {
        const int b0 = b * kStep, nx = b0 + kStep;
        const bool next_full = b + 1 < nfull;
        consume(f, b0 + tid);
        if (next_full) {
#pragma unroll
            for (int u = 0; u < H; ++u) f[u] = load(nx + tid + u * kSelThreads);
        } else if (tail) {
#pragma unroll
            for (int u = 0; u < H; ++u) f[u] = fetch_tail(nx, u);
        }
        consume(f + H, b0 + tid + H * kSelThreads);
        if (next_full) {
#pragma unroll
            for (int u = H; u < U; ++u) f[u] = load(nx + tid + u * kSelThreads);
        } else if (tail) {
#pragma unroll
            for (int u = H; u < U; ++u) f[u] = fetch_tail(nx, u);
        }
    }
    if (tail) {
        const int b0 = nfull * kStep;
        consume(f, b0 + tid);
        consume(f + H, b0 + tid + H * kSelThreads);
    }
}

template <bool VEC>
__global__ void __launch_bounds__(kSelThreads)
    row_select_kernel(const float *__restrict__ logits, int32_t V, int32_t W, float *__restrict__ cand_val,
                      int32_t *__restrict__ cand_tok, float *__restrict__ row_lse)
{
    __shared__ RowShared sh;
    extern __shared__ __align__(16) uint32_t row_buf[];
    float *bval = reinterpret_cast<float *>(row_buf);
    int32_t *btok = reinterpret_cast<int32_t *>(row_buf + kGather);
    grid_dep_launch();
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
    if (tid == 0) sh.count = 0;
    grid_dep_wait();     // the previous kernel of the stream has completed
    __syncthreads();
    const int64_t row = blockIdx.x;
    const float *x = logits + row * static_cast<int64_t>(V);
    const int n4 = (V + 3) >> 2;
    // group maxima kept for the second pass: this thread's j-th group (float4 tid + j *
    // kSelThreads) at halfword tid * kJ + j, kJ = its groups rounded up to whole batches
    const bool stored = n4 <= kMaxStored;
    constexpr int kStep = kRowLoads * kSelThreads;
    const int kJ = kRowLoads * ((n4 + kStep - 1) / kStep);
    // this thread's kJ halfwords, past the gather buffer; allocated and touched only if stored
    uint32_t *smax = row_buf + 2 * kGather + tid * (kJ / 2);
    // float4 group i of the row: logits 4i .. 4i+3 (-inf past V); VEC: V % 4 == 0, so the
    // rows start 16-byte aligned, as the logits do
    auto load_keep = [&](int i) -> float4 {      // first pass: the second reads it again (L2)
        const int e = 4 * i;
        if (VEC) return *reinterpret_cast<const float4 *>(x + e);
        return make_float4(x[e], e + 1 < V ? x[e + 1] : -INFINITY, e + 2 < V ? x[e + 2] : -INFINITY,
                           e + 3 < V ? x[e + 3] : -INFINITY);
    };
    auto load_last = [&](int i) -> float4 {      // second pass: the row's last use
        const int e = 4 * i;
        if (VEC) return __ldcs(reinterpret_cast<const float4 *>(x + e));
        return make_float4(__ldcs(x + e), e + 1 < V ? __ldcs(x + e + 1) : -INFINITY,
                           e + 2 < V ? __ldcs(x + e + 2) : -INFINITY, e + 3 < V ? __ldcs(x + e + 3) : -INFINITY);
    };

    // Pass 1 (HBM): the row's logsumexp, and the maximum of each of this thread's four
    // interleaved groups of logits (components x, y, z, w of its float4 loads).
    constexpr float kL2E = 1.4426950408889634f;
    // Sum of exponentials relative to a lazily raised reference m (base-2 units):
    // e^(x - M) = 2^(x log2e - m) * 2^(m - M log2e); m is raised (the sum rescaled) only
    // when the running maximum exceeds it by more than 2^8, checked once per 16 logits.
    float m = -INFINITY;
    float2 acc = make_float2(0.f, 0.f);
    const float2 l2e2 = make_float2(kL2E, kL2E);
    float4 gmax = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    stream_row(n4, load_keep, [&](const float4 *f, int i0) {
        if (stored) {
            // the four groups' maxima as bf16 truncated toward zero (a monotone map, so a
            // group whose maximum is >= the bound keeps a stored value >= the truncated bound)
            uint32_t b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                b[u] = __float_as_uint(fmaxf(fmaxf(f[u].x, f[u].y), fmaxf(f[u].z, f[u].w)));
            const int j0 = (i0 - tid) / kSelThreads;   // a multiple of 4
            *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(smax) + j0) =
                make_uint2(__byte_perm(b[0], b[1], 0x7632), __byte_perm(b[2], b[3], 0x7632));
        }
        gmax.x = fmaxf(fmaxf(gmax.x, f[0].x), fmaxf(fmaxf(f[1].x, f[2].x), f[3].x));
        gmax.y = fmaxf(fmaxf(gmax.y, f[0].y), fmaxf(fmaxf(f[1].y, f[2].y), f[3].y));
        gmax.z = fmaxf(fmaxf(gmax.z, f[0].z), fmaxf(fmaxf(f[1].z, f[2].z), f[3].z));
        gmax.w = fmaxf(fmaxf(gmax.w, f[0].w), fmaxf(fmaxf(f[1].w, f[2].w), f[3].w));
        // the running maximum so far bounds these 16 logits as well as the batch's own would
        const float ml = fmaxf(fmaxf(gmax.x, gmax.y), fmaxf(gmax.z, gmax.w)) * kL2E;
        if (ml > m + 8.f) {
            const float al = (m == -INFINITY) ? 0.f : ex2(m - ml);
            acc = fmul2(acc, make_float2(al, al));
            m = ml;
        }
        if (m > -INFINITY) {
            const float2 nm = make_float2(-m, -m);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 x01 = ffma2(make_float2(f[u].x, f[u].y), l2e2, nm);
                const float2 x23 = ffma2(make_float2(f[u].z, f[u].w), l2e2, nm);
                acc = fadd2(acc, fadd2(make_float2(ex2(x01.x), ex2(x01.y)), make_float2(ex2(x23.x), ex2(x23.y))));
            }
        }
    });
    // the group maxima into the level-1 histogram (padding-only groups count as -inf)
    atomicAdd(&sh.hist[f2key(gmax.x) >> 20], 1u);
    atomicAdd(&sh.hist[f2key(gmax.y) >> 20], 1u);
    atomicAdd(&sh.hist[f2key(gmax.z) >> 20], 1u);
    atomicAdd(&sh.hist[f2key(gmax.w) >> 20], 1u);
    // logsumexp: back to (max in natural units, sum relative to it), combined over the CTA
    float s = acc.x + acc.y;
    m = m * 0.69314718055994530942f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float mn = fmaxf(m, m2);
        if (mn > -INFINITY) {
            s = s * ex2((m - mn) * kL2E) + s2 * ex2((m2 - mn) * kL2E);
            m = mn;
        }
    }
    if (lane == 0) {
        sh.red_m[warp] = m;
        sh.red_s[warp] = s;
    }
    __syncthreads();
    if (tid == 0) {
        float M = -INFINITY, S = 0.f;
        for (int w = 0; w < kSelThreads / 32; ++w) {
            const float mn = fmaxf(M, sh.red_m[w]);
            if (mn > -INFINITY) {
                S = S * ex2((M - mn) * kL2E) + sh.red_s[w] * ex2((sh.red_m[w] - mn) * kL2E);
                M = mn;
            }
        }
        row_lse[row] = M + __logf(S);
        sh.above = 0;
    }
    __syncthreads();
    // The bound lo: at least W group maxima have keys >= lo, and those maxima are W
    // distinct logits, so every logit with key < lo has W better ones and cannot be kept.
    // The radix narrowing over the maxima stops once at most bound_cap of them are >= lo,
    // which leaves about as many logits >= lo (rarely more than one per group).
    const uint32_t gk[4] = {f2key(gmax.x), f2key(gmax.y), f2key(gmax.z), f2key(gmax.w)};
    bool lo_exact;
    const int bound_cap = min(kBoundCap, W + W / 2 + 32);   // >= W; fewer above the bound, fewer to sort
    const uint32_t lo = radix_cut(sh, static_cast<uint32_t>(W), static_cast<uint32_t>(bound_cap),
                                  [&](auto &&body) {
#pragma unroll
                                      for (int c = 0; c < 4; ++c) body(c, gk[c]);
                                  },
                                  lo_exact);
    const float tf = lo <= 0x007fffffu ? -INFINITY : key2f(lo);   // keys below -inf's: NaN patterns

    // Pass 2: gather every float4 group holding a logit >= tf (its other logits come along as
    // harmless extra entries).
    const uint32_t lt_mask = (1u << lane) - 1u;
    if (stored) {
        // only the groups whose stored maximum passes the truncated bound are read again
        const uint32_t tb = __float_as_uint(tf) >> 16;   // the bound truncated to bf16, twice
        const uint32_t tbb = tb | (tb << 16);
        const __nv_bfloat162 bound2 = *reinterpret_cast<const __nv_bfloat162 *>(&tbb);
        for (int c = 0; c < kJ / 8; ++c) {
            const uint4 w4 = reinterpret_cast<const uint4 *>(smax)[c];
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w[q]), bound2);
                if (m) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int i = tid + (8 * c + 2 * q + h) * kSelThreads;
                        if (((m >> (16 * h)) & 1u) && i < n4) {
                            const float4 f = load_last(i);
                            const int pos = atomicAdd(&sh.count, 4);
                            if (pos + 4 <= kGather) {
                                *reinterpret_cast<float4 *>(bval + pos) = f;
                                *reinterpret_cast<int4 *>(btok + pos) =
                                    make_int4(4 * i, 4 * i + 1, 4 * i + 2, 4 * i + 3);
                            }
                        }
                    }
                }
            }
        }
    } else {
    stream_row(n4, load_last, [&](const float4 *f, int i0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kSelThreads;
            // (padding past the row is -inf: it passes only when tf is -inf, and its tokens
            // past V give it key 0 below)
            const bool hit = fmaxf(fmaxf(f[u].x, f[u].y), fmaxf(f[u].z, f[u].w)) >= tf;
            const uint32_t bal = __ballot_sync(0xffffffffu, hit);
            if (bal) {
                int base = 0;
                if (lane == 0) base = atomicAdd(&sh.count, 4 * __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                const int pos = base + 4 * __popc(bal & lt_mask);
                if (hit && pos + 4 <= kGather) {
                    *reinterpret_cast<float4 *>(bval + pos) = f[u];
                    *reinterpret_cast<int4 *>(btok + pos) = make_int4(4 * i, 4 * i + 1, 4 * i + 2, 4 * i + 3);
                }
            }
        }
    });
    }
    __syncthreads();
    const int n = sh.count;
    // an entry's key; the padding past V of a group takes key 0, below every logit's key
    auto entry_key = [&](int e) -> uint32_t { return btok[e] < V ? f2key(bval[e]) : 0u; };
    uint32_t key = 0u;
    int32_t tok = 0x7fffffff;
    int n_sort;                 // entries to sort, at most kSelThreads
    if (n <= kGather) {
        // the gathered logits with key >= lo (the rest of their groups dropped) into ck/ci
        if (tid == 0) sh.n_cand = 0;
        __syncthreads();
        for (int e0 = 0; e0 < n; e0 += kSelThreads) {
            const int e = e0 + tid;
            const uint32_t k = e < n ? entry_key(e) : 0u;
            const bool keep = e < n && k >= lo && k != 0u;
            const uint32_t bal = __ballot_sync(0xffffffffu, keep);
            if (bal) {
                int base = 0;
                if (lane == 0) base = atomicAdd(&sh.n_cand, __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                const int pos = base + __popc(bal & lt_mask);
                if (keep && pos < kCap) {
                    sh.ck[pos] = k;
                    sh.ci[pos] = btok[e];
                }
            }
        }
        __syncthreads();
        const int kept = sh.n_cand;
        if (kept <= kSelThreads) {
            n_sort = kept;
        } else {
            // narrow the gathered entries to at most kSelThreads containing the W best
            __syncthreads();
            bool st;
            row_reduce(sh, bval, btok, n, V, W, kSelThreads, st);
            n_sort = sh.n_cand;
        }
    } else {
        // more logits at the bound than fit (ties, or a flat row): the full radix selection
        // over the row, a level-1 histogram pass and then the narrowing passes
        for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
        __syncthreads();
        auto rkey = [&](int i) -> uint32_t { return f2key(x[i]); };
        auto visit = [&](auto &&body) { for_each_key(V, rkey, body); };
        visit([&](int, uint32_t k) { atomicAdd(&sh.hist[k >> 20], 1u); });
        __syncthreads();
        select_top(sh, V, W, rkey, visit);
        n_sort = W;           // the W best, already in order
    }
    if (tid < n_sort) {
        key = sh.ck[tid];
        tok = sh.ci[tid];
    }
    __syncthreads();   // ck/ci serve as the sort's exchange buffers next
    int P = 32;
    while (P < n_sort) P <<= 1;
    sort_in_registers(key, tok, P, sh.ck, sh.ci);
    if (tid < W) {
        cand_val[row * W + tid] = key2f(key);
        cand_tok[row * W + tid] = tok;
    }
}

// Merge, level 1: CTA (r, s) selects the W best of the local candidates of beams
// [s*W/S, (s+1)*W/S) of request r and writes their score keys and candidate numbers
// i = b * W + k (its slice is the contiguous range of i starting at b0 * W).
__global__ void __launch_bounds__(kSelThreads)
    merge_part_kernel(const float *__restrict__ cand_val, const float *__restrict__ row_lse,
                      const float *__restrict__ cum, int32_t W, int32_t S, uint32_t *__restrict__ part_key,
                      int32_t *__restrict__ part_idx, const int32_t *__restrict__ cand_tok,
                      int32_t *__restrict__ token_out, int32_t *__restrict__ parent_out, float *__restrict__ score_out)
{
    __shared__ SelShared sh;
    grid_dep_launch();
    const int tid = threadIdx.x;
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
    grid_dep_wait();     // the row selection has completed
    __syncthreads();
    const int64_t r = blockIdx.x / S;
    const int s = static_cast<int>(blockIdx.x - r * S);
    const int b0 = static_cast<int>((static_cast<int64_t>(s) * W) / S);
    const int b1 = static_cast<int>((static_cast<int64_t>(s + 1) * W) / S);
    const int base = b0 * W;
    const int n = (b1 - b0) * W;                      // >= W: every slice holds at least one beam
    const float *val = cand_val + r * W * W;
    const float *lse = row_lse + r * W;
    const float *cr = cum + r * W;
    // local candidate p = candidate base + p: the k-th best token of beam b; its score as a key
    auto score_key = [&](int p) -> uint32_t {
        const int i = base + p;
        const int b = i / W;
        return f2key(cr[b] + (val[i] - lse[b]));
    };
    // the keys once into shared memory when they fit (every selection pass reads them again),
    // with the level-1 histogram on the way
    extern __shared__ __align__(16) uint32_t mkeys[];
    const bool cached = merge_part_cached(W, S);
    for_each_key(n, score_key, [&](int p, uint32_t k) {
        if (cached) mkeys[p] = k;
        atomicAdd(&sh.hist[k >> 20], 1u);
    });
    __syncthreads();
    auto key = [&](int p) -> uint32_t { return cached ? mkeys[p] : score_key(p); };
    // equal scores: the smaller candidate number is the smaller b * V + v (beams in order,
    // and a beam's candidates with equal scores have equal logits, kept in token order)
    select_top(sh, n, W, key, [&](auto &&body) { for_each_key(n, key, body); });
    const int64_t out = blockIdx.x * static_cast<int64_t>(W);
    if (S == 1) {
        // one slice holds the whole request: these are the request's W best
        for (int k = tid; k < W; k += kSelThreads) {
            const int i = base + sh.ci[k];
            token_out[r * W + k] = cand_tok[r * W * W + i];
            parent_out[r * W + k] = i / W;
            score_out[r * W + k] = key2f(sh.ck[k]);
        }
        return;
    }
    for (int k = tid; k < W; k += kSelThreads) {
        part_key[out + k] = sh.ck[k];
        part_idx[out + k] = base + sh.ci[k];
    }
}

// Merge, level 2: one CTA per request selects the W best of its S * W level-1 survivors.
// Survivors are stored slice by slice (beams ascending), each slice best first with equal
// keys by candidate number, so equal keys keep candidate order by their position too.
__global__ void __launch_bounds__(kSelThreads)
    merge_final_kernel(const uint32_t *__restrict__ part_key, const int32_t *__restrict__ part_idx,
                       const int32_t *__restrict__ cand_tok, int32_t W, int32_t S, int32_t *__restrict__ token_out,
                       int32_t *__restrict__ parent_out, float *__restrict__ score_out)
{
    __shared__ SelShared sh;
    grid_dep_launch();
    const int tid = threadIdx.x;
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
    grid_dep_wait();     // level 1 has completed
    __syncthreads();
    const int64_t r = blockIdx.x;
    const int n = S * W;
    const uint32_t *pk = part_key + r * n;
    const int32_t *pi = part_idx + r * n;
    extern __shared__ __align__(16) uint32_t mkeys[];
    for_each_key(
        n, [&](int p) -> uint32_t { return pk[p]; },
        [&](int p, uint32_t k) {
            mkeys[p] = k;
            atomicAdd(&sh.hist[k >> 20], 1u);
        });
    __syncthreads();
    auto key = [&](int p) -> uint32_t { return mkeys[p]; };
    select_top(sh, n, W, key, [&](auto &&body) { for_each_key(n, key, body); });
    for (int k = tid; k < W; k += kSelThreads) {
        const int i = pi[sh.ci[k]];
        token_out[r * W + k] = cand_tok[r * W * W + i];
        parent_out[r * W + k] = i / W;
        score_out[r * W + k] = key2f(sh.ck[k]);
    }
}

}  // namespace

int beam_select_slices(int32_t R, int32_t W)
{
    // one level when a request's W x W candidates fit one CTA's key cache; otherwise about two
    // level-1 CTAs per SM over the requests, every slice keeping at least one beam
    if (static_cast<int64_t>(W) * W <= kMergeCacheKeys) return 1;
    int S = static_cast<int>((2 * 152 + R - 1) / (R > 0 ? R : 1));
    if (S > W) S = W;
    if (S > 16) S = 16;
    return S < 1 ? 1 : S;
}

cudaError_t launch_beam_select(const float *logits, const float *cum, int32_t R, int32_t W, int32_t V,
                               int32_t *token_out, int32_t *parent_out, float *score_out, float *cand_val,
                               int32_t *cand_tok, float *row_lse, uint32_t *part_key, int32_t *part_idx,
                               cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(R) * W;
    if (rows == 0) return cudaSuccess;
    const int S = beam_select_slices(R, W);
    static std::atomic<uint64_t> smem_set_vec{0}, smem_set_any{0};
    const bool vec = (V & 3) == 0;
    auto kern = vec ? row_select_kernel<true> : row_select_kernel<false>;
    cudaError_t e = ensure_smem_attribute(kern, kRowDynSmemMax, vec ? smem_set_vec : smem_set_any);
    if (e != cudaSuccess) return e;
    // the gather buffer, plus the stored group maxima when the row has at most kMaxStored groups
    const int n4 = (V + 3) / 4;
    constexpr int kStep = kRowLoads * kSelThreads;
    const int kj = kRowLoads * ((n4 + kStep - 1) / kStep);
    const size_t dyn = static_cast<size_t>(kGatherSmem) + (n4 <= kMaxStored ? static_cast<size_t>(kSelThreads) * kj * 2 : 0);
    e = launch_dependent(kern, dim3(static_cast<unsigned>(rows)), dim3(kSelThreads), dyn, stream, logits, V, W,
                         cand_val, cand_tok, row_lse);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> smem_set_part{0}, smem_set_final{0};
    e = ensure_smem_attribute(merge_part_kernel, kMergeSmemMax, smem_set_part);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attribute(merge_final_kernel, kMergeSmemMax, smem_set_final);
    if (e != cudaSuccess) return e;
    const size_t part_smem = merge_part_cached(W, S) ? static_cast<size_t>((W + S - 1) / S) * W * 4 : 0;
    const size_t final_smem = static_cast<size_t>(S) * W * 4;
    e = launch_dependent(merge_part_kernel, dim3(static_cast<unsigned>(static_cast<int64_t>(R) * S)),
                         dim3(kSelThreads), part_smem, stream, static_cast<const float *>(cand_val),
                         static_cast<const float *>(row_lse), cum, W, S, part_key, part_idx,
                         static_cast<const int32_t *>(cand_tok), token_out, parent_out, score_out);
    if (e != cudaSuccess || S == 1) return e;   // one slice: level 1 wrote the result
    return launch_dependent(merge_final_kernel, dim3(static_cast<unsigned>(R)), dim3(kSelThreads), final_smem, stream,
                            static_cast<const uint32_t *>(part_key), static_cast<const int32_t *>(part_idx),
                            static_cast<const int32_t *>(cand_tok), W, S, token_out, parent_out, score_out);
}

}  // namespace bg
