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
// Two launches on the caller's stream:
//   1. row_select_kernel, one CTA per beam row: one pass over the row from HBM
//      computes its logsumexp (online max and sum of exponentials) and a
//      4096-bin histogram of the top 12 bits of an order-preserving integer key
//      of every logit; a second pass (the row is still in L2) gathers the
//      logits at or above the bin that holds the W-th largest into shared
//      memory (two more radix levels narrow the bin when it holds too many), a
//      bitonic sort orders them, and the beam's W best (value, token) and its
//      logsumexp go to the workspace.  A beam's W best tokens contain its whole
//      share of the request's W best candidates.
//   2. the merge, the same selection over the W x W local candidates of a request keyed
//      by their scores, in two levels so that more than R CTAs share it:
//      merge_part_kernel selects the W best of each of S slices of beams, and
//      merge_final_kernel the W best of the S * W survivors of each request.
// HBM-bound: the logits are read once; everything else stays on chip or in L2.
#include "bg_internal.h"
#include "bg_ptx.cuh"

#include <stdint.h>

namespace bg {
namespace {

constexpr int kSelThreads = 512;
constexpr int kCap = 2048;          // candidates a CTA can gather and sort
constexpr int kBins = 4096;         // 12-bit radix digits

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

struct SelShared {
    uint32_t hist[kBins];
    uint32_t ck[kCap];
    int32_t ci[kCap];
    float red_m[kSelThreads / 32];
    float red_s[kSelThreads / 32];
    uint32_t warp_tot[kSelThreads / 32];
    int n_cand;
    uint32_t digit;        // selected bin of the current level
    uint32_t above;        // keys in higher bins of the current level (plus earlier levels)
};

// Finds, over hist[0..nbins), the bin d where the count of keys in bins >= d first
// reaches `need` (counting from the top).  Writes sh.digit = d and adds the count of
// keys in bins > d to sh.above.  nbins = kBins or 256; all threads call it.
__device__ void find_digit(SelShared &sh, int nbins, uint32_t need)
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
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += sh.warp_tot[w];
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

// Sorts sh.ck/ci[0..n) (padded to a power of two with sentinels) so that higher keys
// come first and equal keys keep the smaller index first.
__device__ void sort_candidates(SelShared &sh, int n)
{
    int P = 2;
    while (P < n) P <<= 1;
    for (int i = n + threadIdx.x; i < P; i += kSelThreads) {
        sh.ck[i] = 0u;
        sh.ci[i] = 0x7fffffff;
    }
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < P; i += kSelThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const uint32_t ka = sh.ck[i], kb = sh.ck[l];
                    const int32_t ia = sh.ci[i], ib = sh.ci[l];
                    const bool a_first = ka > kb || (ka == kb && ia < ib);
                    const bool first_half = (i & k) == 0;
                    if (first_half != a_first) {
                        sh.ck[i] = kb;
                        sh.ck[l] = ka;
                        sh.ci[i] = ib;
                        sh.ci[l] = ia;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Calls body(i, key(i)) for every element i < n owned by this thread, loading eight
// keys before using any, so that eight loads per thread are in flight (the passes
// over a row are otherwise bound by load latency, not bandwidth).
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

// Selection of the W highest keys of n elements (key(i) for element i; equal keys by
// smaller i), given the level-1 histogram of key >> 20 in sh.hist.  visit(body) calls
// body(i, key(i)) for every element this thread owns, in any order (the bulk passes);
// key(i) itself serves the rare in-order pass over equal keys.  Leaves the W winners
// sorted in sh.ck/ci[0..W).  n >= W >= 1.
template <typename KeyFn, typename VisitFn>
__device__ void select_top(SelShared &sh, int n, int W, KeyFn key, VisitFn visit)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        sh.above = 0;
        sh.n_cand = 0;
    }
    __syncthreads();
    find_digit(sh, kBins, static_cast<uint32_t>(W));
    const uint32_t d1 = sh.digit;
    uint32_t lo_key;                    // gather every key >= lo_key (all fit) ...
    bool exact = false;                 // ... or, at the last level, keys > T and the first equal ones
    if (sh.above + sh.hist[d1] <= static_cast<uint32_t>(kCap)) {
        lo_key = d1 << 20;
    } else {
        // level 2: bits 19..8 of the keys in bin d1
        const uint32_t need1 = static_cast<uint32_t>(W) - sh.above;
        __syncthreads();
        for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
        __syncthreads();
        visit([&](int, uint32_t k) {
            if ((k >> 20) == d1) atomicAdd(&sh.hist[(k >> 8) & 0xfffu], 1u);
        });
        __syncthreads();
        find_digit(sh, kBins, need1);
        const uint32_t d2 = sh.digit;
        if (sh.above + sh.hist[d2] <= static_cast<uint32_t>(kCap)) {
            lo_key = (d1 << 20) | (d2 << 8);
        } else {
            // level 3: bits 7..0 give the exact key T of the W-th element
            const uint32_t need2 = static_cast<uint32_t>(W) - sh.above;
            const uint32_t pre = (d1 << 12) | d2;
            __syncthreads();
            for (int b = tid; b < 256; b += kSelThreads) sh.hist[b] = 0u;
            __syncthreads();
            visit([&](int, uint32_t k) {
                if ((k >> 8) == pre) atomicAdd(&sh.hist[k & 0xffu], 1u);
            });
            __syncthreads();
            find_digit(sh, 256, need2);
            lo_key = (pre << 8) | sh.digit;
            exact = true;
        }
    }
    __syncthreads();
    if (!exact) {
        visit([&](int i, uint32_t k) {
            if (k >= lo_key) {
                const int pos = atomicAdd(&sh.n_cand, 1);
                sh.ck[pos] = k;
                sh.ci[pos] = i;
            }
        });
        __syncthreads();
    } else {
        // keys above T (fewer than W), then the first W - above keys equal to T in index order
        const uint32_t T = lo_key;
        visit([&](int i, uint32_t k) {
            if (k > T) {
                const int pos = atomicAdd(&sh.n_cand, 1);
                sh.ck[pos] = k;
                sh.ci[pos] = i;
            }
        });
        __syncthreads();
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
    sort_candidates(sh, sh.n_cand);
}

__global__ void __launch_bounds__(kSelThreads)
    row_select_kernel(const float *__restrict__ logits, int32_t V, int32_t W, float *__restrict__ cand_val,
                      int32_t *__restrict__ cand_tok, float *__restrict__ row_lse)
{
    __shared__ SelShared sh;
    grid_dep_launch();
    const int tid = threadIdx.x;
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0u;
    grid_dep_wait();     // the previous kernel of the stream has completed
    __syncthreads();
    const int64_t row = blockIdx.x;
    const float *x = logits + row * static_cast<int64_t>(V);
    constexpr float kL2E = 1.4426950408889634f;
    // pass 1: online max / sum of exponentials and the level-1 histogram
    float m = -INFINITY, s = 0.f;
    auto add4 = [&](float a, float b, float c, float d) {
        const float mx = fmaxf(fmaxf(a, b), fmaxf(c, d));
        const float mn = fmaxf(m, mx);
        if (mn > -INFINITY) {
            const float nl = -mn * kL2E;   // 2^(x log2e - mn log2e) = e^(x - mn), one FFMA per exponent
            s = s * ex2(fmaf(m, kL2E, nl)) + ex2(fmaf(a, kL2E, nl)) + ex2(fmaf(b, kL2E, nl)) + ex2(fmaf(c, kL2E, nl)) +
                ex2(fmaf(d, kL2E, nl));
            m = mn;
        }
        atomicAdd(&sh.hist[f2key(a) >> 20], 1u);
        atomicAdd(&sh.hist[f2key(b) >> 20], 1u);
        atomicAdd(&sh.hist[f2key(c) >> 20], 1u);
        atomicAdd(&sh.hist[f2key(d) >> 20], 1u);
    };
    if ((V & 3) == 0) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        const int n4 = V / 4;
        int i = tid;
        for (; i + 3 * kSelThreads < n4; i += 4 * kSelThreads) {
            float4 f[4];   // four loads in flight before any is used
#pragma unroll
            for (int u = 0; u < 4; ++u) f[u] = x4[i + u * kSelThreads];   // default caching: read again by the gather
#pragma unroll
            for (int u = 0; u < 4; ++u) add4(f[u].x, f[u].y, f[u].z, f[u].w);
        }
        for (; i < n4; i += kSelThreads) {
            const float4 f = x4[i];
            add4(f.x, f.y, f.z, f.w);
        }
    } else {
        for (int i = tid; i < V; i += kSelThreads) {
            const float a = x[i];
            const float mn = fmaxf(m, a);
            if (mn > -INFINITY) {
                s = s * ex2((m - mn) * kL2E) + ex2((a - mn) * kL2E);
                m = mn;
            }
            atomicAdd(&sh.hist[f2key(a) >> 20], 1u);
        }
    }
    // combine (m, s) over the CTA
    const int lane = tid & 31, warp = tid >> 5;
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
    }
    // pass 2 onward: the W best logits of the row (the row is still in L2)
    // evict-first: the gather pass is the row's last use
    auto key = [&](int i) -> uint32_t { return f2key(__ldcs(x + i)); };
    auto visit = [&](auto &&body) {
        if ((V & 3) == 0) {
            // four float4 loads in flight per thread, four keys per load
            const float4 *x4 = reinterpret_cast<const float4 *>(x);
            const int n4 = V / 4;
            int j = tid;
            for (; j + 3 * kSelThreads < n4; j += 4 * kSelThreads) {
                float4 f[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) f[u] = __ldcs(x4 + j + u * kSelThreads);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = 4 * (j + u * kSelThreads);
                    body(i, f2key(f[u].x));
                    body(i + 1, f2key(f[u].y));
                    body(i + 2, f2key(f[u].z));
                    body(i + 3, f2key(f[u].w));
                }
            }
            for (; j < n4; j += kSelThreads) {
                const float4 f = __ldcs(x4 + j);
                body(4 * j, f2key(f.x));
                body(4 * j + 1, f2key(f.y));
                body(4 * j + 2, f2key(f.z));
                body(4 * j + 3, f2key(f.w));
            }
        } else {
            for_each_key(V, key, body);
        }
    };
    select_top(sh, V, W, key, visit);
    for (int k = tid; k < W; k += kSelThreads) {
        cand_val[row * W + k] = key2f(sh.ck[k]);
        cand_tok[row * W + k] = sh.ci[k];
    }
}

// Merge, level 1: CTA (r, s) selects the W best of the local candidates of beams
// [s*W/S, (s+1)*W/S) of request r and writes their score keys and candidate numbers
// i = b * W + k (its slice is the contiguous range of i starting at b0 * W).
__global__ void __launch_bounds__(kSelThreads)
    merge_part_kernel(const float *__restrict__ cand_val, const float *__restrict__ row_lse,
                      const float *__restrict__ cum, int32_t W, int32_t S, uint32_t *__restrict__ part_key,
                      int32_t *__restrict__ part_idx)
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
    auto key = [&](int p) -> uint32_t {
        const int i = base + p;
        const int b = i / W;
        return f2key(cr[b] + (val[i] - lse[b]));
    };
    for_each_key(n, key, [&](int, uint32_t k) { atomicAdd(&sh.hist[k >> 20], 1u); });
    __syncthreads();
    // equal scores: the smaller candidate number is the smaller b * V + v (beams in order,
    // and a beam's candidates with equal scores have equal logits, kept in token order)
    select_top(sh, n, W, key, [&](auto &&body) { for_each_key(n, key, body); });
    const int64_t out = blockIdx.x * static_cast<int64_t>(W);
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
    auto key = [&](int p) -> uint32_t { return pk[p]; };
    for_each_key(n, key, [&](int, uint32_t k) { atomicAdd(&sh.hist[k >> 20], 1u); });
    __syncthreads();
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
    // about two level-1 CTAs per SM over the requests; every slice keeps at least one beam
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
    cudaError_t e = launch_dependent(row_select_kernel, dim3(static_cast<unsigned>(rows)), dim3(kSelThreads), 0,
                                     stream, logits, V, W, cand_val, cand_tok, row_lse);
    if (e != cudaSuccess) return e;
    e = launch_dependent(merge_part_kernel, dim3(static_cast<unsigned>(static_cast<int64_t>(R) * S)),
                         dim3(kSelThreads), 0, stream, static_cast<const float *>(cand_val),
                         static_cast<const float *>(row_lse), cum, W, S, part_key, part_idx);
    if (e != cudaSuccess) return e;
    return launch_dependent(merge_final_kernel, dim3(static_cast<unsigned>(R)), dim3(kSelThreads), 0, stream,
                            static_cast<const uint32_t *>(part_key), static_cast<const int32_t *>(part_idx),
                            static_cast<const int32_t *>(cand_tok), W, S, token_out, parent_out, score_out);
}

}  // namespace bg
