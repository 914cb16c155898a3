// reorder.cu -- per-beam suffix K/V reorder by the beam parent index.
//
// "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", section 1.1: after each
// decode step beam selection keeps W candidates and names each one's parent;
// section 1.2: every beam keeps its own short suffix K/V.  The surviving beam
// b therefore continues from its parent's suffix: slots [0, n) of beam b in
// the destination buffer are a copy of slots [0, n) of beam parent[b] in the
// source buffer, and slot n receives the new token's K/V of beam b.
//
// Pure data movement of bf16 bit patterns (bit-exact).  One warp per beam;
// each beam's slots [0, n] are contiguous (n+1) * Hkv * head_dim bf16, so a
// warp moves them with coalesced 16-byte loads and stores, all of a batch's
// loads issued before its stores.  HBM-bound: it
// reads and writes 2 * n * Hkv * head_dim * 2 bytes per beam (+ the append).
#include "bg_internal.h"
#include "bg_ptx.cuh"

namespace bg {

namespace {
constexpr int kWarpsPerBlock = 8;
constexpr int kBatch = 4;           // vectors of K and of V in flight per lane

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    reorder_kernel(const uint4 *__restrict__ src_k, const uint4 *__restrict__ src_v, uint4 *__restrict__ dst_k,
                   uint4 *__restrict__ dst_v, const int32_t *__restrict__ parent, const uint4 *__restrict__ new_k,
                   const uint4 *__restrict__ new_v, int32_t R, int32_t W, int32_t suffix_max, int32_t n,
                   int32_t vec_per_tok, int32_t *dev_status)
{
    grid_dep_launch();
    grid_dep_wait();     // the previous kernel of the stream has completed
    const int64_t beam = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (beam >= static_cast<int64_t>(R) * W) return;
    const int64_t r = beam / W;
    const int32_t par = parent[beam];
    if (par < 0 || par >= W) {
        if (lane == 0 && dev_status) atomicOr(dev_status, BG_DEVSTAT_PARENT);
        return;
    }
    const int64_t slab = static_cast<int64_t>(suffix_max) * vec_per_tok;     // vectors per beam
    const uint4 *sk = src_k + (r * W + par) * slab;
    const uint4 *sv = src_v + (r * W + par) * slab;
    const uint4 *nk = new_k ? new_k + beam * vec_per_tok : nullptr;
    const uint4 *nv = new_v ? new_v + beam * vec_per_tok : nullptr;
    uint4 *dk = dst_k + beam * slab;
    uint4 *dv = dst_v + beam * slab;
    // slots [0, n) from the parent, then slot n from the new token: one contiguous run of dst.
    // Up to kBatch vectors of K and of V per lane are loaded before any is stored, so the warp
    // waits for memory about once per batch instead of once per vector.
    const int moved = n * vec_per_tok;
    const int total = moved + (nk ? vec_per_tok : 0);
    for (int base = 0; base < total; base += 32 * kBatch) {
        uint4 a[kBatch], b[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int i = base + lane + 32 * k;
            if (i < moved) {
                a[k] = sk[i];
                b[k] = sv[i];
            } else if (i < total) {
                a[k] = nk[i - moved];
                b[k] = nv[i - moved];
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int i = base + lane + 32 * k;
            if (i < total) {
                dk[i] = a[k];
                dv[i] = b[k];
            }
        }
    }
}
}  // namespace

cudaError_t launch_suffix_reorder(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                                  const int32_t *parent_idx, const void *new_k, const void *new_v, int32_t R,
                                  int32_t W, int32_t suffix_max, int32_t n_tokens, int32_t Hkv, int32_t head_dim,
                                  int32_t *dev_status, cudaStream_t stream)
{
    const int64_t beams = static_cast<int64_t>(R) * W;
    if (beams == 0) return cudaSuccess;
    const int32_t vec_per_tok = Hkv * head_dim * 2 / 16;
    const int64_t blocks = (beams + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_dependent(reorder_kernel, dim3(static_cast<unsigned>(blocks)), dim3(32 * kWarpsPerBlock), 0, stream,
                            static_cast<const uint4 *>(src_k), static_cast<const uint4 *>(src_v),
                            static_cast<uint4 *>(dst_k), static_cast<uint4 *>(dst_v), parent_idx,
                            static_cast<const uint4 *>(new_k), static_cast<const uint4 *>(new_v), R, W, suffix_max,
                            n_tokens, vec_per_tok, dev_status);
}

}  // namespace bg
