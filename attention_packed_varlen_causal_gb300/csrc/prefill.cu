// prefill.cu -- packed variable-length causal GQA prefill attention.
//
// "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", abstract (Packed
// Prefill) and section 1.2: each sequence keeps its valid length and only its
// valid tokens are computed, so no work depends on the longest sequence.
//
// Two launches on the caller's stream:
//   1. worklist_kernel (one CTA): checks cu_seqlens on the device and writes
//      the list of (sequence start, length, query tile) entries, sequences with more tiles
//      first and, within a sequence, later (costlier) query tiles first.
//      Only tiles of valid tokens exist: a sequence of length L has
//      ceil(L/128) query tiles and tile t streams key tiles 0..t.
//   2. attn_kernel<Prefill>: persistent CTAs walk the list round-robin.
#include "bg_attn_kernel.cuh"
#include "bg_internal.h"

#include <atomic>

namespace bg {

__global__ void __launch_bounds__(1024) worklist_kernel(const int32_t *__restrict__ cu, int32_t B, int32_t T,
                                                        int32_t max_seqlen, int32_t *__restrict__ hdr,
                                                        int4 *__restrict__ work, int32_t *dev_status)
{
    __shared__ int s_err;
    __shared__ int s_count[kMaxTilesPerSeq + 1];   // sequences per tile count
    __shared__ int s_off[kMaxTilesPerSeq + 2];     // first entry of each tile-count bucket
    const int tid = threadIdx.x;
    grid_dep_launch();
    if (tid == 0) s_err = 0;
    for (int i = tid; i <= kMaxTilesPerSeq; i += blockDim.x) s_count[i] = 0;
    grid_dep_wait();
    __syncthreads();

    int err = 0;
    if (B > 0 && tid == 0 && cu[0] != 0) err |= BG_DEVSTAT_CU_SEQLENS;
    for (int i = tid; i < B; i += blockDim.x) {
        const int a = cu[i], b = cu[i + 1];
        if (b < a || a < 0 || b > T) {
            err |= BG_DEVSTAT_CU_SEQLENS;
            continue;
        }
        if (i == B - 1 && b != T) err |= BG_DEVSTAT_CU_SEQLENS;
        if (b - a > max_seqlen) {
            err |= BG_DEVSTAT_SEQ_TOO_LONG;
            continue;
        }
        const int nt = (b - a + kPrefillTileRows - 1) / kPrefillTileRows;
        if (nt > 0) atomicAdd(&s_count[nt], 1);
    }
    if (err) atomicOr(&s_err, err);
    __syncthreads();
    if (s_err) {
        if (tid == 0) {
            hdr[0] = s_err;
            hdr[1] = 0;
            if (dev_status) atomicOr(dev_status, s_err);
        }
        return;
    }
    if (tid == 0) {
        // buckets in decreasing tile count; a sequence with nt tiles owns nt entries
        const int max_nt = (max_seqlen + kPrefillTileRows - 1) / kPrefillTileRows;
        int off = 0;
        for (int nt = max_nt; nt >= 1; --nt) {
            s_off[nt] = off;
            off += s_count[nt] * nt;
        }
        hdr[1] = off;
        hdr[3] = T;      // the packing the list belongs to, checked by every run that reads it
        hdr[4] = B;
        hdr[0] = 0;
    }
    __syncthreads();
    for (int i = tid; i < B; i += blockDim.x) {
        const int L = cu[i + 1] - cu[i];
        const int nt = (L + kPrefillTileRows - 1) / kPrefillTileRows;
        if (nt == 0) continue;
        const int pos = atomicAdd(&s_off[nt], nt);
        // complete item descriptors (start, length, query tile), so readers need one load
        for (int t = 0; t < nt; ++t) work[pos + t] = make_int4(cu[i], L, nt - 1 - t, i);
    }
}

cudaError_t launch_prefill_worklist(const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                    int32_t max_seqlen, int32_t *work_hdr, int4 *work, int32_t *dev_status,
                                    cudaStream_t stream)
{
    return launch_dependent(worklist_kernel, dim3(1), dim3(1024), 0, stream, cu_seqlens, num_seqs, total_tokens,
                            max_seqlen, work_hdr, work, dev_status);
}

namespace {
constexpr int kNH = 2;   // query heads of one kv head per CTA (share every K/V tile)

template <int D, int NK, int NV, int NS, bool QK8>
std::atomic<uint64_t> &smem_attr_done()
{
    static std::atomic<uint64_t> mask{0};
    return mask;
}

template <int D, int NK, int NV, int NS, bool QK8 = false>
cudaError_t launch_one(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                       const CUtensorMap &tm_o, const AttnParams &p, int grid, cudaStream_t stream)
{
    using C = AttnCfg<D, kNH, NK, NV, NS, QK8>;
    auto kern = attn_kernel<Mode::Prefill, D, kNH, NK, NV, NS, QK8>;
    cudaError_t e = ensure_smem_attribute(kern, C::kSmemBytes, smem_attr_done<D, NK, NV, NS, QK8>());
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> split_checked{0};
    e = check_register_split(kern, C::kThreads, C::kSplitRegs, split_checked);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, tm_q, tm_k, tm_v, tm_k, tm_v,
                            tm_o, p);   // no suffix maps
}
}  // namespace

int prefill_heads_per_cta() { return kNH; }

cudaError_t launch_prefill_attn(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                const CUtensorMap &tm_v, const CUtensorMap &tm_o, const AttnParams &p, int grid,
                                cudaStream_t stream)
{
    if (head_dim == 128) return launch_one<128, 2, 3, 2>(tm_q, tm_k, tm_v, tm_o, p, grid, stream);
    if (head_dim == 64) return launch_one<64, 4, 4, 3>(tm_q, tm_k, tm_v, tm_o, p, grid, stream);
    return cudaErrorInvalidValue;
}

// E4M3 Q and K (one 8 KB K stage and one 16 KB Q tile per 128-byte row block), bf16 V: the
// smaller K stages leave room for six K and four V stages (192 KB; measured against four K
// stages: 186.7 vs 191.0 us per Prefill-Only layer).
cudaError_t launch_prefill_attn_fp8(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                    const CUtensorMap &tm_v, const CUtensorMap &tm_o, const AttnParams &p, int grid,
                                    cudaStream_t stream)
{
    if (head_dim == 128) return launch_one<128, 6, 4, 2, true>(tm_q, tm_k, tm_v, tm_o, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bg
