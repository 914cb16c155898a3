// decode.cu -- beam-search decode attention over a shared prompt K/V.
//
// "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", section 1.2: the beams
// of one request share a single prompt K/V and each beam keeps its own short
// suffix K/V.  The shared prompt is what makes the decode step dense: the
// queries of all beams x group heads of one kv head form 128-row tiles that
// run on the tensor cores against the prompt K/V, read once per tile pair
// (and from L2 for the sibling tiles).  The few suffix keys of each beam
// follow as extra key tiles of the same item (see attn_kernel<Decode>).
#include "bg_attn_kernel.cuh"
#include "bg_internal.h"

#include <atomic>

namespace bg {

namespace {
constexpr int kNH = 2;   // query tiles (of the same request and kv head) per CTA

template <int D, int NK, int NV, int NS>
std::atomic<uint64_t> &smem_attr_done()
{
    static std::atomic<uint64_t> mask{0};
    return mask;
}

template <int D, int NK, int NV, int NS>
cudaError_t launch_one(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                       const CUtensorMap &tm_sk, const CUtensorMap &tm_sv, const CUtensorMap &tm_o,
                       const AttnParams &p, int grid, cudaStream_t stream)
{
    using C = AttnCfg<D, kNH, NK, NV, NS>;
    auto kern = attn_kernel<Mode::Decode, D, kNH, NK, NV, NS>;
    cudaError_t e = ensure_smem_attribute(kern, C::kSmemBytes, smem_attr_done<D, NK, NV, NS>());
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> split_checked{0};
    e = check_register_split(kern, C::kThreads, C::kSplitRegs, split_checked);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, tm_q, tm_k, tm_v, tm_sk,
                            tm_sv, tm_o, p);
}
}  // namespace

int decode_tiles_per_cta() { return kNH; }

cudaError_t launch_decode_attn(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const CUtensorMap &tm_sk, const CUtensorMap &tm_sv,
                               const CUtensorMap &tm_o, const AttnParams &p, int grid, cudaStream_t stream)
{
    if (head_dim == 64) return launch_one<64, 6, 6, 3>(tm_q, tm_k, tm_v, tm_sk, tm_sv, tm_o, p, grid, stream);
    if (head_dim == 128) return launch_one<128, 3, 2, 2>(tm_q, tm_k, tm_v, tm_sk, tm_sv, tm_o, p, grid, stream);
    return cudaErrorInvalidValue;
}



}  // namespace bg
