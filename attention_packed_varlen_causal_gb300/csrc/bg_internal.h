// bg_internal.h -- launchers shared between the C-ABI layer and the kernel
// translation units (not part of the public interface).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "bg_attn.h"

namespace bg {

struct AttnParams;

// Host checks of bg_packed_prefill_attn's arguments other than the workspace (sizes, shape
// support, scale, pointers, alignment, aliasing between the tensors; Q and K elements of
// `qk_elem_bytes` bytes, V and the output bf16).  Returns BG_OK or the
// status the entry point returns; *noop is set when the call is a valid no-op.
bg_status_t prefill_check_args(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                               int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                               int32_t Hkv, int32_t head_dim, float scale, const void *out, const float *lse,
                               const int32_t *dev_status, bool *noop, int qk_elem_bytes = 2);

// Prefill: work-list pre-pass + attention kernel.  Maps are built by the
// caller.  Returns cudaSuccess or the launch error.
cudaError_t launch_prefill_worklist(const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                    int32_t max_seqlen, int32_t *work_hdr, int4 *work, int32_t *dev_status,
                                    cudaStream_t stream);
cudaError_t launch_prefill_attn(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                const CUtensorMap &tm_v, const CUtensorMap &tm_o, const AttnParams &p, int grid,
                                cudaStream_t stream);
cudaError_t launch_prefill_attn_fp8(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                    const CUtensorMap &tm_v, const CUtensorMap &tm_o, const AttnParams &p, int grid,
                                    cudaStream_t stream);
int prefill_heads_per_cta();

cudaError_t launch_decode_attn(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const CUtensorMap &tm_sk, const CUtensorMap &tm_sv,
                               const CUtensorMap &tm_o, const AttnParams &p, int grid, cudaStream_t stream);
int decode_tiles_per_cta();

// Attention of each sequence's last valid token (one CTA per sequence and kv head).
cudaError_t launch_last_token_attn(int head_dim, const void *q, const void *k, const void *v, const int32_t *cu,
                                   int32_t B, int32_t T, int32_t max_seqlen, int32_t Hq, int32_t Hkv, float scale,
                                   void *out, float *lse, int32_t *dev_status, cudaStream_t stream);
int last_token_max_group();

// Beam candidate selection: per-beam selection into (cand_val, cand_tok, row_lse), the
// merge's level 1 into (part_key, part_idx) of R * S * W entries, level 2 into the outputs.
int beam_select_slices(int32_t R, int32_t W);
cudaError_t launch_beam_select(const float *logits, const float *cum, int32_t R, int32_t W, int32_t V,
                               int32_t *token_out, int32_t *parent_out, float *score_out, float *cand_val,
                               int32_t *cand_tok, float *row_lse, uint32_t *part_key, int32_t *part_idx,
                               cudaStream_t stream);

cudaError_t launch_suffix_reorder(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                                  const int32_t *parent_idx, const void *new_k, const void *new_v, int32_t R,
                                  int32_t W, int32_t suffix_max, int32_t n_tokens, int32_t Hkv, int32_t head_dim,
                                  int32_t *dev_status, cudaStream_t stream);

// Diagnostic: one kernel whose only wait (bg::mbar_wait on an mbarrier nothing arrives on)
// runs out; it ORs BG_DEVSTAT_TIMEOUT into *dev_status and writes the time it waited.
cudaError_t launch_wait_timeout_selftest(int32_t *dev_status, unsigned long long *waited_ns, cudaStream_t stream);

// Launches `kern` on `stream` with programmatic stream serialization: its CTAs may
// start while the previous kernel of the stream still runs (that kernel lets them
// with griddepcontrol.launch_dependents); every kernel of this library waits
// (griddepcontrol.wait) before its first global-memory access, so only prologue
// work overlaps.  Valid inside CUDA-graph stream capture.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raises the dynamic shared-memory limit of `kern` once per device (bit d of
// `done`), so later launches -- including ones inside a CUDA-graph capture --
// make no attribute call.
template <typename Kern>
cudaError_t ensure_smem_attribute(Kern kern, int bytes, std::atomic<uint64_t> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// The attention kernels split the registers of their launch between warp roles (setmaxnreg),
// and a split larger than the launch's allocation would wait forever.  Before launching, the
// compiled kernel's registers per thread (looked up once per device) times its threads must
// cover the split; otherwise the launch is refused (cudaErrorInvalidConfiguration).
template <typename Kern>
cudaError_t check_register_split(Kern kern, int threads, int split_regs, std::atomic<uint64_t> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    cudaFuncAttributes a{};
    e = cudaFuncGetAttributes(&a, kern);
    if (e != cudaSuccess) return e;
    if (a.numRegs * threads < split_regs) return cudaErrorInvalidConfiguration;
    if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

// Work-list layout inside the caller's workspace.
constexpr size_t kWorkHeaderBytes = 256;
constexpr int kPrefillTileRows = 128;
constexpr int kMaxTilesPerSeq = BG_MAX_SEQLEN / kPrefillTileRows;

}  // namespace bg
