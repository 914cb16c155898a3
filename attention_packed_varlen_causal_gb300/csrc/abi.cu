// abi.cu -- the C ABI (include/bg_attn.h): host-side argument checks, TMA
// tensor-map encoding and kernel launches.  No allocation, no stream
// synchronisation; every call only enqueues work on the caller's stream.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bg_attn.h"
#include "bg_attn_kernel.cuh"
#include "bg_internal.h"

using namespace bg;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) return cached;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Tiled map (bf16 unless `type` says otherwise), 128-byte swizzle, box inner extent 128 bytes.
bool encode_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint64_t *strides_bytes,
                const uint32_t *box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    auto fn = encoder();
    if (!fn) return false;
    cuuint64_t gdim[5], gstr[4];
    cuuint32_t bdim[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gstr[i] = strides_bytes[i];
    std::memset(m, 0, sizeof(*m));
    const CUresult r = fn(m, type, static_cast<cuuint32_t>(rank), const_cast<void *>(base),
                          gdim, gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool supported_head_dim(int32_t d) { return d == 64 || d == 128; }

size_t prefill_entries_bound(int64_t num_seqs, int64_t total_tokens)
{
    return static_cast<size_t>(total_tokens / kPrefillTileRows + num_seqs + 1);
}

}  // namespace

extern "C" {

const char *bg_status_string(bg_status_t s)
{
    switch (s) {
    case BG_OK: return "BG_OK";
    case BG_ERR_INVALID_ARG: return "BG_ERR_INVALID_ARG";
    case BG_ERR_UNSUPPORTED: return "BG_ERR_UNSUPPORTED";
    case BG_ERR_DEVICE_DATA: return "BG_ERR_DEVICE_DATA";
    case BG_ERR_CUDA: return "BG_ERR_CUDA";
    }
    return "BG_ERR_UNKNOWN";
}

size_t bg_packed_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                        int32_t Hkv, int32_t head_dim)
{
    (void)max_seqlen;
    (void)Hq;
    (void)Hkv;
    (void)head_dim;
    if (num_seqs < 0 || total_tokens < 0) return 0;
    const size_t bytes = kWorkHeaderBytes + sizeof(int4) * prefill_entries_bound(num_seqs, total_tokens);
    return (bytes + 255) & ~size_t(255);
}

}  // extern "C"

bg_status_t bg::prefill_check_args(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                   int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                   int32_t Hkv, int32_t head_dim, float scale, const void *out, const float *lse,
                                   const int32_t *dev_status, bool *noop, int qk_elem_bytes)
{
    *noop = false;
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0)
        return BG_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return BG_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return BG_ERR_INVALID_ARG;   // masked logits are -inf
    if (!supported_head_dim(head_dim) || max_seqlen > BG_MAX_SEQLEN) return BG_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_tokens == 0) {
        *noop = true;
        return BG_OK;
    }
    if (!q || !k || !v || !cu_seqlens || !out) return BG_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_seqlens, 4) ||
        (lse && !aligned(lse, 4)) || (dev_status && !aligned(dev_status, 4)))
        return BG_ERR_INVALID_ARG;
    const size_t obytes = static_cast<size_t>(total_tokens) * Hq * head_dim * 2;
    const size_t qbytes = static_cast<size_t>(total_tokens) * Hq * head_dim * qk_elem_bytes;
    const size_t kbytes = static_cast<size_t>(total_tokens) * Hkv * head_dim * qk_elem_bytes;
    const size_t vbytes = static_cast<size_t>(total_tokens) * Hkv * head_dim * 2;
    const size_t lsebytes = lse ? static_cast<size_t>(total_tokens) * Hq * 4 : 0;
    if (overlap(out, obytes, q, qbytes) || overlap(out, obytes, k, kbytes) || overlap(out, obytes, v, vbytes) ||
        overlap(lse, lsebytes, out, obytes) || overlap(lse, lsebytes, q, qbytes) ||
        overlap(lse, lsebytes, k, kbytes) || overlap(lse, lsebytes, v, vbytes))
        return BG_ERR_INVALID_ARG;
    return BG_OK;
}

namespace {

// bg_packed_prefill_attn (qk8 false: bf16 Q/K) and bg_packed_prefill_attn_fp8 (qk8 true: E4M3
// Q/K codes, whose two per-tensor scales the caller has already folded into `scale`).
// with_plan: launch the work-list pre-pass first; otherwise the workspace holds a plan from
// bg_packed_prefill_plan for the same cu_seqlens (bg_packed_prefill_attn_planned).
bg_status_t prefill_impl(const void *q, const void *k, const void *v, const int32_t *cu_seqlens, int32_t num_seqs,
                         int32_t total_tokens, int32_t max_seqlen, int32_t Hq, int32_t Hkv, int32_t head_dim,
                         float scale, void *out, float *lse, void *workspace, size_t workspace_bytes,
                         int32_t *dev_status, cudaStream_t stream, bool qk8, bool with_plan = true)
{
    bool noop = false;
    const bg_status_t chk = prefill_check_args(q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv,
                                               head_dim, scale, out, lse, dev_status, &noop, qk8 ? 1 : 2);
    if (chk != BG_OK || noop) return chk;
    if (qk8 && head_dim != 128) return BG_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256)) return BG_ERR_INVALID_ARG;
    if (workspace_bytes < bg_packed_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim))
        return BG_ERR_INVALID_ARG;
    const size_t qbytes = static_cast<size_t>(total_tokens) * Hq * head_dim * 2;
    const size_t lsebytes = lse ? static_cast<size_t>(total_tokens) * Hq * 4 : 0;
    if (overlap(out, qbytes, workspace, workspace_bytes) || overlap(lse, lsebytes, workspace, workspace_bytes))
        return BG_ERR_INVALID_ARG;

    const int32_t g = Hq / Hkv;
    const int nh = prefill_heads_per_cta();
    const int32_t groups_per_kv = (g + nh - 1) / nh;
    const int64_t items_bound = static_cast<int64_t>(prefill_entries_bound(num_seqs, total_tokens)) * Hkv * groups_per_kv;
    if (items_bound >= (int64_t(1) << 31)) return BG_ERR_UNSUPPORTED;

    const int nsm = sm_count();
    if (nsm <= 0) return BG_ERR_CUDA;

    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    const uint64_t D = static_cast<uint64_t>(head_dim);
    const uint64_t E = qk8 ? 1 : 2;    // bytes per Q/K element
    const uint64_t dq[3] = {D, static_cast<uint64_t>(Hq), static_cast<uint64_t>(total_tokens)};
    const uint64_t sq[2] = {D * 2, static_cast<uint64_t>(Hq) * D * 2};
    const uint64_t sq8[2] = {D * E, static_cast<uint64_t>(Hq) * D * E};
    const uint64_t dkv[3] = {D, static_cast<uint64_t>(Hkv), static_cast<uint64_t>(total_tokens)};
    const uint64_t skv[2] = {D * 2, static_cast<uint64_t>(Hkv) * D * 2};
    const uint64_t sk8[2] = {D * E, static_cast<uint64_t>(Hkv) * D * E};
    // boxes: one 128-byte swizzle span of columns (64 bf16 or 128 E4M3 codes) x one head x the
    // kernel's tile height
    const uint32_t qk_cols = static_cast<uint32_t>(128 / E);
    const uint32_t boxq[3] = {64, 1, static_cast<uint32_t>(bg::kRows)};
    const uint32_t boxkv[3] = {64, 1, static_cast<uint32_t>(bg::kKeys)};
    const uint32_t boxq8[3] = {qk_cols, 1, static_cast<uint32_t>(bg::kRows)};
    const uint32_t boxk8[3] = {qk_cols, 1, static_cast<uint32_t>(bg::kKeys)};
    const CUtensorMapDataType qk_type = qk8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // the output has the (bf16) query's shape: whole 128-row tiles leave through the same box
    if (!encode_map(&tm_q, q, 3, dq, sq8, boxq8, qk_type) || !encode_map(&tm_k, k, 3, dkv, sk8, boxk8, qk_type) ||
        !encode_map(&tm_v, v, 3, dkv, skv, boxkv) || !encode_map(&tm_o, out, 3, dq, sq, boxq))
        return BG_ERR_CUDA;

    int32_t *hdr = static_cast<int32_t *>(workspace);
    int4 *work = reinterpret_cast<int4 *>(static_cast<uint8_t *>(workspace) + kWorkHeaderBytes);
    if (with_plan &&
        launch_prefill_worklist(cu_seqlens, num_seqs, total_tokens, max_seqlen, hdr, work, dev_status, stream) !=
            cudaSuccess)
        return BG_ERR_CUDA;

    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = g;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.dev_status = dev_status;
    p.err_word = hdr + 2;
    p.cu_seqlens = cu_seqlens;
    p.work = work;
    p.work_hdr = hdr;
    p.groups_per_kv = groups_per_kv;
    p.n_head_groups = Hkv * groups_per_kv;
    p.lse = lse;
    p.total_prompt = total_tokens;   // the packing this call expects the work list to be for
    p.R = num_seqs;
    const int grid = static_cast<int>(items_bound < nsm ? items_bound : nsm);
    const cudaError_t e = qk8 ? launch_prefill_attn_fp8(head_dim, tm_q, tm_k, tm_v, tm_o, p, grid, stream)
                              : launch_prefill_attn(head_dim, tm_q, tm_k, tm_v, tm_o, p, grid, stream);
    return e == cudaSuccess ? BG_OK : BG_ERR_CUDA;
}

}  // namespace

extern "C" {

bg_status_t bg_packed_prefill_attn(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                   int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                   int32_t Hkv, int32_t head_dim, float scale, void *out, float *lse, void *workspace,
                                   size_t workspace_bytes, int32_t *dev_status, cudaStream_t stream)
{
    return prefill_impl(q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim, scale, out, lse,
                        workspace, workspace_bytes, dev_status, stream, false);
}

bg_status_t bg_packed_prefill_plan(const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                   int32_t max_seqlen, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                   cudaStream_t stream)
{
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return BG_ERR_INVALID_ARG;
    if (max_seqlen > BG_MAX_SEQLEN) return BG_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_tokens == 0) return BG_OK;   // the planned run is a no-op as well
    if (!cu_seqlens || !aligned(cu_seqlens, 4) || (dev_status && !aligned(dev_status, 4))) return BG_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return BG_ERR_INVALID_ARG;
    if (workspace_bytes < bg_packed_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, 1, 1, 64))
        return BG_ERR_INVALID_ARG;
    if (overlap(cu_seqlens, (static_cast<size_t>(num_seqs) + 1) * 4, workspace, workspace_bytes))
        return BG_ERR_INVALID_ARG;
    int32_t *hdr = static_cast<int32_t *>(workspace);
    int4 *work = reinterpret_cast<int4 *>(static_cast<uint8_t *>(workspace) + kWorkHeaderBytes);
    return launch_prefill_worklist(cu_seqlens, num_seqs, total_tokens, max_seqlen, hdr, work, dev_status, stream) ==
                   cudaSuccess
               ? BG_OK
               : BG_ERR_CUDA;
}

bg_status_t bg_packed_prefill_attn_planned(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                           int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                           int32_t Hkv, int32_t head_dim, float scale, void *out, float *lse,
                                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                           cudaStream_t stream)
{
    return prefill_impl(q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim, scale, out, lse,
                        workspace, workspace_bytes, dev_status, stream, false, false);
}

bg_status_t bg_packed_prefill_attn_fp8(const void *q_codes, float q_scale, const void *k_codes, float k_scale,
                                       const void *v, const int32_t *cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t max_seqlen, int32_t Hq, int32_t Hkv,
                                       int32_t head_dim, float scale, void *out, float *lse, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status, cudaStream_t stream)
{
    if (!std::isfinite(q_scale) || !(q_scale > 0.f) || !std::isfinite(k_scale) || !(k_scale > 0.f))
        return BG_ERR_INVALID_ARG;
    // q . k over the dequantised values = (q_scale * k_scale) * (codes . codes): the tensor
    // cores multiply the codes, the two scales join the softmax scale
    const double s = static_cast<double>(scale) * q_scale * k_scale;
    if (!(s > 0.0) || s > 3.0e38) return BG_ERR_INVALID_ARG;
    return prefill_impl(q_codes, k_codes, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim,
                        static_cast<float>(s), out, lse, workspace, workspace_bytes, dev_status, stream, true);
}

bg_status_t bg_packed_last_token_attn(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                      int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                      int32_t Hkv, int32_t head_dim, float scale, void *out, float *lse,
                                      int32_t *dev_status, cudaStream_t stream)
{
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0)
        return BG_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return BG_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return BG_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || max_seqlen > BG_MAX_SEQLEN || Hq / Hkv > last_token_max_group())
        return BG_ERR_UNSUPPORTED;
    if (num_seqs == 0) return BG_OK;
    if (!q || !k || !v || !cu_seqlens || !out) return BG_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_seqlens, 4) ||
        (lse && !aligned(lse, 4)) || (dev_status && !aligned(dev_status, 4)))
        return BG_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_seqs) * Hkv >= (int64_t(1) << 31)) return BG_ERR_UNSUPPORTED;
    const size_t obytes = static_cast<size_t>(num_seqs) * Hq * head_dim * 2;
    const size_t kvbytes = static_cast<size_t>(total_tokens) * Hkv * head_dim * 2;
    const size_t lsebytes = lse ? static_cast<size_t>(num_seqs) * Hq * 4 : 0;
    if (overlap(out, obytes, q, obytes) || overlap(out, obytes, k, kvbytes) || overlap(out, obytes, v, kvbytes) ||
        overlap(lse, lsebytes, out, obytes) || overlap(lse, lsebytes, q, obytes) || overlap(lse, lsebytes, k, kvbytes) ||
        overlap(lse, lsebytes, v, kvbytes))
        return BG_ERR_INVALID_ARG;
    if (launch_last_token_attn(head_dim, q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv, scale, out,
                               lse, dev_status, stream) != cudaSuccess)
        return BG_ERR_CUDA;
    return BG_OK;
}

}  // extern "C"

namespace {

// Extra operands of a whole decode step (bg_beam_decode_step): the previous step's suffix, the
// parent index and the new token's K/V.  Null for the plain decode attention.
struct StepFuse {
    const void *src_k, *src_v;
    const int32_t *parent;
    const void *new_k, *new_v;
};

// Decode work items: (request, kv head, nh query tiles of BT = 128 / g beams each).
int32_t decode_pairs_per_rk(int32_t W, int32_t g, int nh)
{
    const int32_t BT = 128 / g;
    const int32_t beam_tiles = (W + BT - 1) / BT;
    return (beam_tiles + nh - 1) / nh;
}

bg_status_t decode_impl(const void *q, const void *prompt_k, const void *prompt_v, const int32_t *cu_prompt,
                        int32_t total_prompt_tokens, int32_t max_prompt_len, const void *suffix_k, const void *suffix_v,
                        int32_t suffix_len, int32_t suffix_max, int32_t R, int32_t W, int32_t Hq, int32_t Hkv,
                        int32_t head_dim, float scale, void *out, int32_t *dev_status, const StepFuse *fz,
                        cudaStream_t stream)
{
    if (R < 0 || W <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || total_prompt_tokens < 0 || max_prompt_len < 0 ||
        suffix_len < 0 || suffix_max < 0 || suffix_len > suffix_max)
        return BG_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !std::isfinite(scale) || !(scale > 0.f)) return BG_ERR_INVALID_ARG;
    const int32_t g = Hq / Hkv;
    if (!supported_head_dim(head_dim) || g > 128 || suffix_max > BG_MAX_SUFFIX) return BG_ERR_UNSUPPORTED;
    if (max_prompt_len == 0 && suffix_len == 0) return BG_ERR_INVALID_ARG;   // every softmax would be empty
    if (R == 0) return BG_OK;
    if (static_cast<int64_t>(R) * W >= (int64_t(1) << 31)) return BG_ERR_UNSUPPORTED;
    if (!q || !out || !cu_prompt) return BG_ERR_INVALID_ARG;
    if (total_prompt_tokens > 0 && (!prompt_k || !prompt_v)) return BG_ERR_INVALID_ARG;
    if (suffix_len > 0 && (!suffix_k || !suffix_v)) return BG_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(cu_prompt, 4) || (prompt_k && !aligned(prompt_k, 16)) ||
        (prompt_v && !aligned(prompt_v, 16)) || (suffix_k && !aligned(suffix_k, 16)) ||
        (suffix_v && !aligned(suffix_v, 16)) || (dev_status && !aligned(dev_status, 4)))
        return BG_ERR_INVALID_ARG;
    const size_t qbytes = static_cast<size_t>(R) * W * Hq * head_dim * 2;
    const size_t pbytes = static_cast<size_t>(total_prompt_tokens) * Hkv * head_dim * 2;
    const size_t sbytes = static_cast<size_t>(R) * W * suffix_max * Hkv * head_dim * 2;
    if (overlap(out, qbytes, q, qbytes) || overlap(out, qbytes, prompt_k, pbytes) ||
        overlap(out, qbytes, prompt_v, pbytes) || (suffix_len > 0 && (overlap(out, qbytes, suffix_k, sbytes) ||
                                                                      overlap(out, qbytes, suffix_v, sbytes))))
        return BG_ERR_INVALID_ARG;

    if (fz) {
        // whole step: suffix_k/v receive this step's suffix from the reorder kernel before the
        // attention kernel reads them, so no input may share their bytes
        if (suffix_len < 1 || !fz->parent || !fz->new_k || !fz->new_v) return BG_ERR_INVALID_ARG;
        if (suffix_len > 1 && (!fz->src_k || !fz->src_v)) return BG_ERR_INVALID_ARG;
        if (!aligned(fz->parent, 4) || !aligned(fz->new_k, 16) || !aligned(fz->new_v, 16) ||
            (fz->src_k && !aligned(fz->src_k, 16)) || (fz->src_v && !aligned(fz->src_v, 16)))
            return BG_ERR_INVALID_ARG;
        const size_t nbytes = static_cast<size_t>(R) * W * Hkv * head_dim * 2;
        const size_t srcbytes = suffix_len > 1 ? sbytes : 0;
        const void *rd[9] = {q, prompt_k, prompt_v, cu_prompt, fz->parent, fz->new_k, fz->new_v, fz->src_k, fz->src_v};
        const size_t rdn[9] = {qbytes, pbytes, pbytes, static_cast<size_t>(R + 1) * 4, static_cast<size_t>(R) * W * 4,
                               nbytes, nbytes, srcbytes, srcbytes};
        for (int i = 0; i < 9; ++i)
            if (overlap(suffix_k, sbytes, rd[i], rdn[i]) || overlap(suffix_v, sbytes, rd[i], rdn[i]) ||
                (i >= 4 && overlap(out, qbytes, rd[i], rdn[i])))
                return BG_ERR_INVALID_ARG;
        if (overlap(suffix_k, sbytes, suffix_v, sbytes)) return BG_ERR_INVALID_ARG;
    }

    const int nsm = sm_count();
    if (nsm <= 0) return BG_ERR_CUDA;

    const int nh = decode_tiles_per_cta();
    const int32_t BT = 128 / g;
    const int32_t pairs = decode_pairs_per_rk(W, g, nh);
    const int64_t items = static_cast<int64_t>(R) * Hkv * pairs;
    if (items >= (int64_t(1) << 31)) return BG_ERR_UNSUPPORTED;

    CUtensorMap tm_q, tm_k, tm_v, tm_sk, tm_sv, tm_o;
    const uint64_t D = static_cast<uint64_t>(head_dim);
    const uint64_t dq[4] = {D, static_cast<uint64_t>(g), static_cast<uint64_t>(Hkv), static_cast<uint64_t>(R) * W};
    const uint64_t sq[3] = {D * 2, static_cast<uint64_t>(g) * D * 2, static_cast<uint64_t>(Hq) * D * 2};
    const uint32_t boxq[4] = {64, static_cast<uint32_t>(g), 1, static_cast<uint32_t>(BT)};
    const uint64_t np = total_prompt_tokens > 0 ? static_cast<uint64_t>(total_prompt_tokens) : 1;
    const uint64_t dkv[3] = {D, static_cast<uint64_t>(Hkv), np};
    const uint64_t skv[2] = {D * 2, static_cast<uint64_t>(Hkv) * D * 2};
    const uint32_t boxkv[3] = {64, 1, static_cast<uint32_t>(bg::kKeys)};
    // With no prompt tokens no K/V tile is ever loaded; the maps only need a valid base.
    const void *kbase = total_prompt_tokens > 0 ? prompt_k : q;
    const void *vbase = total_prompt_tokens > 0 ? prompt_v : q;
    // the output has the query's shape: whole tiles of BT beams leave through the same box
    if (!encode_map(&tm_q, q, 4, dq, sq, boxq) || !encode_map(&tm_k, kbase, 3, dkv, skv, boxkv) ||
        !encode_map(&tm_v, vbase, 3, dkv, skv, boxkv) || !encode_map(&tm_o, out, 4, dq, sq, boxq))
        return BG_ERR_CUDA;
    // Suffix key tiles: slots 0..t-1 of suf_bpt consecutive beams per tile (beam-major rows),
    // over [R*W beams][suffix_max slots][Hkv][d]; beams past R*W read as zeros.
    const int32_t t_suf = suffix_len > 0 ? suffix_len : 1;
    int32_t bpt = bg::kKeys / t_suf;
    if (bpt > nh * BT) bpt = nh * BT;
    const uint64_t ds[4] = {D, static_cast<uint64_t>(Hkv), static_cast<uint64_t>(suffix_max > 0 ? suffix_max : 1),
                            static_cast<uint64_t>(R) * W};
    const uint64_t ss[3] = {D * 2, static_cast<uint64_t>(Hkv) * D * 2,
                            static_cast<uint64_t>(suffix_max > 0 ? suffix_max : 1) * Hkv * D * 2};
    const uint32_t boxs[4] = {64, 1, static_cast<uint32_t>(t_suf), static_cast<uint32_t>(bpt)};
    const void *skbase = suffix_len > 0 ? suffix_k : q;
    const void *svbase = suffix_len > 0 ? suffix_v : q;
    if (!encode_map(&tm_sk, skbase, 4, ds, ss, boxs) || !encode_map(&tm_sv, svbase, 4, ds, ss, boxs))
        return BG_ERR_CUDA;

    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = g;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.dev_status = dev_status;
    p.err_word = nullptr;
    p.cu_prompt = cu_prompt;
    p.R = R;
    p.W = W;
    p.BT = BT;
    p.pairs_per_rk = pairs;
    p.max_prompt_len = max_prompt_len;
    p.total_prompt = total_prompt_tokens;
    p.suffix_len = suffix_len;
    p.suf_bpt = bpt;
    p.suf_tx = (head_dim / 64) * 128 * t_suf * bpt;
    p.n_items_decode = static_cast<int32_t>(items);
    const int grid = static_cast<int>(items < nsm ? items : nsm);
    if (fz) {
        // the step's reorder + append first (it moves nothing at t = 1 and then never reads src),
        // then the attention over the new suffix
        const void *sk = fz->src_k ? fz->src_k : suffix_k;
        const void *sv = fz->src_v ? fz->src_v : suffix_v;
        if (launch_suffix_reorder(sk, sv, const_cast<void *>(suffix_k), const_cast<void *>(suffix_v), fz->parent,
                                  fz->new_k, fz->new_v, R, W, suffix_max, suffix_len - 1, Hkv, head_dim, dev_status,
                                  stream) != cudaSuccess)
            return BG_ERR_CUDA;
    }
    if (launch_decode_attn(head_dim, tm_q, tm_k, tm_v, tm_sk, tm_sv, tm_o, p, grid, stream) != cudaSuccess)
        return BG_ERR_CUDA;
    return BG_OK;
}

}  // namespace

extern "C" {

bg_status_t bg_beam_decode_attn(const void *q, const void *prompt_k, const void *prompt_v, const int32_t *cu_prompt,
                                int32_t total_prompt_tokens, int32_t max_prompt_len, const void *suffix_k,
                                const void *suffix_v, int32_t suffix_len, int32_t suffix_max, int32_t R, int32_t W,
                                int32_t Hq, int32_t Hkv, int32_t head_dim, float scale, void *out,
                                int32_t *dev_status, cudaStream_t stream)
{
    return decode_impl(q, prompt_k, prompt_v, cu_prompt, total_prompt_tokens, max_prompt_len, suffix_k, suffix_v,
                       suffix_len, suffix_max, R, W, Hq, Hkv, head_dim, scale, out, dev_status, nullptr, stream);
}

bg_status_t bg_beam_decode_step(const void *q, const void *prompt_k, const void *prompt_v, const int32_t *cu_prompt,
                                int32_t total_prompt_tokens, int32_t max_prompt_len, const void *src_suffix_k,
                                const void *src_suffix_v, const int32_t *parent_idx, const void *new_k,
                                const void *new_v, void *dst_suffix_k, void *dst_suffix_v, int32_t suffix_len,
                                int32_t suffix_max, int32_t R, int32_t W, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                float scale, void *out, int32_t *dev_status, cudaStream_t stream)
{
    if (suffix_len < 1) return BG_ERR_INVALID_ARG;
    const StepFuse fz{src_suffix_k, src_suffix_v, parent_idx, new_k, new_v};
    return decode_impl(q, prompt_k, prompt_v, cu_prompt, total_prompt_tokens, max_prompt_len, dst_suffix_k,
                       dst_suffix_v, suffix_len, suffix_max, R, W, Hq, Hkv, head_dim, scale, out, dev_status, &fz,
                       stream);
}

bg_status_t bg_beam_suffix_reorder(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                                   const int32_t *parent_idx, const void *new_k, const void *new_v, int32_t R,
                                   int32_t W, int32_t suffix_max, int32_t n_tokens, int32_t Hkv, int32_t head_dim,
                                   int32_t *dev_status, cudaStream_t stream)
{
    if (R < 0 || W <= 0 || suffix_max <= 0 || n_tokens < 0 || Hkv <= 0 || head_dim <= 0) return BG_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return BG_ERR_UNSUPPORTED;
    const bool append = new_k != nullptr || new_v != nullptr;
    if (append && (!new_k || !new_v)) return BG_ERR_INVALID_ARG;
    if (n_tokens + (append ? 1 : 0) > suffix_max) return BG_ERR_INVALID_ARG;
    if (R == 0) return BG_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !parent_idx) return BG_ERR_INVALID_ARG;
    if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) || !aligned(dst_v, 16) ||
        !aligned(parent_idx, 4) || (new_k && !aligned(new_k, 16)) || (new_v && !aligned(new_v, 16)) ||
        (dev_status && !aligned(dev_status, 4)))
        return BG_ERR_INVALID_ARG;
    const size_t bytes = static_cast<size_t>(R) * W * suffix_max * Hkv * head_dim * 2;
    const size_t nbytes = static_cast<size_t>(R) * W * Hkv * head_dim * 2;
    if (overlap(dst_k, bytes, src_k, bytes) || overlap(dst_k, bytes, src_v, bytes) ||
        overlap(dst_v, bytes, src_k, bytes) || overlap(dst_v, bytes, src_v, bytes) ||
        overlap(dst_k, bytes, dst_v, bytes) || overlap(dst_k, bytes, new_k, nbytes) ||
        overlap(dst_k, bytes, new_v, nbytes) || overlap(dst_v, bytes, new_k, nbytes) ||
        overlap(dst_v, bytes, new_v, nbytes))
        return BG_ERR_INVALID_ARG;
    if (launch_suffix_reorder(src_k, src_v, dst_k, dst_v, parent_idx, new_k, new_v, R, W, suffix_max, n_tokens, Hkv,
                              head_dim, dev_status, stream) != cudaSuccess)
        return BG_ERR_CUDA;
    return BG_OK;
}

size_t bg_beam_select_workspace_size(int32_t R, int32_t W, int32_t V)
{
    (void)V;
    if (R < 0 || W <= 0) return 0;
    const size_t cand = static_cast<size_t>(R) * W * W;     // per-beam candidates: value + token
    const size_t part = static_cast<size_t>(R) * beam_select_slices(R, W) * W;   // merge level 1: key + index
    auto al = [](size_t b) { return (b + 255) & ~size_t(255); };
    return al(cand * 4) + al(cand * 4) + al(static_cast<size_t>(R) * W * 4) + al(part * 4) + al(part * 4);
}

bg_status_t bg_beam_select(const float *logits, const float *cum, int32_t R, int32_t W, int32_t V,
                           int32_t *token_out, int32_t *parent_out, float *score_out, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream)
{
    if (R < 0) return BG_ERR_INVALID_ARG;
    if (W < 1 || W > BG_MAX_BEAM || V < W || V > BG_MAX_VOCAB) return BG_ERR_UNSUPPORTED;
    if (R == 0) return BG_OK;
    if (!logits || !cum || !token_out || !parent_out || !score_out || !workspace) return BG_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || !aligned(cum, 4) || !aligned(token_out, 4) || !aligned(parent_out, 4) ||
        !aligned(score_out, 4) || !aligned(workspace, 256))
        return BG_ERR_INVALID_ARG;
    if (workspace_bytes < bg_beam_select_workspace_size(R, W, V)) return BG_ERR_INVALID_ARG;
    const size_t rw = static_cast<size_t>(R) * W;
    const size_t lbytes = rw * V * sizeof(float);
    const void *ins[3] = {logits, cum, workspace};
    const size_t in_bytes[3] = {lbytes, rw * sizeof(float), workspace_bytes};
    const void *outs[3] = {token_out, parent_out, score_out};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 3; ++i)
            if (overlap(outs[o], rw * 4, ins[i], in_bytes[i])) return BG_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlap(outs[o], rw * 4, outs[o2], rw * 4)) return BG_ERR_INVALID_ARG;
    }
    const size_t cand = rw * W;
    const size_t part = static_cast<size_t>(R) * beam_select_slices(R, W) * W;
    auto al = [](size_t b) { return (b + 255) & ~size_t(255); };
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *cand_val = reinterpret_cast<float *>(ws);
    int32_t *cand_tok = reinterpret_cast<int32_t *>(ws + al(cand * 4));
    float *row_lse = reinterpret_cast<float *>(ws + 2 * al(cand * 4));
    uint32_t *part_key = reinterpret_cast<uint32_t *>(ws + 2 * al(cand * 4) + al(rw * 4));
    int32_t *part_idx = reinterpret_cast<int32_t *>(ws + 2 * al(cand * 4) + al(rw * 4) + al(part * 4));
    if (launch_beam_select(logits, cum, R, W, V, token_out, parent_out, score_out, cand_val, cand_tok, row_lse,
                           part_key, part_idx, stream) != cudaSuccess)
        return BG_ERR_CUDA;
    return BG_OK;
}

bg_status_t bg_selftest_wait_timeout(int32_t *dev_status, unsigned long long *waited_ns, cudaStream_t stream)
{
    if (!dev_status || !waited_ns || !aligned(dev_status, 4) || !aligned(waited_ns, 8)) return BG_ERR_INVALID_ARG;
    if (launch_wait_timeout_selftest(dev_status, waited_ns, stream) != cudaSuccess) return BG_ERR_CUDA;
    return BG_OK;
}

}  // extern "C"
