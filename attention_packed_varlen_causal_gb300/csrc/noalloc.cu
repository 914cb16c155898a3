// noalloc.cu -- bg_packed_prefill_attn_noalloc: packed prefill attention for
// callers that cannot allocate device memory.
//
// bg_packed_prefill_attn needs a caller-provided workspace for the work list
// it builds on the device.  Some callers have no way to provide one: code
// that runs inside a runtime which owns every device buffer and hands a
// kernel call only its inputs and outputs, or a latency-critical serving loop
// that must not call cudaMalloc (it can synchronise the device and fragment
// memory).  This entry point keeps that scratch in a fixed-size array in the
// library's own device memory instead, so such a caller passes only the
// inputs and outputs.
//
// Cost of that convenience:
//   * every GPU that loads the library holds kNoAllocScratchBytes of device
//     memory until the process exits;
//   * all calls on a device share the one array, so two calls that may run
//     at the same time on the GPU (different streams, overlapping graphs)
//     race on it -- serialise them;
//   * problems whose work list does not fit are rejected.
// No clearing is needed between calls: each call's first kernel rewrites the
// header and every work-list entry before the attention kernel reads them.
#include <mutex>

#include "bg_attn.h"
#include "bg_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = BG_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// The scratch array.  In host code `g_scratch` is only a stand-in for the
// symbol, not a device address: the address kernels must be given comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device (with that device current) and cached.
bg_status_t scratch_for_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return BG_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return BG_OK;
}

}  // namespace

extern "C" bg_status_t bg_packed_prefill_attn_noalloc(const void *q, const void *k, const void *v,
                                                      const int32_t *cu_seqlens, int32_t num_seqs,
                                                      int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                                      int32_t Hkv, int32_t head_dim, float scale, void *out,
                                                      float *lse, int32_t *dev_status, cudaStream_t stream)
{
    if (num_seqs < 0 || total_tokens < 0) return BG_ERR_INVALID_ARG;
    const size_t need = bg_packed_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim);
    if (need > kNoAllocScratchBytes) return BG_ERR_UNSUPPORTED;   // work list would not fit the fixed scratch
    void *scratch = nullptr;
    const bg_status_t st = scratch_for_current_device(&scratch);
    if (st != BG_OK) return st;
    return bg_packed_prefill_attn(q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim, scale,
                                  out, lse, scratch, kNoAllocScratchBytes, dev_status, stream);
}
