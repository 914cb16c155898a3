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
//   * all calls in one context share the one array, so two calls that may run
//     at the same time on the GPU (different streams, overlapping graphs)
//     race on it -- serialise them;
//   * problems whose work list does not fit are rejected.
// No clearing is needed between calls: each call's first kernel rewrites the
// header and every work-list entry before the attention kernel reads them.
#include <cudaTypedefs.h>

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

// The array's device address is looked up once per CUDA context and cached
// under that context's unique ID (cuCtxGetId).  A context made after
// cudaDeviceReset, or a non-primary context the caller makes current, has a
// new ID, so it gets its own lookup instead of a stale address.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_entry_once;

void resolve_entry_points()
{
    std::call_once(g_entry_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
}

constexpr int kCacheSlots = 64;
struct Slot {
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_mutex;
Slot g_cache[kCacheSlots] = {};
int g_next = 0;   // next slot to fill (oldest entry is replaced once all are used)

// ID of the current context; makes the device's primary context current first if the
// calling thread has none yet (cudaSetDevice binds it).
bool current_context_id(unsigned long long *id)
{
    resolve_entry_points();
    if (!g_ctx_current || !g_ctx_id) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
    if (ctx == nullptr) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
        if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    }
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch in the current context.
bg_status_t scratch_for_current_context(void **out)
{
    unsigned long long id = 0;
    if (!current_context_id(&id)) return BG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < kCacheSlots; ++i) {
        if (g_cache[i].ptr != nullptr && g_cache[i].ctx_id == id) {
            *out = g_cache[i].ptr;
            return BG_OK;
        }
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return BG_ERR_CUDA;
    g_cache[g_next] = Slot{id, p};
    g_next = (g_next + 1) % kCacheSlots;
    *out = p;
    return BG_OK;
}

}  // namespace

extern "C" bg_status_t bg_packed_prefill_attn_noalloc(const void *q, const void *k, const void *v,
                                                      const int32_t *cu_seqlens, int32_t num_seqs,
                                                      int32_t total_tokens, int32_t max_seqlen, int32_t Hq,
                                                      int32_t Hkv, int32_t head_dim, float scale, void *out,
                                                      float *lse, int32_t *dev_status, cudaStream_t stream)
{
    // the same argument checks as bg_packed_prefill_attn come first, so an invalid call
    // reports what is wrong with it whatever its size
    bool noop = false;
    const bg_status_t chk = bg::prefill_check_args(q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv,
                                                   head_dim, scale, out, lse, dev_status, &noop);
    if (chk != BG_OK || noop) return chk;
    const size_t need = bg_packed_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim);
    if (need > kNoAllocScratchBytes) return BG_ERR_UNSUPPORTED;   // work list would not fit the fixed scratch
    void *scratch = nullptr;
    const bg_status_t st = scratch_for_current_context(&scratch);
    if (st != BG_OK) return st;
    return bg_packed_prefill_attn(q, k, v, cu_seqlens, num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim, scale,
                                  out, lse, scratch, kNoAllocScratchBytes, dev_status, stream);
}
