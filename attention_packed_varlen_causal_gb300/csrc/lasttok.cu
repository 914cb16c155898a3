// lasttok.cu -- attention of each packed sequence's last valid token.
//
// "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", abstract and section
// 1.1: a Prefill-Only request is served from the next-token logits at the last
// valid position of each sequence, so the last layer needs the attention
// output of that one row, over all L keys of its sequence (row L-1 of the
// causal prefill, no mask).  That is O(L) work per sequence and head instead of
// O(L^2), and it is bound by reading each sequence's K and V once per kv head,
// so it runs on the CUDA cores, not the tensor cores.
//
// One CTA (256 threads, 8 warps) per (sequence, kv head) serves the g query
// heads of that kv head, over chunks of 128 keys with an online softmax in fp32:
//   stage   the chunk's K and V rows of this kv head are copied into shared
//           memory with cp.async, 16 bytes per copy, all in flight at once and
//           costing no registers;
//   scores  thread t owns 8 columns (16 bytes) of K and every (256/(d/8))-th key
//           of the chunk: partial dot products with its columns of the g scaled
//           queries, summed over the lanes of a row with shuffles;
//   softmax warp w takes heads w, w + 8, ...: chunk max, the running max and
//           rescale, exp2, chunk sum;
//   values  the same thread mapping over V, accumulated for all g heads in
//           registers;
// then the partial outputs are summed (shuffles inside a warp, shared memory
// across the 8 warps), normalised and stored (bf16), with the LSE if asked for.
#include "bg_internal.h"
#include "bg_ptx.cuh"

#include <cuda_bf16.h>

#include <cmath>

namespace bg {

namespace {
constexpr int kLtThreads = 256;
constexpr int kLtWarps = kLtThreads / 32;
constexpr int kLtChunk = 128;          // keys per chunk

// dynamic shared memory: K and V of a chunk (bf16 [128][D] each; after the last chunk the
// per-warp partial outputs [8][g][D] fp32 reuse this space), then qs[g][D] | sc[g][128] |
// st[3][g] (m, l, alpha), fp32
__host__ __device__ constexpr size_t lt_smem_bytes(int g, int D)
{
    return 2 * static_cast<size_t>(kLtChunk) * D * 2 +
           (static_cast<size_t>(g) * D + static_cast<size_t>(g) * kLtChunk + 3 * static_cast<size_t>(g)) * 4;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// G: a power of two >= g = Hq / Hkv; the per-thread arrays are sized by it
template <int D, int G>
__global__ void __launch_bounds__(kLtThreads)
    last_token_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ v, const int32_t *__restrict__ cu, int32_t B, int32_t T,
                      int32_t max_seqlen, int32_t Hq, int32_t Hkv, float scale_log2, __nv_bfloat16 *__restrict__ out,
                      float *__restrict__ lse, int32_t *dev_status)
{
    extern __shared__ __align__(16) uint8_t lt_smem[];
    const int g = Hq / Hkv;
    const int seq = static_cast<int>(blockIdx.x) / Hkv;
    const int kh = static_cast<int>(blockIdx.x) - seq * Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dep_launch();
    grid_dep_wait();     // the previous kernel of the stream has completed
    __nv_bfloat16 *ks = reinterpret_cast<__nv_bfloat16 *>(lt_smem);    // [128][D]
    __nv_bfloat16 *vs = ks + kLtChunk * D;                              // [128][D]
    float *part = reinterpret_cast<float *>(lt_smem);                   // [8][g][D], after the last chunk
    float *qs = reinterpret_cast<float *>(vs + kLtChunk * D);          // [g][D], scaled by scale * log2(e)
    float *sc = qs + g * D;                    // [g][128]
    float *st_m = sc + g * kLtChunk;           // [g] running max (base-2 units)
    float *st_l = st_m + g;                    // [g] running sum
    float *st_a = st_l + g;                    // [g] rescale factor of the current chunk

    const int a = cu[seq], b = cu[seq + 1];
    const bool bad = a < 0 || b < a || b > T || b - a > max_seqlen || (seq == 0 && a != 0) || (seq == B - 1 && b != T);
    if (bad) {
        if (tid == 0 && dev_status) atomicOr(dev_status, BG_DEVSTAT_CU_SEQLENS);
        return;
    }
    const int L = b - a;
    if (L == 0) return;

    for (int i = tid; i < g * D; i += kLtThreads) {
        const int h = i / D, c = i - h * D;
        qs[i] = __bfloat162float(q[(static_cast<int64_t>(seq) * Hq + kh * g + h) * D + c]) * scale_log2;
    }
    for (int h = tid; h < g; h += kLtThreads) {
        st_m[h] = -INFINITY;
        st_l[h] = 0.f;
    }
    // value pass mapping: thread tid owns the 8 columns of column block cb = tid % NCB and
    // the keys tid / NCB + KPT m of a chunk
    constexpr int NCB = D / 8;                 // 16-byte column blocks of a row
    constexpr int KPT = kLtThreads / NCB;      // threads per column block
    constexpr int NM = kLtChunk / KPT;         // keys per thread and chunk
    const int cb = tid % NCB, kr0 = tid / NCB;
    float acc[G][8];                           // g <= G heads x this thread's 8 columns
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    __syncthreads();

    // this thread's 8 columns of every scaled query (zero for heads past g)
    float qf[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[h][e] = (h < g) ? qs[h * D + 8 * cb + e] : 0.f;
    const int64_t row_stride = static_cast<int64_t>(Hkv) * D;    // elements between tokens
    const __nv_bfloat16 *kb = k + static_cast<int64_t>(a) * row_stride + kh * D;
    const __nv_bfloat16 *vb = v + static_cast<int64_t>(a) * row_stride + kh * D;
    for (int c0 = 0; c0 < L; c0 += kLtChunk) {
        const int n = (L - c0 < kLtChunk) ? L - c0 : kLtChunk;
        // ---- stage K and V rows c0 .. c0 + n - 1 (16-byte blocks, all copies in flight)
        for (int i = tid; i < n * NCB; i += kLtThreads) {
            const int r = i / NCB, c = i - r * NCB;
            cp_async16(ks + r * D + 8 * c, kb + (c0 + r) * row_stride + 8 * c);
            cp_async16(vs + r * D + 8 * c, vb + (c0 + r) * row_stride + 8 * c);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        // ---- scores: thread tid reads block cb of keys kr0 + KPT m (a warp reads whole rows,
        // conflict-free); the NCB partial dot products of a key are summed with shuffles
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            const int j = kr0 + KPT * m;
            const uint4 kw = *reinterpret_cast<const uint4 *>(ks + j * D + 8 * cb);
            const __nv_bfloat162 *w2 = reinterpret_cast<const __nv_bfloat162 *>(&kw);
            float kf[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(w2[e]);
                kf[2 * e] = f.x;
                kf[2 * e + 1] = f.y;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float dsum = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) dsum = fmaf(qf[h][e], kf[e], dsum);
#pragma unroll
                for (int o = 1; o < NCB; o <<= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
                if (h < g && cb == 0 && j < n) sc[h * kLtChunk + j] = dsum;
            }
        }
        __syncthreads();
        // ---- softmax of the chunk: warp w takes heads w, w + 8, ...
        for (int h = warp; h < g; h += kLtWarps) {
            float* sh = sc + h * kLtChunk;
            float mx = -INFINITY;
            for (int j = lane; j < n; j += 32) mx = fmaxf(mx, sh[j]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = st_m[h];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int j = lane; j < n; j += 32) {
                const float p = exp2f(sh[j] - m_new);
                sh[j] = p;
                sum += p;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) {
                const float alpha = exp2f(m_old - m_new);   // 0 on the first chunk (m_old = -inf)
                st_a[h] = alpha;
                st_l[h] = st_l[h] * alpha + sum;
                st_m[h] = m_new;
            }
        }
        __syncthreads();
        // ---- values: warp w, keys c0 + 32w ..; lane owns columns E*lane .. E*lane + E-1
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if (h < g) {
                const float al = st_a[h];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] *= al;
            }
        }
        // ---- values: the same mapping over V
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            const int j = kr0 + KPT * m;
            if (j < n) {
                const uint4 vw = *reinterpret_cast<const uint4 *>(vs + j * D + 8 * cb);
                const __nv_bfloat162 *w2 = reinterpret_cast<const __nv_bfloat162 *>(&vw);
                float vf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(w2[e]);
                    vf[2 * e] = f.x;
                    vf[2 * e + 1] = f.y;
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    if (h < g) {
                        const float pw = sc[h * kLtChunk + j];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pw, vf[e], acc[h][e]);
                    }
                }
            }
        }
        __syncthreads();   // K, V and sc are rewritten by the next chunk
    }
    // ---- combine the 8 warps' partial outputs, normalise, store
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int o = NCB; o < 32; o <<= 1) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
    if (lane < NCB) {
#pragma unroll
        for (int h = 0; h < G; ++h)
            if (h < g)
#pragma unroll
                for (int e = 0; e < 8; ++e) part[(warp * g + h) * D + 8 * cb + e] = acc[h][e];
    }
    __syncthreads();
    for (int i = tid; i < g * D; i += kLtThreads) {
        const int h = i / D, c = i - h * D;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kLtWarps; ++w) s += part[(w * g + h) * D + c];
        out[(static_cast<int64_t>(seq) * Hq + kh * g + h) * D + c] = __float2bfloat16_rn(s / st_l[h]);
    }
    if (lse) {
        for (int h = tid; h < g; h += kLtThreads)
            lse[static_cast<int64_t>(seq) * Hq + kh * g + h] = (st_m[h] + log2f(st_l[h])) * 0.69314718055994530942f;
    }
}

template <int D, int G>
cudaError_t launch_lt(const void *q, const void *k, const void *v, const int32_t *cu, int32_t B, int32_t T,
                      int32_t max_seqlen, int32_t Hq, int32_t Hkv, float scale_log2, void *out, float *lse,
                      int32_t *dev_status, cudaStream_t stream)
{
    const int g = Hq / Hkv;
    const size_t smem = lt_smem_bytes(g, D);
    auto kern = last_token_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = static_cast<int64_t>(B) * Hkv;
    return launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(kLtThreads), smem, stream,
                            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                            static_cast<const __nv_bfloat16 *>(v), cu, B, T, max_seqlen, Hq, Hkv, scale_log2,
                            static_cast<__nv_bfloat16 *>(out), lse, dev_status);
}
}  // namespace

int last_token_max_group() { return 16; }

cudaError_t launch_last_token_attn(int head_dim, const void *q, const void *k, const void *v, const int32_t *cu,
                                   int32_t B, int32_t T, int32_t max_seqlen, int32_t Hq, int32_t Hkv, float scale,
                                   void *out, float *lse, int32_t *dev_status, cudaStream_t stream)
{
    const float sl2 = scale * 1.4426950408889634f;
    const int g = Hq / Hkv;
#define BG_LT(DD, GG) \
    if (head_dim == DD && g <= GG) return launch_lt<DD, GG>(q, k, v, cu, B, T, max_seqlen, Hq, Hkv, sl2, out, lse, dev_status, stream)
    BG_LT(128, 2); BG_LT(128, 4); BG_LT(128, 8); BG_LT(128, 16);
    BG_LT(64, 2); BG_LT(64, 4); BG_LT(64, 8); BG_LT(64, 16);
#undef BG_LT
    return cudaErrorInvalidValue;
}

}  // namespace bg
