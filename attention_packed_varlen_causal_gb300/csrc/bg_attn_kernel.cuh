// bg_attn_kernel.cuh -- warp-specialised tcgen05 attention kernel for sm_103a.
//
// One kernel body serves both hot-path attention modes of the bounded-
// generation engine ("SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化",
// abstract and section 1.2):
//   * Prefill: packed variable-length causal GQA attention.  A work item is
//     (sequence, 128-row query tile, NH query heads of one kv head); its key
//     tiles are 0..qtile (causal), the last one masked on the diagonal.
//   * Decode (shared-prompt phase): a work item is (request, kv head, NH
//     tiles of beams x group heads); every tile is a dense 128-row block of
//     queries of several beams against the one prompt K/V of the request,
//     followed in the epilogue by each beam's own suffix keys and the merge.
//
// Per CTA (persistent, one per SM, static round-robin over items):
//   warp 0      TMA producer: Q tiles of the item, then K/V tiles through an
//               NSTAGE ring (one K and one V slot per stage)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer:
//               S_h = Q_h K^T (SMEM x SMEM), then O_h += P_h V (P_h read from
//               TMEM, where the softmax warps wrote it over S_h)
//   warps 2-3   idle
//   warps 4..   NH softmax warpgroups; thread t of group h owns query row t
//               of tile h (TMEM lane t): online softmax in fp32 with the
//               exponent in base 2, lazy rescaling of O (only when the row
//               maximum grows by more than 2^8), epilogue normalisation and
//               bf16 store.
// TMEM: S_h at columns [128h, 128h+128), O_h at [128 NH + D h, ... + D).
// Every wait is bounded (bg::mbar_wait); on a time-out every role leaves its
// loop, in-flight copies and MMAs are drained, TMEM is freed and the kernel
// reports BG_DEVSTAT_TIMEOUT.
#pragma once

#include "bg_attn.h"
#include "bg_ptx.cuh"

namespace bg {

constexpr int kRows = 128;                 // query rows per tile = TMEM lanes
constexpr int kKeys = 128;                 // keys per K/V tile
constexpr int kBoxBytes = 128 * 128;       // 128 rows x 64 bf16 (one swizzle-128B column block)
constexpr float kRescaleLog2 = 8.0f;       // rescale O only if the max grew by > 2^8
constexpr int kMaxSuffix = 16;

enum class Mode : int { Prefill = 0, Decode = 1 };

struct AttnParams {
    int32_t Hq, Hkv, g;            // g = Hq / Hkv
    float scale_log2;              // softmax scale * log2(e)
    __nv_bfloat16 *out;
    int32_t *dev_status;           // may be null
    int32_t *err_word;             // extra device word that receives timeouts, or null
    // prefill
    const int32_t *cu_seqlens;
    const int2 *work;              // (sequence, query tile) entries, longest sequences first
    const int32_t *work_hdr;       // [0] status, [1] number of entries
    int32_t n_head_groups;         // items per entry = Hkv * groups_per_kv
    int32_t groups_per_kv;         // ceil(g / NH)
    float *lse;                    // may be null
    // decode
    const int32_t *cu_prompt;
    int32_t R, W, BT;              // BT = beams per query tile = 128 / g
    int32_t pairs_per_rk;          // ceil(ceil(W / BT) / NH)
    int32_t max_prompt_len, total_prompt;
    const __nv_bfloat16 *q;        // decode queries (for the suffix dot products)
    const __nv_bfloat16 *suffix_k, *suffix_v;
    int32_t suffix_len, suffix_max;
    int32_t n_items_decode;
};

template <int D, int NH, int NSTAGE>
struct AttnCfg {
    static constexpr int NB = D / 64;                       // 128-byte column blocks per row
    static constexpr int kQBytes = NH * NB * kBoxBytes;
    static constexpr int kTileBytes = NB * kBoxBytes;       // one K or V tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + NSTAGE * kTileBytes;
    static constexpr int kOffBar = kOffV + NSTAGE * kTileBytes;
    // q_full, q_empty, mma_final, k_full[NS], v_full[NS], kv_empty[NS], s_full[NH], p_full[NH], pv_done[NH]
    static constexpr int kNumBars = 3 + 3 * NSTAGE + 3 * NH;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-byte alignment
    static constexpr int kThreads = 128 * (1 + NH);
    static constexpr int kColS = 0;
    static constexpr int kColO = 128 * NH;
    static constexpr int kColsUsed = 128 * NH + D * NH;
    static constexpr int kTmemCols = kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64 : kColsUsed <= 128 ? 128
                                   : kColsUsed <= 256 ? 256 : 512;
    static_assert(kColsUsed <= 512, "TMEM overflow");
    static_assert(kSmemBytes <= 232448, "shared memory overflow");
};

// Everything every role needs to know about one work item.
struct Item {
    int valid;       // 0: skip entirely (bad device data)
    int n_tiles;     // K/V tiles to stream (may be 0 in decode)
    int kh;          // kv head
    int kv_row0;     // first packed K/V row of the sequence / prompt
    int kv_len;      // sequence length (prefill) or prompt length (decode)
    // prefill
    int seq_start, qt, head0;
    // decode
    int r, bt0;
};

template <Mode MODE, int NH>
__device__ __forceinline__ Item load_item(const AttnParams &p, int it)
{
    Item I;
    if constexpr (MODE == Mode::Prefill) {
        const int e = it / p.n_head_groups;
        const int hg = it - e * p.n_head_groups;
        const int2 ent = p.work[e];
        I.kh = hg / p.groups_per_kv;
        const int hp = hg - I.kh * p.groups_per_kv;
        I.head0 = I.kh * p.g + hp * NH;
        I.seq_start = p.cu_seqlens[ent.x];
        I.kv_len = p.cu_seqlens[ent.x + 1] - I.seq_start;
        I.qt = ent.y;
        I.kv_row0 = I.seq_start;
        I.n_tiles = ent.y + 1;
        I.valid = 1;
        I.r = 0;
        I.bt0 = 0;
    } else {
        const int per_r = p.Hkv * p.pairs_per_rk;
        I.r = it / per_r;
        const int rem = it - I.r * per_r;
        I.kh = rem / p.pairs_per_rk;
        I.bt0 = (rem - I.kh * p.pairs_per_rk) * NH;
        const int a = p.cu_prompt[I.r];
        const int b = p.cu_prompt[I.r + 1];
        const bool ok = a >= 0 && b >= a && b <= p.total_prompt && (b - a) <= p.max_prompt_len &&
                        (b - a) + p.suffix_len > 0;
        I.valid = ok ? 1 : 0;
        I.kv_row0 = a;
        I.kv_len = ok ? b - a : 0;
        I.n_tiles = ok ? (b - a + kKeys - 1) / kKeys : 0;
        I.seq_start = 0;
        I.qt = 0;
        I.head0 = 0;
    }
    return I;
}

// Lane 0 waits, the result is broadcast: the whole warp leaves together.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

template <Mode MODE, int D, int NH, int NSTAGE>
__global__ void __launch_bounds__(128 * (1 + NH), 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p)
{
    using C = AttnCfg<D, NH, NSTAGE>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the shared-window offset (swizzle-128B atoms need it)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *q_full = bars + 0;
    uint64_t *q_empty = bars + 1;
    uint64_t *mma_final = bars + 2;
    uint64_t *k_full = bars + 3;
    uint64_t *v_full = k_full + NSTAGE;
    uint64_t *kv_empty = v_full + NSTAGE;
    uint64_t *s_full = kv_empty + NSTAGE;
    uint64_t *p_full = s_full + NH;
    uint64_t *pv_done = p_full + NH;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int n_items;
    if constexpr (MODE == Mode::Prefill) {
        n_items = (p.work_hdr[0] == 0) ? p.work_hdr[1] * p.n_head_groups : 0;
    } else {
        n_items = p.n_items_decode;
    }

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(mma_final, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int h = 0; h < NH; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&p_full[h], 128);
            mbar_init(&pv_done[h], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if constexpr (MODE == Mode::Decode) {
        // Decode query tiles fill only BT*g <= 128 rows; keep the rest zero.
        uint4 *q4 = reinterpret_cast<uint4 *>(smem + C::kOffQ);
        for (int i = threadIdx.x; i < C::kQBytes / 16; i += blockDim.x) q4[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // =============================================================== producer
        if (lane == 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            uint32_t n_q = 0;          // Q loads issued
            uint32_t n_kv = 0;         // K/V tiles issued
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const Item I = load_item<MODE, NH>(p, it);
                if (!I.valid || I.n_tiles == 0) continue;
                if (n_q > 0 && !mbar_wait(q_empty, (n_q - 1) & 1, abort_flag)) { ok = false; break; }
                if constexpr (MODE == Mode::Prefill) {
                    mbar_arrive_expect_tx(q_full, NH * C::NB * kBoxBytes);
                    const int row = I.seq_start + I.qt * kRows;
                    for (int h = 0; h < NH; ++h)
                        for (int b = 0; b < C::NB; ++b)
                            tma_load_3d(smem + C::kOffQ + (h * C::NB + b) * kBoxBytes, &tm_q, q_full, b * 64,
                                        I.head0 + h, row, pol_q);
                } else {
                    const uint32_t box = static_cast<uint32_t>(p.BT * p.g * 128);
                    mbar_arrive_expect_tx(q_full, NH * C::NB * box);
                    for (int h = 0; h < NH; ++h)
                        for (int b = 0; b < C::NB; ++b)
                            tma_load_4d(smem + C::kOffQ + (h * C::NB + b) * kBoxBytes, &tm_q, q_full, b * 64, 0,
                                        I.kh, I.r * p.W + (I.bt0 + h) * p.BT, pol_q);
                }
                ++n_q;
                for (int j = 0; j < I.n_tiles; ++j) {
                    const int st = n_kv % NSTAGE;
                    const uint32_t use = n_kv / NSTAGE;
                    if (use > 0 && !mbar_wait(&kv_empty[st], (use - 1) & 1, abort_flag)) { ok = false; break; }
                    const int row = I.kv_row0 + j * kKeys;
                    mbar_arrive_expect_tx(&k_full[st], C::kTileBytes);
                    for (int b = 0; b < C::NB; ++b)
                        tma_load_3d(smem + C::kOffK + st * C::kTileBytes + b * kBoxBytes, &tm_k, &k_full[st],
                                    b * 64, I.kh, row, pol_kv);
                    mbar_arrive_expect_tx(&v_full[st], C::kTileBytes);
                    for (int b = 0; b < C::NB; ++b)
                        tma_load_3d(smem + C::kOffV + st * C::kTileBytes + b * kBoxBytes, &tm_v, &v_full[st],
                                    b * 64, I.kh, row, pol_kv);
                    ++n_kv;
                }
            }
            // Let every copy this thread started land before the CTA exits.
            if (n_q > 0) mbar_wait_drain(q_full, (n_q - 1) & 1);
            for (int st = 0; st < NSTAGE; ++st) {
                const uint32_t uses = n_kv / NSTAGE + (st < static_cast<int>(n_kv % NSTAGE) ? 1u : 0u);
                if (uses > 0) {
                    mbar_wait_drain(&k_full[st], (uses - 1) & 1);
                    mbar_wait_drain(&v_full[st], (uses - 1) & 1);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // =============================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kKeys, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 1);
            const uint32_t sq = smem_u32(smem + C::kOffQ);
            const uint32_t sk = smem_u32(smem + C::kOffK);
            const uint32_t sv = smem_u32(smem + C::kOffV);
            uint32_t n_q = 0, n_kv = 0;
            uint32_t n_pv[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) n_pv[h] = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const Item I = load_item<MODE, NH>(p, it);
                if (!I.valid || I.n_tiles == 0) continue;
                if (!mbar_wait(q_full, n_q & 1, abort_flag)) { ok = false; break; }
                ++n_q;
                for (int j = 0; j < I.n_tiles; ++j) {
                    const int st = n_kv % NSTAGE;
                    const uint32_t par = (n_kv / NSTAGE) & 1;
                    if (!mbar_wait(&k_full[st], par, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    for (int h = 0; h < NH; ++h) {
                        // S_h is free once the previous P_h (stored over it) has been consumed.
                        if (n_pv[h] > 0 && !mbar_wait(&pv_done[h], (n_pv[h] - 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_s = tmem + C::kColS + 128 * h;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                            const uint64_t a = sdesc_sw128(sq + h * C::NB * kBoxBytes + off, 16, 1024);
                            const uint64_t b = sdesc_sw128(sk + st * C::kTileBytes + off, 16, 1024);
                            mma_ss(d_s, a, b, kIdescQK, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&s_full[h]);
                    }
                    if (!ok) break;
                    if (j == I.n_tiles - 1) mma_commit(q_empty);   // Q of this item no longer needed
                    if (!mbar_wait(&v_full[st], par, abort_flag)) { ok = false; break; }
                    for (int h = 0; h < NH; ++h) {
                        if (!mbar_wait(&p_full[h], n_pv[h] & 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t d_o = tmem + C::kColO + D * h;
                        const uint32_t a_p = tmem + C::kColS + 128 * h;
#pragma unroll
                        for (int kk = 0; kk < kKeys / 16; ++kk) {
                            // V tile: 128 key rows of 128 bytes per column block; K = 16 rows per step.
                            const uint64_t b = sdesc_sw128(sv + st * C::kTileBytes + kk * 16 * 128, kBoxBytes, 1024);
                            mma_ts(d_o, a_p + kk * 8, b, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&pv_done[h]);
                        ++n_pv[h];
                    }
                    if (!ok) break;
                    mma_commit(&kv_empty[st]);
                    ++n_kv;
                }
            }
            // Drain: every MMA issued above completes before TMEM is released.
            mma_commit(mma_final);
            mbar_wait_drain(mma_final, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // =============================================================== softmax + epilogue
        const int h = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + C::kColS + 128 * h;
        const uint32_t tO = tmem + lane_addr + C::kColO + D * h;
        const float sl2 = p.scale_log2;
        uint32_t n_s = 0;     // S tiles consumed by this thread
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item I = load_item<MODE, NH>(p, it);
            if (!I.valid) {
                if constexpr (MODE == Mode::Decode) {
                    if (h == 0 && row == 0 && p.dev_status) {
                        const int a = p.cu_prompt[I.r], b = p.cu_prompt[I.r + 1];
                        const bool bad_cu = !(a >= 0 && b >= a && b <= p.total_prompt && (b - a) <= p.max_prompt_len);
                        atomicOr(p.dev_status, bad_cu ? BG_DEVSTAT_CU_PROMPT : BG_DEVSTAT_EMPTY_ROW);
                    }
                }
                continue;
            }
            float m = -INFINITY;   // running max of scaled logits (base-2 units)
            float l = 0.f;         // running sum of exp2(logit - m)
            for (int j = 0; j < I.n_tiles; ++j) {
                if (!warp_wait(&s_full[h], n_s & 1, abort_flag)) { ok = false; break; }
                ++n_s;
                tc_fence_after();
                float s[kKeys];
#pragma unroll
                for (int c = 0; c < kKeys / 32; ++c) tmem_ld32(tS + 32 * c, s + 32 * c);
                int lim = kKeys;   // columns < lim are valid keys for this row
                if (j == I.n_tiles - 1) {
                    if constexpr (MODE == Mode::Prefill) lim = row + 1;          // causal diagonal
                    else lim = I.kv_len - j * kKeys;                             // prompt tail
                }
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < kKeys; ++c) {
                    if (c >= lim) s[c] = -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
                const float m_new = fmaxf(m, mx * sl2);
                const bool grow = (j > 0) && (m_new > m + kRescaleLog2);
                if (j == 0) m = m_new;
                if (__any_sync(0xffffffffu, grow)) {
                    // O holds the sum of the previous tiles: wait for the last P.V, rescale in place.
                    if (!warp_wait(&pv_done[h], (n_s - 2) & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const float alpha = ex2(m - m_new);
                    m = m_new;
                    l *= alpha;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tO + 32 * c, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32f(tO + 32 * c, o);
                    }
                    tmem_st_wait();
                }
                float rs = 0.f;
#pragma unroll
                for (int c = 0; c < kKeys / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float a = ex2(fmaf(s[32 * c + 2 * i], sl2, -m));
                        const float b = ex2(fmaf(s[32 * c + 2 * i + 1], sl2, -m));
                        rs += a + b;
                        pk[i] = pack_bf16x2(a, b);
                    }
                    tmem_st16(tS + 16 * c, pk);   // P (bf16 pairs) over the first 64 columns of S
                }
                tmem_st_wait();
                l += rs;
                tc_fence_before();
                mbar_arrive(&p_full[h]);
            }
            if (!ok) break;

            // ------------------------------------------------------- epilogue
            if (I.n_tiles > 0) {
                if (!warp_wait(&pv_done[h], (n_s - 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
            }
            if constexpr (MODE == Mode::Prefill) {
                const int qrow = I.qt * kRows + row;
                const int head = I.head0 + h;
                const bool valid = qrow < I.kv_len && (head - I.kh * p.g) < p.g;
                const float inv_l = 1.f / l;
                __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(I.seq_start + qrow) * p.Hq + head) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tO + 32 * c, o);
                    if (valid) {
                        uint4 w[4];
                        uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
                        for (int i = 0; i < 16; ++i) wp[i] = pack_bf16x2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = w[i];
                    }
                }
                if (valid && p.lse) {
                    // natural-log sum-exp: (m + log2 l) * ln 2
                    p.lse[static_cast<int64_t>(I.seq_start + qrow) * p.Hq + head] =
                        (m + __log2f(l)) * 0.69314718055994530942f;
                }
            } else {
                const int local_beam = row / p.g;
                const int hh = row - local_beam * p.g;
                const int beam = (I.bt0 + h) * p.BT + local_beam;
                const bool valid = local_beam < p.BT && beam < p.W;
                const int head = I.kh * p.g + hh;
                const int64_t rb = static_cast<int64_t>(I.r) * p.W + beam;
                // suffix logits
                float z[kMaxSuffix];
                float m2 = m;
#pragma unroll
                for (int s = 0; s < kMaxSuffix; ++s) {
                    z[s] = -INFINITY;
                    if (valid && s < p.suffix_len) {
                        const uint4 *qp = reinterpret_cast<const uint4 *>(p.q + (rb * p.Hq + head) * D);
                        const uint4 *kp = reinterpret_cast<const uint4 *>(
                            p.suffix_k + ((rb * p.suffix_max + s) * p.Hkv + I.kh) * D);
                        float acc = 0.f;
#pragma unroll
                        for (int c = 0; c < D / 8; ++c) {
                            const uint4 qa = qp[c], ka = kp[c];
                            const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qa);
                            const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&ka);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 qf = __bfloat1622float2(q2[e]);
                                const float2 kf = __bfloat1622float2(k2[e]);
                                acc = fmaf(qf.x, kf.x, acc);
                                acc = fmaf(qf.y, kf.y, acc);
                            }
                        }
                        z[s] = acc * sl2;
                        m2 = fmaxf(m2, z[s]);
                    }
                }
                const float alpha = (I.n_tiles > 0) ? ex2(m - m2) : 0.f;
                float l2 = l * alpha;
                float ps[kMaxSuffix];
#pragma unroll
                for (int s = 0; s < kMaxSuffix; ++s) {
                    ps[s] = (s < p.suffix_len && valid) ? ex2(z[s] - m2) : 0.f;
                    l2 += ps[s];
                }
                const float inv_l = valid ? 1.f / l2 : 0.f;
                __nv_bfloat16 *dst = p.out + (rb * p.Hq + head) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    if (I.n_tiles > 0) {
                        tmem_ld32(tO + 32 * c, o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0.f;
                    }
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        for (int s = 0; s < p.suffix_len; ++s) {
                            const uint4 *vp = reinterpret_cast<const uint4 *>(
                                p.suffix_v + ((rb * p.suffix_max + s) * p.Hkv + I.kh) * D + 32 * c);
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint4 va = vp[u];
                                const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&va);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 vf = __bfloat1622float2(v2[e]);
                                    o[8 * u + 2 * e] = fmaf(ps[s], vf.x, o[8 * u + 2 * e]);
                                    o[8 * u + 2 * e + 1] = fmaf(ps[s], vf.y, o[8 * u + 2 * e + 1]);
                                }
                            }
                        }
                        uint4 w[4];
                        uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
                        for (int i = 0; i < 16; ++i) wp[i] = pack_bf16x2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = w[i];
                    }
                }
            }
        }
        (void)ok;
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) {
        if (p.err_word) atomicOr(p.err_word, BG_DEVSTAT_TIMEOUT);
        if (p.dev_status) atomicOr(p.dev_status, BG_DEVSTAT_TIMEOUT);
    }
}

}  // namespace bg
