// bg_attn_kernel.cuh -- warp-specialised tcgen05 attention kernel for sm_103a.
//
// One kernel body serves both hot-path attention modes of the bounded-
// generation engine ("SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化",
// abstract and section 1.2):
//   * Prefill: packed variable-length causal GQA attention.  A work item is
//     (sequence, 128-row query tile, NH query heads of one kv head); it
//     streams the 64-key tiles up to its diagonal (only valid tokens).
//   * Decode: a work item is (request, kv head, NH tiles of beams x group
//     heads); each tile is a dense 128-row block of queries of several beams
//     against the request's one prompt K/V.  The beams' own suffix keys follow
//     as a few more 64-key tiles of the same item: each holds the suffix slots
//     of a run of consecutive beams (TMA-gathered, beam-major), and every query
//     row keeps only the columns of its own beam.
//
// Per CTA (persistent, one per SM, static round-robin over items):
//   warp 0      TMA producer of Q and K: Q tiles of each item into one of two Q
//               buffers (the next item's Q loads while the current one
//               computes), K tiles of 64 keys through an NK-stage ring.  A K
//               stage is released by a plain arrive of each softmax
//               warpgroup once it has seen its S of that tile (so the QK
//               that read the stage has completed; no extra tcgen05.commit),
//               a Q buffer after the item's last QK.
//   warp 2      TMA producer of V: V tiles through an NV-stage ring.  A V stage
//               is released by the softmax warpgroups' same arrive, NS tiles
//               later: S of tile t complete implies every MMA issued before
//               that QK, the P.V of tile t-NS included, has completed.  Each
//               extra tcgen05.commit costs the MMA warps ~160 cycles, so stage
//               release piggybacks on barriers that exist anyway.
//   warps 1, 3  tcgen05.mma issuers, one per query tile h (warp 1 also
//               allocates TMEM); lane 0 alone runs the issue loop.  For every
//               key tile t the thread of tile h
//               issues S_h(t) = Q_h K(t)^T into one of NS S buffers of
//               tile h, NS-1 tiles ahead of O_h += P_h(t-NS+1) V,
//               so the tensor cores compute the next scores while the softmax
//               warps work on the current ones; the lookahead also crosses
//               item boundaries.  P is read from TMEM (written there by the
//               softmax warps over their S buffer).
//   warps 4..   NH softmax warpgroups; thread t of group h owns query row t of
//               tile h (TMEM lane t): masked running max in base-2 units,
//               lazy rescaling of O (only when the max grows by > 2^8),
//               exp2 on the SFU, bf16 P back to TMEM.  Epilogue (deferred to
//               after the next item's first tile): O read from TMEM,
//               normalised and packed to bf16 in registers, the buffer handed
//               back to the next P.V, then stored 32 columns at a time through a
//               2 KB per-warp staging area, so that each store instruction
//               writes 64-byte row segments of 8 rows.
//               Warps whose 32 rows are all masked for a key tile skip it.
// TMEM columns: S(h,b) at 64*(NS*h+b), O_h at 64*NS*NH + D*h.
// Ordering: the MMA warp issues ... QK(t+1), PV(t), QK(t+2), PV(t+1) ... from
// one thread, and tcgen05.mma executes in issue order, so QK(t+2) may be
// issued right after PV(t) although it overwrites the S buffer PV(t) reads P
// from.  The commit after QK(t) therefore also tells the softmax warps that
// PV(t-2) and everything before it has completed, which keeps every parity
// wait on pv_done unambiguous.
// Every wait is bounded (bg::mbar_wait); on a time-out every role leaves its
// loop, in-flight copies and MMAs are drained, TMEM is freed and the kernel
// reports BG_DEVSTAT_TIMEOUT.
#pragma once

#include "bg_attn.h"
#include "bg_ptx.cuh"

namespace bg {

constexpr int kRows = 128;                 // query rows per tile = TMEM lanes
constexpr int kKeys = 64;                  // keys per K/V tile
constexpr int kQBox = 128 * 128;           // 128 rows x 128 bytes (one 128-byte-swizzled column block)
constexpr int kKVBox = 64 * 128;           // 64 rows x 128 bytes
constexpr float kRescaleLog2 = 8.0f;       // rescale O only if the max grew by more than 2^8

enum class Mode : int { Prefill = 0, Decode = 1 };

struct AttnParams {
    int32_t Hq, Hkv, g;            // g = Hq / Hkv
    float scale_log2;              // softmax scale * log2(e)
    __nv_bfloat16 *out;
    int32_t *dev_status;           // may be null
    int32_t *err_word;             // extra device word that receives timeouts, or null
    // prefill
    const int32_t *cu_seqlens;
    const int4 *work;              // (sequence start, length, query tile, sequence) entries
    const int32_t *work_hdr;       // [0] status, [1] number of entries
    int32_t n_head_groups;         // items per entry = Hkv * groups_per_kv
    int32_t groups_per_kv;         // ceil(g / NH)
    float *lse;                    // may be null
    // decode
    const int32_t *cu_prompt;
    int32_t R, W, BT;              // BT = beams per query tile = 128 / g
    int32_t pairs_per_rk;          // ceil(ceil(W / BT) / NH)
    int32_t max_prompt_len, total_prompt;   // prefill: total_prompt = total tokens, R = sequences
    int32_t suffix_len;            // suffix slots per beam (t)
    int32_t suf_bpt;               // beams per suffix key tile (suf_bpt * t <= 64)
    int32_t suf_tx;                // bytes one suffix key tile brings (all column blocks)
    int32_t n_items_decode;
};

// QK8: Q and K arrive as one-byte E4M3 codes and Q.K^T runs as kind::f8f6f4 (V, P and P.V
// stay bf16); otherwise every operand is bf16.
template <int D, int NH, int NK, int NV, int NS, bool QK8 = false>
struct AttnCfg {
    static constexpr int NB = D / 64;                       // 128-byte column blocks of a bf16 row (V, O)
    static constexpr int NBQ = QK8 ? D / 128 : D / 64;      // 128-byte column blocks of a Q or K row
    static constexpr int kQKElemsPerBlock = QK8 ? 128 : 64; // Q/K elements per column block
    static constexpr int kQBytes = NH * NBQ * kQBox;        // one Q buffer (NH tiles)
    static constexpr int kKTileBytes = NBQ * kKVBox;        // one K tile
    static constexpr int kTileBytes = NB * kKVBox;          // one V tile
    static constexpr int kOffQ = 0;                         // two Q buffers
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + NK * kKTileBytes;
    static constexpr int kOffStage = kOffV + NV * kTileBytes;     // 2 KB per softmax warp
    static_assert(!QK8 || D == 128, "E4M3 Q/K rows are one 128-byte column block (head_dim 128)");
    static constexpr int kStageBytes = 32 * 64;
    static constexpr int kOffBar = kOffStage + 4 * NH * kStageBytes;
    // q_full[2] q_empty[2] mma_final k_full[NK] k_empty[NK] v_full[NV] v_empty[NV] s_full[NH][NS]
    // p_full[NH][NS] (one arrive per softmax warp) pv_done[NH][NS] o_staged[NH][2]
    static constexpr int kNumBars = 5 + 2 * NK + 2 * NV + 3 * NS * NH + 2 * NH;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-byte alignment
    static constexpr int kThreads = 128 * (1 + NH);
    // Register split (setmaxnreg): the kernel is compiled for kRegsLaunch registers per thread
    // (__maxnreg__), which the launcher checks against the compiled kernel before every launch;
    // warps 0-3 (TMA and MMA) then run with kRegsLight and the 8 softmax warps with kRegsSoftmax,
    // within the launch's total (kSplitRegs).
    static constexpr int kRegsLaunch = 168;
    static constexpr int kRegsLight = 64;
    static constexpr int kRegsSoftmax = 216;
    static constexpr int kSplitRegs = 4 * 32 * kRegsLight + 8 * 32 * kRegsSoftmax;
    static_assert(kThreads * kRegsLaunch <= 65536, "the launch must fit the register file");
    static_assert(kSplitRegs <= kThreads * kRegsLaunch, "register split exceeds the launch's allocation");
    static constexpr int kColO = 64 * NS * NH;
    static constexpr int kColsUsed = 64 * NS * NH + D * NH;
    static constexpr int kTmemCols = kColsUsed <= 128 ? 128 : kColsUsed <= 256 ? 256 : 512;
    static_assert(kColsUsed <= 512, "TMEM overflow");
    static_assert(kSmemBytes <= 232448, "shared memory overflow");
    static_assert(NK >= 2 && NV >= 2 && NS >= 2 && NS <= 3, "ring / buffer counts");
    // TMEM column of S buffer b of query tile h
    static __device__ __forceinline__ uint32_t col_s(int h, int b) { return static_cast<uint32_t>(64 * (NS * h + b)); }
};

// Everything every role needs to know about one work item.
struct Item {
    int valid;       // 0: skip entirely (bad device data)
    int n_tiles;     // 64-key K/V tiles to stream
    int n_prompt;    // of which from the sequence / prompt; decode: the rest hold suffix keys
    int kh;          // kv head
    int kv_row0;     // first packed K/V row of the sequence / prompt
    int kv_len;      // sequence length (prefill) or prompt length (decode)
    int seq_start, qt, head0;   // prefill
    int r, bt0;                 // decode
};

// The raw descriptor of item `it` in global memory (one 16-byte work entry in
// prefill, the two prompt offsets in decode).  Fetched one item ahead, so the
// load latency hides behind the current item.
template <Mode MODE>
__device__ __forceinline__ int4 fetch_raw(const AttnParams &p, int it)
{
    if constexpr (MODE == Mode::Prefill) {
        return p.work[it / p.n_head_groups];
    } else {
        const int r = it / (p.Hkv * p.pairs_per_rk);
        return make_int4(p.cu_prompt[r], p.cu_prompt[r + 1], 0, 0);
    }
}

template <Mode MODE, int NH>
__device__ __forceinline__ Item make_item(const AttnParams &p, int it, int4 raw)
{
    Item I;
    if constexpr (MODE == Mode::Prefill) {
        const int hg = it % p.n_head_groups;
        I.kh = hg / p.groups_per_kv;
        const int hp = hg - I.kh * p.groups_per_kv;
        I.head0 = I.kh * p.g + hp * NH;
        I.seq_start = raw.x;
        I.kv_len = raw.y;
        I.qt = raw.z;
        I.kv_row0 = I.seq_start;
        // keys up to the tile's last row, and never past the sequence end
        const int causal_tiles = 2 * raw.z + 2;
        const int len_tiles = (I.kv_len + kKeys - 1) / kKeys;
        I.n_tiles = causal_tiles < len_tiles ? causal_tiles : len_tiles;
        I.n_prompt = I.n_tiles;
        I.valid = 1;
        I.r = 0;
        I.bt0 = 0;
    } else {
        const int per_r = p.Hkv * p.pairs_per_rk;
        I.r = it / per_r;
        const int rem = it - I.r * per_r;
        I.kh = rem / p.pairs_per_rk;
        I.bt0 = (rem - I.kh * p.pairs_per_rk) * NH;
        const int a = raw.x;
        const int b = raw.y;
        const bool ok = a >= 0 && b >= a && b <= p.total_prompt && (b - a) <= p.max_prompt_len &&
                        (b - a) + p.suffix_len > 0;
        I.valid = ok ? 1 : 0;
        I.kv_row0 = a;
        I.kv_len = ok ? b - a : 0;
        I.n_prompt = ok ? (b - a + kKeys - 1) / kKeys : 0;
        // suffix tiles: the item's beams (NH tiles of BT, cut at W), suf_bpt per tile
        int nb = p.W - I.bt0 * p.BT;
        if (nb > NH * p.BT) nb = NH * p.BT;
        const int n_suf = (ok && p.suffix_len > 0) ? (nb + p.suf_bpt - 1) / p.suf_bpt : 0;
        I.n_tiles = I.n_prompt + n_suf;
        I.seq_start = 0;
        I.qt = 0;
        I.head0 = 0;
    }
    return I;
}

// Whether query tile h of a decode item is stored through the TMA unit out of its Q buffer
// (see the epilogue): only when all of its BT beams are beams of the request.  The MMA thread
// and the softmax warpgroup of h both evaluate it, so they agree on who releases the item's Q
// buffer: the MMA thread right after the item's last QK (the tile is then stored row by row),
// or the epilogue once the TMA unit has read the tile out of it.  Prefill tiles always take the
// row-by-row path: the prefill kernel is at its register limit, and the extra epilogue code made
// it slower than the store overlap gained.
template <Mode MODE>
__device__ __forceinline__ bool tile_store_via_tma(const AttnParams &p, const Item &I, int h)
{
    if constexpr (MODE == Mode::Prefill) {
        return false;
    } else {
        return (I.bt0 + h) * p.BT + p.BT <= p.W;
    }
}

// Walks the (item, key tile) sequence of one CTA, skipping items without
// tiles.  Every role walks the same sequence, so all agree on global tile
// numbers (which pick K/V stages, S buffers and barrier phases).
template <Mode MODE, int NH>
struct TileWalker {
    int it, j;           // current item index and tile within it
    int n_items;
    Item I;
    int4 nxt_raw;        // raw descriptor of item it + gridDim.x (prefetched)
    int n_q;             // items with tiles entered so far (selects the Q buffer)
    bool valid;

    __device__ void first(const AttnParams &p, int n_items_)
    {
        n_items = n_items_;
        n_q = 0;
        it = static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x);
        j = 0;
        valid = false;
        nxt_raw = make_int4(0, 0, 0, 0);
        if (static_cast<int>(blockIdx.x) < n_items) nxt_raw = fetch_raw<MODE>(p, blockIdx.x);
        next_item(p);
    }
    __device__ void next_item(const AttnParams &p)
    {
        for (it += gridDim.x; it < n_items; it += gridDim.x) {
            const int4 raw = nxt_raw;
            if (it + static_cast<int>(gridDim.x) < n_items) nxt_raw = fetch_raw<MODE>(p, it + gridDim.x);
            I = make_item<MODE, NH>(p, it, raw);
            if (I.valid && I.n_tiles > 0) {
                j = 0;
                valid = true;
                ++n_q;
                return;
            }
        }
        valid = false;
    }
    __device__ void advance(const AttnParams &p)
    {
        if (++j >= I.n_tiles) next_item(p);
    }
    __device__ int qbuf() const { return (n_q - 1) & 1; }
    __device__ uint32_t quse() const { return static_cast<uint32_t>((n_q - 1) >> 1); }
};

// Lane 0 waits, the result is broadcast: the whole warp leaves together.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

template <Mode MODE, int D, int NH, int NK, int NV, int NS, bool QK8 = false>
__global__ void __maxnreg__((AttnCfg<D, NH, NK, NV, NS, QK8>::kRegsLaunch))
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_sk,
                const __grid_constant__ CUtensorMap tm_sv, const __grid_constant__ CUtensorMap tm_o,
                const AttnParams p)
{
    using C = AttnCfg<D, NH, NK, NV, NS, QK8>;
    static_assert(!QK8 || MODE == Mode::Prefill, "E4M3 Q/K is a prefill variant");
    static_assert(NH == 2, "the register split and the warp roles assume two query tiles per CTA");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the shared-window offset (swizzle-128B atoms need it)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *q_full = bars + 0;         // [2]
    uint64_t *q_empty = bars + 2;        // [2]
    uint64_t *mma_final = bars + 4;
    uint64_t *k_full = bars + 5;            // [NK]
    uint64_t *k_empty = k_full + NK;        // [NK]
    uint64_t *v_full = k_empty + NK;        // [NV]
    uint64_t *v_empty = v_full + NV;        // [NV]
    uint64_t *s_full = v_empty + NV;        // [NH][NS]
    uint64_t *p_full = s_full + NS * NH;    // [NH][NS]
    // pv_done[h][b] completes when P.V of a tile stored in S buffer b is done.
    // One barrier per buffer (not per head): every wait on it is then for
    // the phase right after the last one its waiter already saw complete,
    // which is what makes a parity wait unambiguous.
    uint64_t *pv_done = p_full + NS * NH;   // [NH][NS]
    // o_staged[h][e & 1] completes when the four warps of softmax warpgroup h have written their
    // rows of its e-th TMA-stored output tile into the Q buffer.  No warp can arrive for the
    // group's next such tile before this phase completes: its next epilogue runs after the scores
    // of the item after next, whose Q load waits for the buffer this tile leaves from.  The second
    // barrier per group keeps consecutive phases apart all the same.
    uint64_t *o_staged = pv_done + NS * NH;   // [NH][2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    grid_dep_launch();   // the next kernel's CTAs may start their prologue (they wait before any global access)

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&q_full[b], 1);
            mbar_init(&q_empty[b], NH);   // one arrive per softmax warpgroup, from its epilogue
        }
        mbar_init(mma_final, NH);
        for (int s = 0; s < NK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], NH);   // one arrive per softmax warpgroup
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], NH);   // one arrive per softmax warpgroup
        }
        for (int i = 0; i < NS * NH; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);     // one arrive per softmax warp
            mbar_init(&pv_done[i], 1);
        }
        for (int i = 0; i < 2 * NH; ++i) mbar_init(&o_staged[i], 4);   // one arrive per warp
        *abort_flag = 0;
        fence_barrier_init();
    }
    if constexpr (MODE == Mode::Decode) {
        // Decode query tiles fill only BT*g <= 128 rows and suffix key tiles only suf_bpt*t
        // <= 64 rows; the rows past them keep what an earlier tile left (finite) or these
        // zeros, so the masked columns they feed multiply finite values only.
        uint4 *z4 = reinterpret_cast<uint4 *>(smem + C::kOffQ);
        for (int i = threadIdx.x; i < C::kOffStage / 16; i += blockDim.x) z4[i] = make_uint4(0, 0, 0, 0);
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
        tma_prefetch_desc(&tm_o);
        if constexpr (MODE == Mode::Decode) {
            tma_prefetch_desc(&tm_sk);
            tma_prefetch_desc(&tm_sv);
            // The first item's Q tiles into L2 while the previous kernel still runs: their place
            // depends on the item number only (not on cu_prompt), and the Q load after the wait
            // then comes from L2.
            const int it = static_cast<int>(blockIdx.x);
            if (it < p.n_items_decode) {
                const int per_r = p.Hkv * p.pairs_per_rk;
                const int r = it / per_r;
                const int rem = it - r * per_r;
                const int kh = rem / p.pairs_per_rk;
                const int bt0 = (rem - kh * p.pairs_per_rk) * NH;
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                    for (int b = 0; b < C::NB; ++b) tma_prefetch_4d(&tm_q, b * 64, 0, kh, r * p.W + (bt0 + h) * p.BT);
            }
        }
    }
    grid_dep_wait();     // the previous kernel of the stream has completed: inputs may be read
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int n_items;
    if constexpr (MODE == Mode::Prefill) {
        // a list the pre-pass accepted, for this call's packing (total tokens, sequences)
        const bool planned_here = p.work_hdr[3] == p.total_prompt && p.work_hdr[4] == p.R;
        n_items = (p.work_hdr[0] == 0 && planned_here) ? p.work_hdr[1] * p.n_head_groups : 0;
        if (p.work_hdr[0] == 0 && !planned_here && blockIdx.x == 0 && threadIdx.x == 0 && p.dev_status)
            atomicOr(p.dev_status, BG_DEVSTAT_PLAN);
    } else {
        n_items = p.n_items_decode;
    }

    // Register split (see AttnCfg).  setmaxnreg must be executed by all four warps of a warpgroup
    // at the same instruction, so the split is made per warpgroup before the roles branch: the
    // TMA / MMA warpgroup (warps 0-3) returns registers, the softmax warpgroups take them.
    if (warp < 4) {
    reg_dealloc<C::kRegsLight>();
    if (warp == 0) {
        // =============================================================== producer
        // The whole warp runs the loop (warp-uniform control flow and operands); lane 0
        // issues each copy.
        const uint32_t leader = (lane == 0) ? 1u : 0u;
        const uint64_t pol_q = l2_policy_evict_first();
        const uint64_t pol_kv = l2_policy_evict_last();
        TileWalker<MODE, NH> w;
        w.first(p, n_items);
        uint32_t n_kv = 0;                 // K/V tiles issued (global tile number)
        while (w.valid) {
            if (w.j == 0) {
                const int qb = w.qbuf();
                const uint32_t use = w.quse();
                if (use > 0 && !warp_wait(&q_empty[qb], (use - 1) & 1, abort_flag)) break;
                uint8_t *qdst = smem + C::kOffQ + qb * C::kQBytes;
                if constexpr (MODE == Mode::Prefill) {
                    mbar_arrive_expect_tx_w(leader, &q_full[qb], NH * C::NBQ * kQBox);
                    const int row = w.I.seq_start + w.I.qt * kRows;
#pragma unroll
                    for (int h = 0; h < NH; ++h)
#pragma unroll
                        for (int b = 0; b < C::NBQ; ++b)
                            tma_load_3d_w(leader, qdst + (h * C::NBQ + b) * kQBox, &tm_q, &q_full[qb],
                                          b * C::kQKElemsPerBlock, w.I.head0 + h, row, pol_q);
                } else {
                    const uint32_t box = static_cast<uint32_t>(p.BT * p.g * 128);
                    mbar_arrive_expect_tx_w(leader, &q_full[qb], NH * C::NB * box);
#pragma unroll
                    for (int h = 0; h < NH; ++h)
#pragma unroll
                        for (int b = 0; b < C::NB; ++b)
                            tma_load_4d_w(leader, qdst + (h * C::NB + b) * kQBox, &tm_q, &q_full[qb], b * 64, 0, w.I.kh,
                                          w.I.r * p.W + (w.I.bt0 + h) * p.BT, pol_q);
                }
            }
            const int st = n_kv % NK;
            const uint32_t use = n_kv / NK;
            if (use > 0 && !warp_wait(&k_empty[st], (use - 1) & 1, abort_flag)) break;
            uint8_t *kdst = smem + C::kOffK + st * C::kKTileBytes;
            if (MODE == Mode::Prefill || w.j < w.I.n_prompt) {
                const int row = w.I.kv_row0 + w.j * kKeys;
                mbar_arrive_expect_tx_w(leader, &k_full[st], C::kKTileBytes);
#pragma unroll
                for (int b = 0; b < C::NBQ; ++b)
                    tma_load_3d_w(leader, kdst + b * kKVBox, &tm_k, &k_full[st], b * C::kQKElemsPerBlock, w.I.kh, row,
                                  pol_kv);
            } else {
                // suffix slots 0..t-1 of suf_bpt consecutive beams: rows beam-major
                const int beam = w.I.r * p.W + w.I.bt0 * p.BT + (w.j - w.I.n_prompt) * p.suf_bpt;
                mbar_arrive_expect_tx_w(leader, &k_full[st], p.suf_tx);
#pragma unroll
                for (int b = 0; b < C::NB; ++b)
                    tma_load_4d_w(leader, kdst + b * kKVBox, &tm_sk, &k_full[st], b * 64, w.I.kh, 0, beam, pol_q);
            }
            ++n_kv;
            w.advance(p);
        }
        // Let every copy this warp started land before the CTA exits.
        if (lane == 0) {
            for (int qb = 0; qb < 2; ++qb) {
                const int uses = (w.n_q - qb + 1) / 2;
                if (uses > 0) mbar_wait_drain(&q_full[qb], (uses - 1) & 1);
            }
            for (int st = 0; st < NK; ++st) {
                const uint32_t uses = n_kv / NK + (st < static_cast<int>(n_kv % NK) ? 1u : 0u);
                if (uses > 0) mbar_wait_drain(&k_full[st], (uses - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // =============================================================== V producer
        const uint32_t leader = (lane == 0) ? 1u : 0u;
        const uint64_t pol_kv = l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_first();
        TileWalker<MODE, NH> w;
        w.first(p, n_items);
        uint32_t n_v = 0;
        while (w.valid) {
            const int st = n_v % NV;
            const uint32_t use = n_v / NV;
            if (use > 0 && !warp_wait(&v_empty[st], (use - 1) & 1, abort_flag)) break;
            uint8_t *vdst = smem + C::kOffV + st * C::kTileBytes;
            if (MODE == Mode::Prefill || w.j < w.I.n_prompt) {
                const int row = w.I.kv_row0 + w.j * kKeys;
                mbar_arrive_expect_tx_w(leader, &v_full[st], C::kTileBytes);
#pragma unroll
                for (int b = 0; b < C::NB; ++b)
                    tma_load_3d_w(leader, vdst + b * kKVBox, &tm_v, &v_full[st], b * 64, w.I.kh, row, pol_kv);
            } else {
                const int beam = w.I.r * p.W + w.I.bt0 * p.BT + (w.j - w.I.n_prompt) * p.suf_bpt;
                mbar_arrive_expect_tx_w(leader, &v_full[st], p.suf_tx);
#pragma unroll
                for (int b = 0; b < C::NB; ++b)
                    tma_load_4d_w(leader, vdst + b * kKVBox, &tm_sv, &v_full[st], b * 64, w.I.kh, 0, beam, pol_q);
            }
            ++n_v;
            w.advance(p);
        }
        if (lane == 0) {
            for (int st = 0; st < NV; ++st) {
                const uint32_t uses = n_v / NV + (st < static_cast<int>(n_v % NV) ? 1u : 0u);
                if (uses > 0) mbar_wait_drain(&v_full[st], (uses - 1) & 1);
            }
        }
        __syncwarp();
    } else {
        // =============================================================== MMA issuers (warps 1, 3)
        // One thread per query tile (lane 0 of warp 1: tile 0, of warp 3: tile 1), so the two
        // tiles' QK -> softmax -> P.V chains do not wait for each other.  The thread waits on
        // the barriers itself and issues every tcgen05.mma and commit of its tile: no
        // warp-wide broadcast of wait results and no per-instruction predicate on the issue
        // path (each costs the issuing loop tens of cycles per step).
        if (lane == 0) {
            const int h = (warp == 1) ? 0 : 1;
            constexpr uint32_t kIdescQK = QK8 ? idesc_e4m3_f32(128, kKeys) : idesc_bf16_f32(128, kKeys, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 1);
            // Base descriptors, built once; an operand at byte offset `off` from a base is the
            // base plus off / 16 (the start-address field, no carry: shared memory < 256 KB).
            const uint64_t dq0 = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(smem + C::kOffV), kKVBox, 1024);
            // `b` walks the tiles whose S is computed next, `a` (one behind) the tiles whose
            // P.V is accumulated next.
            TileWalker<MODE, NH> b, a;
            b.first(p, n_items);
            a = b;
            uint32_t gb = 0, ga = 0;           // global tile numbers of b and a
            bool ok = true;

            auto issue_qk = [&](const TileWalker<MODE, NH> &t, uint32_t g) -> bool {
                if (t.j == 0 && !mbar_wait(&q_full[t.qbuf()], t.quse() & 1, abort_flag)) return false;
                const int st = g % NK;
                if (!mbar_wait(&k_full[st], (g / NK) & 1, abort_flag)) return false;
                const uint64_t dqb = dq0 + static_cast<uint64_t>((t.qbuf() * C::kQBytes) >> 4);
                const uint64_t dks = dk0 + static_cast<uint64_t>((st * C::kKTileBytes) >> 4);
                // S(h, g%NS) holds P of tile g-NS, read by the P.V this thread issued just before
                // this QK.  tcgen05.mma operations issued by one thread execute in issue order, so
                // this QK cannot overwrite P before that P.V has read it: no wait for its completion.
                tc_fence_after();
                const uint64_t dqh = dqb + static_cast<uint64_t>((h * C::NBQ * kQBox) >> 4);
                static_assert(kQBox == 16384 && kKVBox == 8192, "mma_qk_tile hard-codes the column-block strides");
                if constexpr (QK8)
                    mma_qk_tile_e4m3(tmem + C::col_s(h, g % NS), dqh, dks, kIdescQK, &s_full[NS * h + g % NS]);
                else
                    mma_qk_tile<C::NBQ>(tmem + C::col_s(h, g % NS), dqh, dks, kIdescQK, &s_full[NS * h + g % NS]);
                // the item's Q buffer is free once its last QK has completed, unless the epilogue
                // stores the output tile out of it
                if (t.j == t.I.n_tiles - 1 && !tile_store_via_tma<MODE>(p, t.I, h))
                    mma_commit(&q_empty[t.qbuf()]);
                return true;
            };

            // QK runs NS-1 tiles ahead of P.V: QK(t + NS - 1) reuses the S buffer of P(t - 1),
            // whose P.V was issued before it.
            for (int i = 0; i < NS - 1 && ok && b.valid; ++i) {
                ok = issue_qk(b, gb);
                b.advance(p);
                ++gb;
            }
            while (ok && a.valid) {
                if (b.valid) {
                    if (!issue_qk(b, gb)) break;
                    b.advance(p);
                    ++gb;
                }
                const int st = ga % NV;
                if (!mbar_wait(&v_full[st], (ga / NV) & 1, abort_flag)) break;
                const uint64_t dvs = dv0 + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
                if (!mbar_wait(&p_full[NS * h + ga % NS], (ga / NS) & 1, abort_flag)) break;
                tc_fence_after();
                // V tile: 64 key rows of 128 bytes per column block; K = 16 rows per step.
                static_assert(kKeys == 64, "mma_pv_tile issues four 16-key steps");
                mma_pv_tile(tmem + C::kColO + D * h, tmem + C::col_s(h, ga % NS), dvs, kIdescPV, a.j > 0 ? 1u : 0u,
                            &pv_done[NS * h + ga % NS]);
                a.advance(p);
                ++ga;
            }
            // Drain: every MMA issued above completes before TMEM is released.
            mma_commit(mma_final);
            mbar_wait_drain(mma_final, 0);
        }
        __syncwarp();
    }
    } else if (warp < 4 + 4 * NH) {
        reg_alloc<C::kRegsSoftmax>();
        // =============================================================== softmax + epilogue
        const int h = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tO = tmem + lane_addr + C::kColO + D * h;
        const float sl2 = p.scale_log2;
        uint32_t g = 0;       // global tile number (same sequence as the MMA issuer)
        bool ok = true;
        int4 nxt_raw = make_int4(0, 0, 0, 0);
        if (static_cast<int>(blockIdx.x) < n_items) nxt_raw = fetch_raw<MODE>(p, blockIdx.x);
        // Epilogue of one finished item: wait for its last P.V (the commit covers all earlier
        // MMAs too), normalise O and store it.  It runs after the NEXT item's first tile has
        // been turned into P (which reads no O), so the wait for the last P.V overlaps that
        // work; the next item's first P.V, which overwrites O, is released only after this.
        // `release` runs once O is in registers: the caller lets the next P.V overwrite O from
        // then on, while the stores below still run.
        // A decode tile whose BT beams all belong to the request goes out through the TMA unit:
        // every thread writes its row into the item's Q buffer (free once the item's last QK has
        // completed, which its last P.V completing implies; same 128-byte-swizzled layout and box
        // as the Q load), and one thread issues the tile stores and, once the TMA unit has read the
        // buffer, hands it back to the Q producer.  The warps do not wait for the global writes.
        // Other tiles, and every prefill tile, are stored row by row through the staging area.
        uint32_t n_tma = 0;   // output tiles this warpgroup stored through the TMA unit so far
        // Q buffer (+1) that the group leader still has to hand back once the TMA unit has read
        // the output tile it staged there, or 0.  Handed back after the next tile's scores are
        // turned into P, or at the end of the item at the latest -- before the Q load of the item
        // after next, which waits for it.
        int q_release = 0;
        auto release_q_buffer = [&]() {
            if (q_release) {
                bulk_wait_read_all();
                mbar_arrive(&q_empty[q_release - 1]);
                q_release = 0;
            }
        };
        auto epilogue = [&](const Item &I, float m, float l, uint32_t g_last, int qbi, bool via_tma,
                            auto &&release) -> bool {
                // The commit after the item's last P.V covers every earlier MMA too.  (Items always
                // have tiles here; the test stays because ptxas allocates the prefill kernel's
                // registers with fewer spills with it: 235 vs 297 us on the Prefill-Only batch.)
                if (I.n_tiles > 0) {
                    if (!warp_wait(&pv_done[NS * h + g_last % NS], (g_last / NS) & 1, abort_flag)) return false;
                    tc_fence_after();
                }
                // destination of tile row r, or nullptr when the row is not a valid output row
                auto row_dst = [&](int r) -> __nv_bfloat16 * {
                    if constexpr (MODE == Mode::Prefill) {
                        const int qrow = I.qt * kRows + r;
                        const int head = I.head0 + h;
                        if (qrow >= I.kv_len || head - I.kh * p.g >= p.g) return nullptr;
                        return p.out + (static_cast<int64_t>(I.seq_start + qrow) * p.Hq + head) * D;
                    } else {
                        const int lb = r / p.g;
                        const int hh = r - lb * p.g;
                        const int beam = (I.bt0 + h) * p.BT + lb;
                        if (lb >= p.BT || beam >= p.W) return nullptr;
                        return p.out + ((static_cast<int64_t>(I.r) * p.W + beam) * p.Hq + I.kh * p.g + hh) * D;
                    }
                };
                // Each warp stores its 32 rows chunk by chunk: a row's 64-byte chunk goes to the warp's
                // staging area (slot c ^ ((r >> 1) & 3): conflict-free both ways), then every lane
                // stores 16 bytes of rows lane/4 + 8i, so a store instruction covers 8 whole 64-byte
                // segments.  dst[i] is this lane's destination row for pass i.
                uint8_t *stage = smem + C::kOffStage + (warp - 4) * C::kStageBytes;
                __nv_bfloat16 *dst[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = row_dst(quad * 32 + i * 8 + (lane >> 2));
                // row's 32 bf16 of chunk c (16 packed pairs) -> staging -> coalesced stores
                auto put_chunk = [&](int c, const uint32_t *wp) {
                    __syncwarp();                       // the previous chunk's reads are done
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *reinterpret_cast<uint4 *>(stage + lane * 64 + ((u ^ ((lane >> 1) & 3)) * 16)) =
                            make_uint4(wp[4 * u], wp[4 * u + 1], wp[4 * u + 2], wp[4 * u + 3]);
                    __syncwarp();
                    const int cc = lane & 3;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = i * 8 + (lane >> 2);
                        const uint4 val = *reinterpret_cast<const uint4 *>(stage + rr * 64 + ((cc ^ ((rr >> 1) & 3)) * 16));
                        if (dst[i]) __stcs(reinterpret_cast<uint4 *>(dst[i] + 32 * c) + cc, val);   // streamed: never re-read
                    }
                };
                // O is read 64 columns at a time, normalised and packed to bf16 pairs (half the
                // registers), and handed back to the next item's P.V before the stores
                const float inv_l = 1.f / l;
                const float2 il = make_float2(inv_l, inv_l);
                uint32_t pk[D / 2];
#pragma unroll
                for (int c2 = 0; c2 < D / 64; ++c2) {
                    float o[64];
                    tmem_ld64(tO + 64 * c2, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 x = fmul2(make_float2(o[2 * i], o[2 * i + 1]), il);
                        pk[32 * c2 + i] = pack_bf16x2(x.x, x.y);
                    }
                }
                release();
                const bool leader = quad == 0 && lane == 0;
                if (MODE == Mode::Decode && via_tma) {
                    // row `row` of column block cb: 16-byte chunk c at (c ^ (row % 8)) in its 128-byte row
                    uint8_t *tile = smem + C::kOffQ + qbi * C::kQBytes + h * C::NB * kQBox;
#pragma unroll
                    for (int cb = 0; cb < C::NB; ++cb)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(tile + cb * kQBox + row * 128 + ((c ^ (row & 7)) << 4)) =
                                make_uint4(pk[32 * cb + 4 * c], pk[32 * cb + 4 * c + 1], pk[32 * cb + 4 * c + 2],
                                           pk[32 * cb + 4 * c + 3]);
                    fence_proxy_async_smem();          // generic-proxy writes -> the TMA unit's reads
                    __syncwarp();
                    uint64_t *staged = &o_staged[2 * h + (n_tma & 1)];
                    if (lane == 0) mbar_arrive(staged);
                    const uint32_t staged_parity = (n_tma >> 1) & 1u;
                    ++n_tma;
                    if (leader) {
                        // a bounded wait (not a named barrier): if another warp of the group has
                        // given up, this one gives up too instead of waiting forever
                        if (!mbar_wait(staged, staged_parity, abort_flag)) return false;
#pragma unroll
                        for (int cb = 0; cb < C::NB; ++cb) {
                            if constexpr (MODE == Mode::Prefill)
                                tma_store_3d(&tm_o, tile + cb * kQBox, cb * 64, I.head0 + h, I.seq_start + I.qt * kRows);
                            else
                                tma_store_4d(&tm_o, tile + cb * kQBox, cb * 64, 0, I.kh, I.r * p.W + (I.bt0 + h) * p.BT);
                        }
                        bulk_commit_group();
                        // the Q buffer goes back to its producer once the TMA unit has read the
                        // tile out of it; that wait happens later (release_q_buffer), so that this
                        // thread's softmax work does not wait for it
                        q_release = qbi + 1;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) put_chunk(c, pk + 16 * c);
                }
                if constexpr (MODE == Mode::Prefill) {
                    if (p.lse) {
                        if (row_dst(row)) {
                            // natural-log sum-exp: (m + log2 l) * ln 2
                            p.lse[static_cast<int64_t>(I.seq_start + I.qt * kRows + row) * p.Hq + I.head0 + h] =
                                (m + __log2f(l)) * 0.69314718055994530942f;
                        }
                    }
                }
            return true;
        };
        bool pend = false;    // an item whose epilogue still has to run
        Item Ip;
        float mp = 0.f, lp = 0.f;
        uint32_t gp = 0;
        int nq = 0, qbp = 0;  // items with tiles entered so far (selects the Q buffer, as in TileWalker)
        bool tmap = false;    // the pending item's tile leaves through the TMA unit
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const int4 raw = nxt_raw;
            if (it + static_cast<int>(gridDim.x) < n_items) nxt_raw = fetch_raw<MODE>(p, it + gridDim.x);
            const Item I = make_item<MODE, NH>(p, it, raw);
            if (!I.valid) {
                if constexpr (MODE == Mode::Decode) {
                    if (h == 0 && row == 0 && p.dev_status) {
                        const int a = raw.x, b = raw.y;
                        const bool bad_cu =
                            !(a >= 0 && b >= a && b <= p.total_prompt && (b - a) <= p.max_prompt_len);
                        atomicOr(p.dev_status, bad_cu ? BG_DEVSTAT_CU_PROMPT : BG_DEVSTAT_EMPTY_ROW);
                    }
                }
                continue;
            }
            if (I.n_tiles == 0) continue;   // not produced by make_item for a valid item; skipped by every role
            ++nq;
            const bool tma_I = tile_store_via_tma<MODE>(p, I, h);
            float m = -INFINITY;   // running max of scaled logits (base-2 units)
            float l = 0.f;         // running sum of exp2(logit - m)
            for (int j = 0; j < I.n_tiles; ++j, ++g) {
                const uint32_t tS = tmem + lane_addr + C::col_s(h, g % NS);
                // valid key columns of this tile: c < lim for this row (lim_lo..lim_hi over the
                // warp's rows); a decode suffix tile keeps c in [c0, c0 + nsuf) instead
                int lim, lim_lo, lim_hi;
                bool suf = false;
                int c0 = 0, nsuf = 0;
                if constexpr (MODE == Mode::Prefill) {
                    lim_lo = I.qt * kRows + quad * 32 - j * kKeys + 1;
                    lim = lim_lo + lane;
                    lim_hi = lim_lo + 31;
                } else {
                    lim_lo = I.kv_len - j * kKeys;
                    lim = lim_lo;
                    lim_hi = lim_lo;
                    if (j >= I.n_prompt) {
                        // this row's beam, counted from the item's first beam, and its place in the tile
                        suf = true;
                        const int lb = row / p.g;
                        const int pos = h * p.BT + lb - (j - I.n_prompt) * p.suf_bpt;
                        const bool mine = lb < p.BT && (I.bt0 + h) * p.BT + lb < p.W && pos >= 0 && pos < p.suf_bpt;
                        c0 = pos * p.suffix_len;
                        nsuf = mine ? p.suffix_len : 0;
                        lim_hi = __any_sync(0xffffffffu, nsuf > 0) ? 1 : 0;
                    }
                }
                if (!warp_wait(&s_full[NS * h + g % NS], (g / NS) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                // this tile's QK has completed: its K stage can be reloaded (one arrive per warpgroup)
                // ... and so has every MMA its warp issued before that QK, which includes the P.V of
                // tile g - NS: that V stage can be reloaded too
                if (quad == 0 && lane == 0) {
                    mbar_arrive(&k_empty[g % NK]);
                    if (g >= NS) mbar_arrive(&v_empty[(g - NS) % NV]);
                }
                if (lim_hi <= 0) {
                    // every row of this warp is masked for this tile: P = 0
                    uint32_t zr[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) zr[i] = 0u;
                    tmem_st16(tS, zr);
                    tmem_st16(tS + 16, zr);
                } else {
                    float s[kKeys];
                    static_assert(kKeys == 64, "one tmem_ld64 per S tile");
                    tmem_ld64(tS, s);
                    if (suf) {
#pragma unroll
                        for (int c = 0; c < kKeys; ++c)
                            if (static_cast<unsigned>(c - c0) >= static_cast<unsigned>(nsuf)) s[c] = -INFINITY;
                    } else if (lim_lo < kKeys) {
#pragma unroll
                        for (int c = 0; c < kKeys; ++c)
                            if (c >= lim) s[c] = -INFINITY;
                    }
                    // row max: four independent 3-input-max chains (short dependency chains)
                    float mq[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) mq[q] = fmaxf(s[16 * q], s[16 * q + 1]);
#pragma unroll
                    for (int c = 2; c < 16; c += 2)
#pragma unroll
                        for (int q = 0; q < 4; ++q) mq[q] = fmax3f(mq[q], s[16 * q + c], s[16 * q + c + 1]);
                    const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                    const float m_new = fmaxf(m, mx * sl2);
                    const bool grow = (j > 0) && (m_new > m + kRescaleLog2);
                    if (j == 0) m = m_new;
                    if (__any_sync(0xffffffffu, grow)) {
                        // O holds the previous tiles: wait for their last P.V, rescale in place.
                        if (!warp_wait(&pv_done[NS * h + (g - 1) % NS], ((g - 1) / NS) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // decode: a row with no valid key so far has O = 0 and l = 0 (alpha 0, not
                        // the NaN of -inf - -inf when its max is still -inf)
                        const float alpha = (MODE == Mode::Decode && m == -INFINITY) ? 0.f : ex2(m - m_new);
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
                    }
                    // p = 2^(s * scale * log2e - m), two columns per packed FMA; row sum in four
                    // independent pair accumulators.
                    float2 rs[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) rs[q] = make_float2(0.f, 0.f);
                    const float2 sl2x2 = make_float2(sl2, sl2);
                    // decode: a row that has seen no valid key yet (max -inf) gets p = 0, not NaN;
                    // a prefill row always has key 0 in its first tile
                    const float mu = (MODE == Mode::Decode && m == -INFINITY) ? 0.f : m;
                    const float2 negm = make_float2(-mu, -mu);
                    // P.V multiplies the bf16-rounded weights.  The row's largest weight is the
                    // largest of its tile, and under the lazy rescale it can be anything up to 2^8,
                    // so its rounding (up to 2^-9 of it) would scale the whole output row; the sum
                    // takes that weight rounded as P.V sees it, which makes the dominant term of
                    // O / l exact.  The other weights' roundings are smaller and partly cancel.
                    const float pmax = ex2(ffma2(make_float2(mx, mx), sl2x2, negm).x);
                    const float pmax_fix = __uint_as_float(pack_bf16x2(pmax, 0.f) << 16) - pmax;
#pragma unroll
                    for (int c = 0; c < kKeys / 32; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 x = ffma2(make_float2(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), sl2x2, negm);
                            const float2 e = make_float2(ex2(x.x), ex2(x.y));
                            rs[i & 3] = fadd2(rs[i & 3], e);
                            pk[i] = pack_bf16x2(e.x, e.y);
                        }
                        tmem_st16(tS + 16 * c, pk);   // P (bf16 pairs) over the first 32 columns of S
                    }
                    const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
                    l += ((r01.x + r23.x) + (r01.y + r23.y)) + pmax_fix;
                }
                tmem_st_wait();
                tc_fence_before();
                if (j == 0 && pend) {
                    // the previous item's O is read before this tile's P.V may overwrite it
                    if (!epilogue(Ip, mp, lp, gp, qbp, tmap, [&]() {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&p_full[NS * h + g % NS]);
                        })) {
                        ok = false;
                        break;
                    }
                    pend = false;
                } else {
                    // one arrive per warp: every lane's P stores are complete (wait::st) and
                    // fenced (fence::before_thread_sync) before the warp synchronises, and the
                    // arrive releases them to the MMA thread (32 arrives on one barrier from one
                    // warp would be serialised, about 600 cycles per tile on this critical path)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[NS * h + g % NS]);
                    if (quad == 0 && lane == 0) release_q_buffer();
                }
            }
            if (quad == 0 && lane == 0) release_q_buffer();   // an item of one tile
            if (!ok) break;
            pend = true;
            qbp = (nq - 1) & 1;
            tmap = tma_I;
            Ip = I;
            mp = m;
            lp = l;
            gp = g - 1;
        }
        if (ok && pend) ok = epilogue(Ip, mp, lp, gp, qbp, tmap, []() {});
        // every tile store this thread issued has written global memory before the CTA exits
        if (quad == 0 && lane == 0) {
            release_q_buffer();
            bulk_wait_all();
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
