// fwd_bf16_pair.cu -- bf16 attention forward for D = 128 (D = 64 runs the
// variant in fwd_bf16_duo.cu, with an issuer and a P buffer per tile): each CTA owns a
// pair of 128-row query tiles of one (batch, head) and streams 128-key K/V
// tiles past both.  Same algorithm as fwd_bf16.cu ("Learning Metal with
// FlashAttention", section "FlashAttention"; metalworking "Flash Attention",
// kernel anatomy items 1-5; metal-flash-attention forward pseudocode): Q tiles
// resident, S = Q K^T in TMEM, online base-2 softmax with running max m and
// sum l, O += P V in TMEM, O / l and L = m + ln(l) written once; causal tiles
// above the diagonal are never loaded.
//
// GB300 mapping (why a pair): one softmax warpgroup owns each query tile, so a
// thread owns a whole row (its TMEM lane) and the row max / sum are
// thread-local -- no exchange between warps -- and the tensor core works on
// one tile's S or PV while the other tile's softmax runs.
//   warp 0      TMA producer: per block Q_A, Q_B, and K_j, V_j (128 rows) into a ring
//   warp 1      TMEM allocator + the one tcgen05 issuer, in the fixed order
//                 S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//   warps 2-5   softmax of tile A; warps 6-9 softmax of tile B
// TMEM (512 columns): S_A, S_B (128 fp32 columns each), O_A, O_B (D columns
// each).  128-key tiles keep the S MMA at N = 128, where it runs at the full
// tensor rate (at N = 64 it is shared-memory-bound).  P_X(j) is written as
// bf16 pairs over the first 64 columns of S_X(j), which the softmax has
// already read, so S_X(j+1) is issued only after PV_X(j) has completed
// (pv_done).  The O correction is lazy (only when the running max grows by
// more than 2^8).
// Ordering: MMAs on different accumulators are not ordered with each other
// and a commit tracks only its own thread's MMAs, so every reuse is explicit:
// S_X(j+1) is issued after pv_done_X(j), which also orders the softmax's O
// rescale of step j+1 after PV_X(j); the epilogue reads O_X after the block's
// last pv_done_X, and the next block's first PV_X waits until it has (o_free).
// Persistent grid: one CTA per SM walks a sequence of blocks (persistent_work_index),
// so a block's Q load and first S products overlap the previous block's last
// products and epilogue instead of a CTA exit, launch and pipeline fill
// (measured +10 % at B=2 H=16 N=4096 D=128 causal, +5 % at N=32768 D=64).
// Every role computes the CTA's blocks itself (the static deal), so the
// causal order here is the plain rank order over all heads: blocks drawn from
// a counter and handed to the issuer warp through shared memory (sched.cuh,
// as the D = 64 kernel does) measured 10-15 % slower at D = 128, however the
// hand-over was written.
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBM = 128;            // rows per query tile (TMEM lanes)
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kTiles = 2;           // query tiles per CTA
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kThreads = 32 * kFirstSoftmaxWarp + 128 * kTiles;

enum : int { kSiteQ = 61, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePFull, kSitePV, kSiteFinal, kSiteDrain,
             kSiteQEmpty, kSiteOFree, kSiteStage };

template <int D, int NSLOT>
struct PairSmem {
    static constexpr int kPanels = D / 64;
    static constexpr int kQBytes = kBM * D * 2;    // one query tile
    static constexpr int kSlotBytes = kBN * D * 2;  // one K or V tile
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = kTiles * kQBytes;
    static constexpr int kStageOff = kSlotOff + NSLOT * kSlotBytes;  // one query tile's O, staged for TMA stores
    static constexpr int kBarOff = kStageOff + kQBytes;
    // q_full, q_empty, slot_full[NSLOT], slot_empty[NSLOT], per tile: s_full, p_full, pv_done, o_free,
    // stage_full; final, stage_free
    static constexpr int kNumBars = 2 + 2 * NSLOT + 5 * kTiles + 2;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

// The work of one block of this CTA: which query rows, and how many K/V tiles each of its two query
// tiles reads.  Every role of the CTA walks the same sequence of blocks and computes these alike.
struct PairBlock {
    int bh, row0, n_kv0, n_kv1, n_all, n_q_tiles;
};

__device__ __forceinline__ PairBlock pair_block(const FwdArgs &a, int L, int n_blk) {
    PairBlock w;
    int rank;
    tile_order_at(L, n_blk, a.B * a.H, a.causal, a.head_group, &rank, &w.bh);
    const int blk = n_blk - 1 - rank;  // causal: the last block has the most keys
    w.row0 = blk * (kTiles * kBM);
    auto tiles_of = [&](int x) -> int {
        const int r0 = w.row0 + x * kBM;
        const int kv_end = a.causal ? min(a.N, r0 + kBM) : a.N;
        return r0 < a.N ? (kv_end + kBN - 1) / kBN : 0;
    };
    w.n_kv0 = tiles_of(0);
    w.n_kv1 = tiles_of(1);
    w.n_all = max(w.n_kv0, w.n_kv1);  // >= 1
    w.n_q_tiles = (w.row0 + kBM < a.N) ? kTiles : 1;  // a query tile wholly past N is not loaded
    return w;
}

// Persistent: the grid has at most one CTA per SM, each walking its blocks in turn, so the next block's
// Q load and first S products overlap the previous block's last products and epilogue.  The K/V ring
// and every barrier's phase run on across blocks.
template <int D, int NSLOT>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                         FwdArgs a) {
    using L = PairSmem<D, NSLOT>;
    constexpr int kPanels = L::kPanels;
    constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S_A, S_B (P_X over the first kBN/2 columns of S_X), then O_A, O_B
    constexpr uint32_t kColS = 0, kColO = kTiles * kBN;
    static_assert(kColO + kTiles * D <= kTmemCols, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem + L::kQOff;
    uint8_t *slots = smem + L::kSlotOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;                // block b's Q tiles landed (phase b)
    uint64_t *q_empty = bars + 1;           // every S MMA of block b has completed (phase b)
    uint64_t *slot_full = bars + 2;
    uint64_t *slot_empty = slot_full + NSLOT;
    uint64_t *s_full = slot_empty + NSLOT;  // [tile]: S_X of step g complete (phase g, steps counted across blocks)
    uint64_t *p_full = s_full + kTiles;     // [tile]: P_X of step g written (and O_X corrected)
    uint64_t *pv_done = p_full + kTiles;    // [tile]: PV_X of step g complete
    uint64_t *o_free = pv_done + kTiles;    // [tile]: the epilogue has read O_X (phase = X's blocks with work)
    uint64_t *final_bar = o_free + kTiles;  // every MMA of the CTA has completed
    // The epilogue of a query tile writes O into the one staging buffer and stores it by TMA.  Within a
    // block tile A uses the buffer before tile B, so every role can count the uses from the blocks:
    uint64_t *stage_full = final_bar + 1;      // [tile]: the tile's four warps have written the buffer
    uint64_t *stage_free = stage_full + kTiles;  // the last store has finished reading it (phase = use)
    uint8_t *stage = smem + L::kStageOff;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_blk = (a.N + kTiles * kBM - 1) / (kTiles * kBM);
    const int n_work = n_blk * a.B * a.H;
    const int N = a.N;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int x = 0; x < kTiles; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);  // one arrive per softmax warp of tile x
            mbar_init(&pv_done[x], 1);
            mbar_init(&o_free[x], 4);
        }
        mbar_init(final_bar, 1);
        for (int x = 0; x < kTiles; ++x) mbar_init(&stage_full[x], 4);
        mbar_init(stage_free, 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            int last_round[NSLOT];
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) last_round[s] = -1;
            int gidx = 0;  // K/V loads so far (ring position)
            int nb = 0;    // blocks so far
            bool ok = true;
            for (int k = 0; ok && k * (int)gridDim.x < n_work; ++k) {
                const int Lw = persistent_work_index(k, n_work);
                if (Lw < 0) continue;
                const PairBlock w = pair_block(a, Lw, n_blk);
                // Q of this block goes after its first K and V tiles: its buffer frees only when the
                // previous block's last S products complete, and K_0 / V_0 need not wait for that
                const int q_at = nb == 0 ? 0 : 2;
                for (int idx = 0; ok && idx <= 2 * w.n_all; ++idx) {
                    if (idx == q_at) {
                        if (nb > 0 && !(ok = mbar_wait(q_empty, (nb - 1) & 1, a.status, kSiteQEmpty))) break;
                        mbar_arrive_expect_tx(q_full, w.n_q_tiles * L::kQBytes);
                        for (int x = 0; x < w.n_q_tiles; ++x)
#pragma unroll
                            for (int p = 0; p < kPanels; ++p)
                                tma_load_3d(q_s + x * L::kQBytes + p * (kBM * 128), &tmap_q, q_full, p * 64,
                                            w.row0 + x * kBM, w.bh);
                    }
                    if (idx == 2 * w.n_all) break;
                    const int g = gidx + idx;
                    const int slot = g % NSLOT, round = g / NSLOT;
                    if (!(ok = mbar_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty))) break;
                    uint8_t *dst = slots + slot * L::kSlotBytes;
                    const CUtensorMap *map = (idx & 1) ? &tmap_v : &tmap_k;
                    mbar_arrive_expect_tx(&slot_full[slot], L::kSlotBytes);
#pragma unroll
                    for (int p = 0; p < kPanels; ++p)
                        tma_load_3d(dst + p * (kBN * 128), map, &slot_full[slot], p * 64, (idx >> 1) * kBN, w.bh);
#pragma unroll
                    for (int s = 0; s < NSLOT; ++s)
                        if (s == slot) last_round[s] = round;
                }
                gidx += 2 * w.n_all;
                ++nb;
            }
            // Drain: never leave the CTA with a TMA write still in flight.
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            if (nb > 0) mbar_wait(q_full, (nb - 1) & 1, a.status, kSiteDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ the tcgen05 issuer
        // The whole warp runs the loop (operands stay warp-uniform); one elected lane issues the MMAs
        // and the commits that track them.  Per block the order is
        //   S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, false, true);
        const uint64_t q_desc = sdesc_sw128(smem_u32(q_s), 16, 1024);
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = true;
        int gidx = 0;                 // ring position of this block's K_0
        int step0[kTiles] = {0, 0};   // steps of tile x before this block
        int blocks[kTiles] = {0, 0};  // earlier blocks in which tile x had work (epilogues)
        int nb = 0;
        for (int k = 0; ok && k * (int)gridDim.x < n_work; ++k) {
            const int Lw = persistent_work_index(k, n_work);
            if (Lw < 0) continue;
            const PairBlock w = pair_block(a, Lw, n_blk);
            const int n_kv[kTiles] = {w.n_kv0, w.n_kv1};
            if (!(ok = warp_wait(q_full, nb & 1, a.status, kSiteQ))) break;
            tc_fence_after();
            // S_X(j) = Q_X K_j^T into S_X
            auto issue_s = [&](int x, int j) {
                if (!ok || j >= n_kv[x]) return;
                const int g = gidx + 2 * j;
                const int slot = g % NSLOT;
                if (!(ok = warp_wait(&slot_full[slot], (g / NSLOT) & 1, a.status, kSiteSlotFull))) return;
                // S_X overwrites P_X of the step before (this block's or the previous one's)
                const int st = step0[x] + j;
                if (st >= 1 && !(ok = warp_wait(&pv_done[x], (st - 1) & 1, a.status, kSitePV))) return;
                tc_fence_after();
                const uint64_t k_desc = sdesc_sw128(slot_addr + slot * L::kSlotBytes, 16, 1024);
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * (kBM * 128) + (ks & 3) * 32;
                        mma_ss(tmem + kColS + x * kBN, sdesc_add(q_desc, x * L::kQBytes + off),
                               sdesc_add(k_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32), idesc_s, ks > 0);
                    }
                    mma_commit(&s_full[x]);
                }
                __syncwarp();
            };
            // O_X += P_X(j) V_j, P_X from TMEM
            auto issue_pv = [&](int x, int j) {
                if (!ok || j >= n_kv[x]) return;
                const int g = gidx + 2 * j + 1;
                const int slot = g % NSLOT;
                if (!(ok = warp_wait(&slot_full[slot], (g / NSLOT) & 1, a.status, kSiteSlotFull))) return;
                if (!(ok = warp_wait(&p_full[x], (step0[x] + j) & 1, a.status, kSitePFull))) return;
                // the first PV of a block overwrites O_X, which the previous block's epilogue reads
                if (j == 0 && blocks[x] >= 1 && !(ok = warp_wait(&o_free[x], (blocks[x] - 1) & 1, a.status, kSiteOFree)))
                    return;
                tc_fence_after();
                const uint64_t v_desc = sdesc_sw128(slot_addr + slot * L::kSlotBytes, kBN * 128, 1024);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_ts(tmem + kColO + x * D, tmem + kColS + x * kBN + kk * 8, sdesc_add(v_desc, kk * 2048),
                               idesc_o, (j > 0 || kk > 0));
                    mma_commit(&pv_done[x]);
                }
                __syncwarp();
            };
            // a slot is released by a commit after the last MMA that reads it (a commit tracks every
            // earlier MMA of this thread); the same goes for the Q buffer after the block's last S
            auto commit_to = [&](uint64_t *bar) {
                if (leader) mma_commit(bar);
                __syncwarp();
            };
            issue_s(0, 0);
            issue_s(1, 0);
            if (ok && w.n_all == 1) commit_to(q_empty);
            if (ok) commit_to(&slot_empty[gidx % NSLOT]);  // K_0
            for (int j = 0; ok && j < w.n_all; ++j) {
                issue_pv(0, j);
                issue_s(0, j + 1);
                issue_pv(1, j);
                if (ok) commit_to(&slot_empty[(gidx + 2 * j + 1) % NSLOT]);  // V_j
                issue_s(1, j + 1);
                if (ok && j + 2 == w.n_all) commit_to(q_empty);  // the block's last S products
                if (ok && j + 1 < w.n_all) commit_to(&slot_empty[(gidx + 2 * j + 2) % NSLOT]);  // K_{j+1}
            }
#pragma unroll
            for (int x = 0; x < kTiles; ++x) {
                step0[x] += n_kv[x];
                blocks[x] += n_kv[x] > 0;
            }
            gidx += 2 * w.n_all;
            ++nb;
        }
        // every MMA complete: TMEM may be released
        if (leader) mma_commit(final_bar);
        __syncwarp();
        warp_wait(final_bar, 0, a.status, kSiteFinal);
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int x = (warp - kFirstSoftmaxWarp) >> 2;  // query tile of this warpgroup
        const int quarter = warp & 3;                   // TMEM lanes [32*quarter, 32*quarter + 32)
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_col = kColS + x * kBN, o_col = kColO + x * D;
        const float c = a.scale_log2;
        bool ok = true;
        int step0 = 0;     // steps of this tile before the current block
        int uses = 0;      // uses of the staging buffer (by both tiles) before the current block
        int blocks_x = 0;  // epilogues of this tile so far (phase of stage_full[x])
        for (int k = 0; ok && k * (int)gridDim.x < n_work; ++k) {
            const int Lw = persistent_work_index(k, n_work);
            if (Lw < 0) continue;
            const PairBlock w = pair_block(a, Lw, n_blk);
            const int n = x == 0 ? w.n_kv0 : w.n_kv1;
            const int tile_row0 = w.row0 + x * kBM;
            const int row = tile_row0 + r;
            float m = -INFINITY, l = 0.f;  // running max (log2 units) and sum
            for (int j = 0; j < n; ++j) {
                // S_X(j) was issued after PV_X(j-1) completed, so O_X and the P columns are free as well
                ok = mbar_wait(&s_full[x], (step0 + j) & 1, a.status, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t raw[kBN];
#pragma unroll
                for (int ch = 0; ch < kBN / 32; ++ch) tmem_ld32(tmem + lane_base + s_col + ch * 32, raw + ch * 32);
                tmem_wait_ld();
                const int key0 = j * kBN;
                const bool need_mask = (key0 + kBN > N) || (a.causal && key0 + kBN - 1 > tile_row0);
                if (need_mask) {
                    const int lim = a.causal ? min(N - 1, row) : N - 1;  // last visible key
#pragma unroll
                    for (int i = 0; i < kBN; ++i)
                        if (key0 + i > lim) raw[i] = 0xff800000u;  // -inf
                }
                // row max of the raw scores (scale > 0 commutes with max): four chains of three-input maxima
                float mx[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) mx[u] = __uint_as_float(raw[u]);
#pragma unroll
                for (int i = 4; i + 8 <= kBN; i += 8)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        mx[u] = fmax3(mx[u], __uint_as_float(raw[i + 2 * u]), __uint_as_float(raw[i + 2 * u + 1]));
#pragma unroll
                for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], __uint_as_float(raw[kBN - 4 + u]));
                const float mt = c * fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
                const float m_new = fmaxf(m, mt);
                // Lazy correction: keep the stale max unless the row max grew by > 8 (factor 256).
                const bool need = m_new > m + 8.f;
                const float m_use = need ? m_new : m;
                const float m_base = (m_use == -INFINITY) ? 0.f : m_use;
                const float alpha = need ? ex2_approx(m - m_base) : 1.f;
                // P = 2^(s c - m) as bf16 pairs over the first kBN/2 columns of S_X, 16 columns per store;
                // the scaling FMA and the row sum run on fp32 pairs
                const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_base, -m_base);
                uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                for (int h = 0; h < kBN / 32; ++h) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint64_t y2 = f2_fma(f2_pack(__uint_as_float(raw[32 * h + 2 * i]),
                                                           __uint_as_float(raw[32 * h + 2 * i + 1])), c2, nm2);
                        float y0, y1;
                        f2_unpack(y2, y0, y1);
                        const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                        acc2[i & 1] = f2_add(acc2[i & 1], f2_pack(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tmem + lane_base + s_col + h * 16, pk);
                }
                float r0, r1, r2, r3;
                f2_unpack(acc2[0], r0, r1);
                f2_unpack(acc2[1], r2, r3);
                l = l * alpha + ((r0 + r1) + (r2 + r3));
                m = m_use;
                if (j >= 1 && __any_sync(0xffffffffu, need)) {
                    uint32_t ov[32];
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        tmem_ld32(tmem + lane_base + o_col + ch * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(tmem + lane_base + o_col + ch * 32, ov);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                warp_arrive(&p_full[x]);
            }
            // the staging buffer's use number of this tile's epilogue in this block (tile A's before tile B's)
            const int use = uses + (x == 1 && w.n_kv0 > 0);
            uses += (w.n_kv0 > 0) + (w.n_kv1 > 0);
            if (!ok || n == 0) continue;
            // the block's last PV_X has completed: O_X is final
            step0 += n;
            ok = mbar_wait(&pv_done[x], (step0 - 1) & 1, a.status, kSiteFinal);
            // the previous use's TMA store has finished reading the staging buffer
            if (ok && use >= 1) ok = mbar_wait(stage_free, (use - 1) & 1, a.status, kSiteStage);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const float inv_l = 1.f / l;
            // O / l as bf16 into the staging buffer: 128-byte-swizzled panels of 64 columns, row r of panel
            // p at p * 16 KB + r * 128, its 16-byte chunk k at k ^ (r % 8) (conflict-free across the lanes)
            uint32_t ov[32];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                tmem_ld32(tmem + lane_base + o_col + ch * 32, ov);
                tmem_wait_ld();
                if (ch == D / 32 - 1) {
                    // every read of O_X is done: the next block's first PV_X may overwrite it
                    tc_fence_before();
                    warp_arrive(&o_free[x]);
                }
                uint8_t *prow = stage + (ch >> 1) * (kBM * 128) + r * 128;
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    st_shared_v4(prow + ((((ch & 1) * 4 + v4) ^ (r & 7)) << 4),
                                 pack_bf16x2(__uint_as_float(ov[v4 * 8 + 0]) * inv_l, __uint_as_float(ov[v4 * 8 + 1]) * inv_l),
                                 pack_bf16x2(__uint_as_float(ov[v4 * 8 + 2]) * inv_l, __uint_as_float(ov[v4 * 8 + 3]) * inv_l),
                                 pack_bf16x2(__uint_as_float(ov[v4 * 8 + 4]) * inv_l, __uint_as_float(ov[v4 * 8 + 5]) * inv_l),
                                 pack_bf16x2(__uint_as_float(ov[v4 * 8 + 6]) * inv_l, __uint_as_float(ov[v4 * 8 + 7]) * inv_l));
            }
            fence_proxy_async_smem();  // the staged tile is read by the TMA (async proxy)
            warp_arrive(&stage_full[x]);
            if (row < N) a.lse[(size_t)w.bh * N + row] = (m + __log2f(l)) * 0.69314718055994531f;
            if (quarter == kFirstSoftmaxWarp % 4 && lane == 0) {
                // one thread of the tile stores the staged panels (rows past N and columns past the caller's
                // D are clipped by the tensor map) and frees the buffer once the stores have read it
                if (mbar_wait(&stage_full[x], blocks_x & 1, a.status, kSiteStage)) {
#pragma unroll
                    for (int p = 0; p < kPanels; ++p)
                        if (p * 64 < a.D) tma_store_3d(&tmap_o, stage + p * (kBM * 128), p * 64, tile_row0, w.bh);
                    tma_store_commit();
                    tma_store_wait_read();
                    mbar_arrive(stage_free);
                } else {
                    ok = false;
                }
            }
            ++blocks_x;
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int NSLOT>
cudaError_t launch_spec(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &to, cudaStream_t s) {
    using L = PairSmem<D, NSLOT>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    auto kern = fwd_bf16_pair_kernel<D, NSLOT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    const int n_work = ((a.N + kTiles * kBM - 1) / (kTiles * kBM)) * a.H * a.B;
    const int sms = a.num_sms > 0 ? a.num_sms : kNumSms;
    dim3 grid(n_work < sms ? n_work : sms);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, to, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16_pair(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t s) {
    switch (kernel_head_dim(a.D)) {
        case 128: return launch_spec<128, fwd_nslot(128)>(a, tq, tk, tv, to, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
