// fwd_bf16_duo.cu -- bf16 attention forward for D = 64: the two-tile
// persistent kernel of fwd_bf16_pair.cu with ONE tcgen05 ISSUER WARP PER QUERY
// TILE and a P buffer of its own per tile.  Same algorithm
// ("Learning Metal with FlashAttention", section "FlashAttention";
// metalworking "Flash Attention", kernel anatomy items 1-5; metal-flash-
// attention forward pseudocode).
//
// With one issuer for both tiles, a wait on one tile's product (S_X(j+1) may
// only overwrite S_X once PV_X(j), which reads P_X from it, has completed)
// also holds back the other tile's ready products.  Here each tile's issuer
// waits only for its own tile.  At D = 64 the 512 TMEM columns hold S_A, S_B
// (128 each), O_A, O_B (64 each) and P_A, P_B (64 each): S_X(j+1) is then
// issued as soon as the softmax has loaded S_X(j) (s_free), before P_X(j) is
// even written, and the softmax writes P_X(j+1) once PV_X(j) has completed.
// Measured at B=1 H=32 N=32768 causal: 4.49 -> 4.17 ms against fwd_bf16_pair.cu.
// (At D = 128 there is no room for P buffers; two issuers with P over S
// measured 12-15 % slower than the pair kernel's single issuer, which keeps
// D = 128.)
//   warp 0      TMA producer (as in fwd_bf16_pair.cu)
//   warp 1      TMEM allocator + issuer of tile A; warp 2 issuer of tile B
//   warps 3-6   softmax of tile A; warps 7-10 softmax of tile B
// A K/V slot and the Q buffer are released when BOTH issuers have committed
// after their last product that reads them (barriers of count 2); in a causal
// block tile A has one K/V tile fewer and just commits for the last one.
#include "fa_internal.h"
#include "sched.cuh"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBM = 128;            // rows per query tile (TMEM lanes)
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kTiles = 2;           // query tiles per CTA
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kThreads = 32 * kFirstSoftmaxWarp + 128 * kTiles;

enum : int { kSiteQ = 161, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePFull, kSitePV, kSiteFinal, kSiteDrain,
             kSiteQEmpty, kSiteOFree, kSiteSFree, kSiteWork };

template <int D, int NSLOT>
struct DuoSmem {
    static constexpr int kPanels = D / 64;
    static constexpr int kQBytes = kBM * D * 2;    // one query tile
    static constexpr int kSlotBytes = kBN * D * 2;  // one K or V tile
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = kTiles * kQBytes;
    static constexpr int kBarOff = kSlotOff + NSLOT * kSlotBytes;
    // q_full, q_empty, slot_full[NSLOT], slot_empty[NSLOT], per tile: s_full, p_full, pv_done, o_free, s_free,
    // final; the work ring's full[kWorkRing], empty[kWorkRing]
    static constexpr int kNumBars = 2 + 2 * NSLOT + 5 * kTiles + kTiles + 2 * kWorkRing;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kWorkOff = kTmemHolderOff + 16;  // the work ring's items
    static constexpr int kAlloc = kWorkOff + 4 * kWorkRing + 1024;
};

// The work of one block of this CTA: which query rows, and how many K/V tiles each of its two query
// tiles reads.  Every role of the CTA walks the same sequence of blocks (the work ring) and computes
// these alike.
struct DuoBlock {
    int bh, row0, n_kv0, n_kv1, n_all, n_q_tiles;
};

__device__ __forceinline__ DuoBlock duo_block(const FwdArgs &a, int L, int n_blk) {
    DuoBlock w;
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
    fwd_bf16_duo_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, FwdArgs a) {
    using L = DuoSmem<D, NSLOT>;
    constexpr int kPanels = L::kPanels;
    constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S_A, S_B, then O_A, O_B, then P_A, P_B (128 keys of bf16 pairs each)
    constexpr uint32_t kColS = 0, kColO = kTiles * kBN, kColP = kColO + kTiles * D;
    static_assert(kColP + kTiles * kBN / 2 <= kTmemCols, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem + L::kQOff;
    uint8_t *slots = smem + L::kSlotOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;                // block b's Q tiles landed (phase b)
    uint64_t *q_empty = bars + 1;           // both issuers' S MMAs of block b have completed (phase b)
    uint64_t *slot_full = bars + 2;
    uint64_t *slot_empty = slot_full + NSLOT;  // both issuers are done with the slot's tile
    uint64_t *s_full = slot_empty + NSLOT;  // [tile]: S_X of step g complete (phase g, steps counted across blocks)
    uint64_t *p_full = s_full + kTiles;     // [tile]: P_X of step g written (and O_X corrected)
    uint64_t *pv_done = p_full + kTiles;    // [tile]: PV_X of step g complete
    uint64_t *o_free = pv_done + kTiles;    // [tile]: the epilogue has read O_X (phase = X's blocks with work)
    uint64_t *s_free = o_free + kTiles;     // [tile]: the softmax has loaded S_X of step g
    uint64_t *final_bar = s_free + kTiles;  // [tile]: every MMA of that tile's issuer has completed
    // the blocks of this CTA, from the producer to the two issuers and the softmax warps (10 consumer warps)
    const WorkRing ring{reinterpret_cast<int *>(smem + L::kWorkOff), final_bar + kTiles,
                        final_bar + kTiles + kWorkRing};
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_blk = (a.N + kTiles * kBM - 1) / (kTiles * kBM);
    const int n_work = n_blk * a.B * a.H;
    const int N = a.N;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, kTiles);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], kTiles);
        }
        for (int x = 0; x < kTiles; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);  // one arrive per softmax warp of tile x
            mbar_init(&pv_done[x], 1);
            mbar_init(&o_free[x], 4);
            mbar_init(&s_free[x], 4);
            mbar_init(&final_bar[x], 1);
        }
        for (int i = 0; i < kWorkRing; ++i) {
            mbar_init(&ring.full[i], 1);
            mbar_init(&ring.empty[i], kTiles + 4 * kTiles);
        }
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
            int Lw = work_draw(a, 0, n_work);
            bool ok = work_publish(ring, 0, Lw, a.status, kSiteWork);
            while (ok && Lw >= 0) {
                const DuoBlock w = duo_block(a, Lw, n_blk);
                // Q of this block goes first, ahead of its K and V tiles, although its buffer frees only when the
                // previous block's last S products complete (after the first K / V pair measured 0.3-0.7 % slower)
                const int q_at = 0;
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
                if (!ok) break;
                // the next block, drawn once this one's loads are issued
                Lw = work_draw(a, nb, n_work);
                ok = work_publish(ring, nb, Lw, a.status, kSiteWork);
            }
            work_finish(a);
            // Drain: never leave the CTA with a TMA write still in flight.
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            if (nb > 0) mbar_wait(q_full, (nb - 1) & 1, a.status, kSiteDrain);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ the tcgen05 issuer of tile x
        // The whole warp runs the loop (operands stay warp-uniform); one elected lane issues the MMAs and
        // the commits.  Over a block's K/V stream j = 0 .. n_all - 1 it issues S_X(j) -- which needs only the
        // softmax's load of S_X(j - 1) -- and then PV_X(j - 1), and after each tile it has no more use for
        // commits to that slot's release; for j at or past its own tile count it only releases.
        const int x = warp - 1;
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, false, true);
        const uint64_t q_desc = sdesc_sw128(smem_u32(q_s) + x * L::kQBytes, 16, 1024);
        const uint32_t slot_addr = smem_u32(slots);
        const uint32_t p_col = kColP + x * (kBN / 2);
        const bool leader = elect_one();
        bool ok = true;
        int gidx = 0;    // ring position of this block's K_0
        int step0 = 0;   // steps of this tile before this block
        int blocks = 0;  // earlier blocks in which this tile had work (epilogues)
        int nb = 0;
        auto commit_to = [&](uint64_t *bar) {
            if (leader) mma_commit(bar);
            __syncwarp();
        };
        while (ok) {
            const int Lw = work_take(ring, nb, a.status, kSiteWork, ok);
            if (!ok || Lw < 0) break;
            const DuoBlock w = duo_block(a, Lw, n_blk);
            const int n = x == 0 ? w.n_kv0 : w.n_kv1;
            if (!(ok = warp_wait(q_full, nb & 1, a.status, kSiteQ))) break;
            tc_fence_after();
            if (n == 0) commit_to(q_empty);  // this tile has no rows in the block
            // S_X(j) = Q_X K_j^T into S_X
            auto issue_s = [&](int j) {
                const int g = gidx + 2 * j;
                const int slot = g % NSLOT;
                if (ok && j < n) {
                    if (!(ok = warp_wait(&slot_full[slot], (g / NSLOT) & 1, a.status, kSiteSlotFull))) return;
                    const int st = step0 + j;
                    if (st >= 1 && !(ok = warp_wait(&s_free[x], (st - 1) & 1, a.status, kSiteSFree))) return;
                    tc_fence_after();
                    const uint64_t k_desc = sdesc_sw128(slot_addr + slot * L::kSlotBytes, 16, 1024);
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t off = (ks >> 2) * (kBM * 128) + (ks & 3) * 32;
                            mma_ss(tmem + kColS + x * kBN, sdesc_add(q_desc, off),
                                   sdesc_add(k_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32), idesc_s, ks > 0);
                        }
                        mma_commit(&s_full[x]);
                    }
                    __syncwarp();
                    if (j == n - 1) commit_to(q_empty);  // this issuer's last S product of the block
                } else if (ok) {
                    // no product of this tile reads K_j, but its release waits until K_j has landed: the
                    // release barrier counts arrivals, and an issuer running ahead would otherwise complete
                    // a later round of the slot before the other issuer has used the earlier one
                    ok = warp_wait(&slot_full[slot], (g / NSLOT) & 1, a.status, kSiteSlotFull);
                }
                if (ok) commit_to(&slot_empty[slot]);  // this issuer is done with K_j
            };
            // O_X += P_X(j) V_j, P_X from TMEM
            auto issue_pv = [&](int j) {
                const int g = gidx + 2 * j + 1;
                const int slot = g % NSLOT;
                if (ok && j < n) {
                    if (!(ok = warp_wait(&slot_full[slot], (g / NSLOT) & 1, a.status, kSiteSlotFull))) return;
                    if (!(ok = warp_wait(&p_full[x], (step0 + j) & 1, a.status, kSitePFull))) return;
                    // the first PV of a block overwrites O_X, which the previous block's epilogue reads
                    if (j == 0 && blocks >= 1 &&
                        !(ok = warp_wait(&o_free[x], (blocks - 1) & 1, a.status, kSiteOFree)))
                        return;
                    tc_fence_after();
                    const uint64_t v_desc = sdesc_sw128(slot_addr + slot * L::kSlotBytes, kBN * 128, 1024);
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            mma_ts(tmem + kColO + x * D, tmem + p_col + kk * 8, sdesc_add(v_desc, kk * 2048),
                                   idesc_o, (j > 0 || kk > 0));
                        mma_commit(&pv_done[x]);
                    }
                    __syncwarp();
                } else if (ok) {
                    ok = warp_wait(&slot_full[slot], (g / NSLOT) & 1, a.status, kSiteSlotFull);  // as for K_j
                }
                if (ok) commit_to(&slot_empty[slot]);  // this issuer is done with V_j
            };
            for (int j = 0; ok && j <= w.n_all; ++j) {
                if (j < w.n_all) issue_s(j);
                if (j >= 1) issue_pv(j - 1);
            }
            step0 += n;
            blocks += n > 0;
            gidx += 2 * w.n_all;
            ++nb;
        }
        // every MMA of this issuer complete: TMEM may be released
        if (leader) mma_commit(&final_bar[x]);
        __syncwarp();
        warp_wait(&final_bar[x], 0, a.status, kSiteFinal);
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int x = (warp - kFirstSoftmaxWarp) >> 2;  // query tile of this warpgroup
        const int quarter = warp & 3;                   // TMEM lanes [32*quarter, 32*quarter + 32)
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_col = kColS + x * kBN, o_col = kColO + x * D;
        const uint32_t p_col = kColP + x * (kBN / 2);
        const float c = a.scale_log2;
        bool ok = true;
        int step0 = 0;  // steps of this tile before the current block
        for (int k = 0; ok; ++k) {
            const int Lw = work_take(ring, k, a.status, kSiteWork, ok);
            if (!ok || Lw < 0) break;
            const DuoBlock w = duo_block(a, Lw, n_blk);
            const int n = x == 0 ? w.n_kv0 : w.n_kv1;
            const int tile_row0 = w.row0 + x * kBM;
            const int row = tile_row0 + r;
            float m = -INFINITY, l = 0.f;  // running max (log2 units) and sum
            for (int j = 0; j < n; ++j) {
                const int st = step0 + j;
                ok = mbar_wait(&s_full[x], st & 1, a.status, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t raw[kBN];
#pragma unroll
                for (int ch = 0; ch < kBN / 32; ++ch) tmem_ld32(tmem + lane_base + s_col + ch * 32, raw + ch * 32);
                tmem_wait_ld();
                // S_X(j) is in registers: the issuer may compute S_X(j + 1) into the buffer
                tc_fence_before();
                warp_arrive(&s_free[x]);
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
                // P_X and O_X are read by PV_X(j - 1): it must have completed before they are rewritten
                if (st >= 1) {
                    ok = mbar_wait(&pv_done[x], (st - 1) & 1, a.status, kSitePV);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                }
                // P = 2^(s c - m) as bf16 pairs, 16 columns per store; the scaling FMA and the row sum run on
                // fp32 pairs
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
                    tmem_st16(tmem + lane_base + p_col + h * 16, pk);
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
            if (!ok || n == 0) continue;
            // the block's last PV_X has completed: O_X is final
            step0 += n;
            ok = mbar_wait(&pv_done[x], (step0 - 1) & 1, a.status, kSiteFinal);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const float inv_l = 1.f / l;
            // row stride and stored columns: the caller's D (at most this kernel's D; the columns past it
            // hold zeros from the TMA's out-of-bounds fill)
            const int Dr = a.D;
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.o) + ((size_t)w.bh * N + row) * Dr;
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
                if (row < N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        if (ch * 32 + v4 * 8 >= Dr) break;
                        uint4 w4;
                        w4.x = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 0]) * inv_l, __uint_as_float(ov[v4 * 8 + 1]) * inv_l);
                        w4.y = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 2]) * inv_l, __uint_as_float(ov[v4 * 8 + 3]) * inv_l);
                        w4.z = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 4]) * inv_l, __uint_as_float(ov[v4 * 8 + 5]) * inv_l);
                        w4.w = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 6]) * inv_l, __uint_as_float(ov[v4 * 8 + 7]) * inv_l);
                        dst[v4] = w4;
                    }
                }
            }
            if (row < N) a.lse[(size_t)w.bh * N + row] = (m + __log2f(l)) * 0.69314718055994531f;
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
                        cudaStream_t s) {
    using L = DuoSmem<D, NSLOT>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    auto kern = fwd_bf16_duo_kernel<D, NSLOT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    const int n_work = ((a.N + kTiles * kBM - 1) / (kTiles * kBM)) * a.H * a.B;
    const int sms = a.num_sms > 0 ? a.num_sms : kNumSms;
    dim3 grid(n_work < sms ? n_work : sms);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16_duo(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, cudaStream_t s) {
    switch (kernel_head_dim(a.D)) {
        case 64: return launch_spec<64, fwd_nslot(64)>(a, tq, tk, tv, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
