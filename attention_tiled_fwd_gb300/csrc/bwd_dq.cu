// bwd_dq.cu -- first kernel of the atomic-free split backward ("backward
// query" of the metal-flash-attention page's pseudocode): one CTA per 128-row
// query tile of one (batch, head), iterating over K/V tiles.
//
//   D_i = sum_d dO_id O_id                          (prologue, written out)
//   per K/V tile j:  S = Q K_j^T,  P = exp(S scale - L)  (base 2 here),
//                    dP = dO V_j^T,  dS = P * (dP - D),
//                    dQ += dS K_j
//   dQ written once after the last tile, times the softmax scale (which every
//   dS carries; applied once here instead of per score).  Three GEMMs per tile; no atomics and
//   no scratch: each CTA owns its dQ rows outright (the design the page adopts
//   because float atomics are emulated on its GPU; it parallelises fully over
//   query rows here as there).
//
// GB300 mapping: warp 0 TMA producer (Q and dO once; 64-row K_j, V_j tiles
// through a ring); two tcgen05 issuer warps, warp 1 (also the TMEM allocator)
// for S and dP and warp 2 for dQ, so that one keeps the tensor core fed while
// the other waits on a barrier; warps 3-10 compute:
// two warpgroups, each thread owning one query row (its TMEM lane) and one
// half (32 keys) of every tile's columns -- dS is elementwise given the row's
// L and D, so the halves never exchange data, and two warps per SM
// sub-partition hide each other's latencies (four warpgroups of 16 keys
// measured 3 % slower here).  The producer stages O's tile beside Q and dO
// (TMA), and each warpgroup sums its share of D_i = rowsum(dO * O) from the two
// shared tiles; reading O and dO rows from global memory took ~4 us per CTA,
// a third of a CTA's fixed cost.
// TMEM (128 lanes = queries): S[b] = [64b, 64b+64), dP[b] = [128+64b, ...),
// dQ [256, 256+D), b = j % 2, dS[b] = [256+D+32b, +32), then Q as bf16
// pairs.  This kernel serves D = 128 (D = 64 runs bwd_dq_k128.cu, whose
// 128-key tiles make S and dP N = 128 products).  The key tile is 64 rows so
// that S and dP are double-buffered: the tensor core computes S_{j+1},
// dP_{j+1} and dQ_{j-1} while the compute warps turn tile j into dS.  Q sits in TMEM so that
// S = Q K_j^T runs as a TS MMA reading only K_j from shared memory: an N = 64
// product with both operands in shared memory is bound by its bandwidth at two
// thirds of the tensor rate.  (dO has no room beside it: the 512 columns are
// full, so dP reads both operands from shared memory.)  The compute warps copy
// Q from the swizzled shared tiles into TMEM once per CTA.  dS (bf16) is the TMEM A operand of
// dQ += dS K_j; K_j is the B operand in MN-major form (keys are the
// reduction).  tcgen05.mma operations on different accumulators are not
// ordered with each other, so every buffer is rewritten only after its
// previous reader is known complete: the compute warps write dS_j after
// waiting for dQ_{j-2}, the previous reader of dS[j % 2]; S_{j+2} / dP_{j+2}
// overwrite S[b] / dP[b] only after the compute warps finished tile j.  K_j is
// released after dQ_j, which is issued only after S_j completed.
//
// Wider heads (D = 192, 256) run the same kernel with two changes.  Q stays in
// shared memory and S = Q K_j^T is an SS product, because dQ needs D of the 512
// columns.  At D = 192 S and dP stay double-buffered beside dQ's 192 columns.
// At D = 256 dQ takes 256 columns, so S and dP have one buffer each, which every
// compute warp empties into registers first thing (s_free, dp_free) so that
// S_{j+1} and dP_{j+1} can follow at once: TMEM S [0, 64), dP [64, 128), dQ
// [128, 384), dS[b] [384 + 32b, +32).  (Two CTAs per query tile, each keeping
// one half of dQ and both computing S and dP over all of D, measured 37-42 %
// slower: the tensor core did 5/3 of the useful products.)
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBM = 128;          // queries per CTA (TMEM lanes)
constexpr int kBN = kDqKRows;     // keys per tile
constexpr int kComputeWG = 2;     // compute warpgroups, one 32-key half of every tile each
constexpr int kFirstComputeWarp = 3;
constexpr int kThreads = 32 * kFirstComputeWarp + 128 * kComputeWG;

enum : int { kSiteQ = 21, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSiteDsFull, kSiteDq, kSiteFinal, kSiteDrain,
             kSiteDqDone, kSiteQt, kSiteSFree };

template <int D, int NSLOT>
struct DqSmem {
    static constexpr int kQBytes = kBM * D * 2;     // Q, dO and O: 128 x D bf16 each
    static constexpr int kTileBytes = kBN * D * 2;  // one K_j or V_j tile
    static constexpr int kQOff = 0;
    static constexpr int kDoOff = kQBytes;
    static constexpr int kSlotOff = 2 * kQBytes;
    static constexpr int kOOff = kSlotOff + NSLOT * kTileBytes;
    // q_full, slot_full[NSLOT], slot_empty[NSLOT], s_full[2], ds_full[2], final, a_final, dq_done[2], qt_ready,
    // o_full, dp_full[2]
    static constexpr int kNumBars = 1 + 2 * NSLOT + 14;
    static constexpr int kRest = kComputeWG * kBM * 4 + kNumBars * 8 + 16 + 1024;
    // O's tile is staged by TMA where it fits (D = 128): D_i is then summed from shared memory.  At larger D
    // the compute warps read the O and dO rows from global memory instead.
    static constexpr bool kOTile = kOOff + kQBytes + kRest <= 232448;
    static constexpr int kDeltaOff = kOOff + (kOTile ? kQBytes : 0);  // [kComputeWG][kBM] partial sums
    static constexpr int kBarOff = kDeltaOff + kComputeWG * kBM * 4;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

// D: the contraction width the kernel is built for (64-column panels); DQ: the columns of dQ one
// CTA accumulates (D here; D / DQ CTAs per query tile, grid y choosing the columns); QT: Q kept in
// TMEM as the A operand of S (else S reads Q from shared memory).
template <int D, int DQ, bool QT, int NSLOT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                  const __grid_constant__ CUtensorMap tmap_o, const __grid_constant__ CUtensorMap tmap_dq,
                  BwdArgs a) {
    using L = DqSmem<D, NSLOT>;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kTmemCols = 512;
    // kSingle (D = 256 with all of dQ in one CTA): S and dP in one buffer each, emptied by the compute warps into
    // registers first thing (s_free, dp_free), so that dQ's 256 columns fit beside them
    constexpr bool kSingle = !QT && DQ == D && D == 256;
    constexpr uint32_t kColDP0 = kSingle ? 64 : 128;  // dP[b] at kColDP0 + 64 b (b = 0 when kSingle)
    constexpr uint32_t kColDQ = kSingle ? 128 : 256, kColDS = kColDQ + DQ, kColQ = kColDS + 64;
    static_assert(kColQ + (QT ? D / 2 : 0) <= 512, "TMEM budget");
    static_assert(DQ % 64 == 0 && D % DQ == 0, "dQ columns per CTA: whole panels");
    constexpr bool kSplitDp = !QT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem + L::kQOff;
    uint8_t *do_s = smem + L::kDoOff;
    uint8_t *slots = smem + L::kSlotOff;
    uint8_t *o_s = smem + L::kOOff;  // O's tile (kOTile only)
    float *delta_s = reinterpret_cast<float *>(smem + L::kDeltaOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + NSLOT;
    uint64_t *s_full = slot_empty + NSLOT;  // [2]: S_j (and dP_j unless kSplitDp) complete
    uint64_t *ds_full = s_full + 2;         // [2]: dS_j written (and S_j, dP_j read)
    uint64_t *final_bar = ds_full + 2;  // issuer B: every dQ MMA has completed
    uint64_t *a_final = final_bar + 1;  // issuer A: every S / dP MMA has completed
    uint64_t *dq_done = a_final + 1;    // [2]: dQ_j completed (its dS buffer j % 2 is free)
    uint64_t *qt_ready = dq_done + 2;   // Q is in TMEM
    uint64_t *o_full = qt_ready + 1;    // O's tile landed (kOTile)
    // [2]: dP_j complete, with its own barrier at D = 192, 256 (kSplitDp): P_j's exponentials then run while
    // the dP product still executes, which measured 7-18 % faster there.  At D = 128 (Q in TMEM) s_full
    // covers S_j and dP_j both: the split measured 10 % slower.
    uint64_t *dp_full = o_full + 1;
    uint64_t *s_free = dp_full + 2;  // kSingle: every compute warp has loaded S_j
    uint64_t *dp_free = s_free + 1;  // kSingle: every compute warp has loaded dP_j
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    __shared__ int epi_abort;  // a compute warp's wait ran out: the epilogue stores nothing
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    tile_order((a.N + kBM - 1) / kBM, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int q_tile = (a.N + kBM - 1) / kBM - 1 - rank;  // causal: the last query tile has the most keys
    const int N = a.N;
    const int kv_end = a.causal ? min(N, (q_tile + 1) * kBM) : N;
    const int n_kv = (kv_end + kBN - 1) / kBN;  // >= 1
    const int dq0 = blockIdx.y * DQ;            // first dQ column of this CTA
    const int Dr = a.D;                         // row stride and real columns (<= D; the rest are zeros)

    if (threadIdx.x == 0) {
        epi_abort = 0;
        mbar_init(q_full, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&dp_full[b], 1);
            mbar_init(&ds_full[b], 4 * kComputeWG);  // one arrive per compute warp
        }
        mbar_init(final_bar, 1);
        mbar_init(a_final, 1);
        for (int b = 0; b < 2; ++b) mbar_init(&dq_done[b], 1);
        mbar_init(qt_ready, 4 * kComputeWG);  // one arrive per compute warp
        mbar_init(o_full, 1);
        mbar_init(s_free, 4 * kComputeWG);
        mbar_init(dp_free, 4 * kComputeWG);
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
        if (lane == 0) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            tma_prefetch_desc(&tmap_do);
            mbar_arrive_expect_tx(q_full, 2 * L::kQBytes);
#pragma unroll
            for (int p = 0; p < kPanels; ++p) {
                tma_load_3d(q_s + p * (kBM * 128), &tmap_q, q_full, p * 64, q_tile * kBM, bh);
                tma_load_3d(do_s + p * (kBM * 128), &tmap_do, q_full, p * 64, q_tile * kBM, bh);
            }
            if constexpr (L::kOTile) {
                tma_prefetch_desc(&tmap_o);
                mbar_arrive_expect_tx(o_full, L::kQBytes);
#pragma unroll
                for (int p = 0; p < kPanels; ++p)
                    tma_load_3d(o_s + p * (kBM * 128), &tmap_o, o_full, p * 64, q_tile * kBM, bh);
            }
            int last_round[NSLOT];
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) last_round[s] = -1;
            for (int idx = 0; idx < 2 * n_kv; ++idx) {
                const int slot = idx % NSLOT, round = idx / NSLOT;
                if (!mbar_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty)) break;
                uint8_t *dst = slots + slot * L::kTileBytes;
                const CUtensorMap *map = (idx & 1) ? &tmap_v : &tmap_k;
                mbar_arrive_expect_tx(&slot_full[slot], L::kTileBytes);
#pragma unroll
                for (int p = 0; p < kPanels; ++p)
                    tma_load_3d(dst + p * (kBN * 128), map, &slot_full[slot], p * 64, (idx >> 1) * kBN, bh);
#pragma unroll
                for (int s = 0; s < NSLOT; ++s)
                    if (s == slot) last_round[s] = round;
            }
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            mbar_wait(q_full, 0, a.status, kSiteDrain);
            if constexpr (L::kOTile) mbar_wait(o_full, 0, a.status, kSiteDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // Issuer A: S_j = Q K_j^T and dP_j = dO V_j^T into buffer j % 2.  The whole warp runs the loop
        // (operands stay warp-uniform); one elected lane issues the MMAs and their commits.
        constexpr uint32_t idesc_sq = idesc_bf16_f32(kBM, kBN, false, false);  // S, dP: 128 x 64
        const uint64_t q_desc = sdesc_sw128(smem_u32(q_s), 16, 1024);
        const uint64_t do_desc = sdesc_sw128(smem_u32(do_s), 16, 1024);
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = warp_wait(q_full, 0, a.status, kSiteQ) && (!QT || warp_wait(qt_ready, 0, a.status, kSiteQt));
        tc_fence_after();
        for (int j = 0; ok && j < n_kv; ++j) {
            const int k_slot = (2 * j) % NSLOT, k_round = (2 * j) / NSLOT;
            const int v_slot = (2 * j + 1) % NSLOT, v_round = (2 * j + 1) / NSLOT;
            const uint32_t b = j & 1;
            // S[b], dP[b] last held tile j-2, which the compute warps have finished with
            if (!kSingle && j >= 2 && !(ok = warp_wait(&ds_full[b], ((j - 2) >> 1) & 1, a.status, kSiteDsFull))) break;
            if constexpr (!kSplitDp) {
                if (!(ok = warp_wait(&slot_full[k_slot], k_round & 1, a.status, kSiteSlotFull))) break;
                if (!(ok = warp_wait(&slot_full[v_slot], v_round & 1, a.status, kSiteSlotFull))) break;
                tc_fence_after();
                const uint64_t k_desc = sdesc_sw128(slot_addr + k_slot * L::kTileBytes, 16, 1024);
                const uint64_t v_desc = sdesc_sw128(slot_addr + v_slot * L::kTileBytes, 16, 1024);
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ts(tmem + 64 * b, tmem + kColQ + ks * 8,
                               sdesc_add(k_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32), idesc_sq, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tmem + 128 + 64 * b, sdesc_add(do_desc, (ks >> 2) * (kBM * 128) + (ks & 3) * 32),
                               sdesc_add(v_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32), idesc_sq, ks > 0);
                    mma_commit(&s_full[b]);
                    mma_commit(&slot_empty[v_slot]);  // V_j is no longer needed
                }
                __syncwarp();
            } else {
                if (!(ok = warp_wait(&slot_full[k_slot], k_round & 1, a.status, kSiteSlotFull))) break;
                // kSingle: S_j overwrites S_{j-1}, which every compute warp must have loaded
                if (kSingle && j >= 1 && !(ok = warp_wait(s_free, (j - 1) & 1, a.status, kSiteSFree))) break;
                tc_fence_after();
                const uint32_t sb = kSingle ? 0 : b;  // the S / dP buffer
                const uint64_t k_desc = sdesc_sw128(slot_addr + k_slot * L::kTileBytes, 16, 1024);
                const uint64_t v_desc = sdesc_sw128(slot_addr + v_slot * L::kTileBytes, 16, 1024);
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tmem + 64 * sb, sdesc_add(q_desc, (ks >> 2) * (kBM * 128) + (ks & 3) * 32),
                               sdesc_add(k_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32), idesc_sq, ks > 0);
                    mma_commit(&s_full[sb]);
                }
                __syncwarp();
                if (!(ok = warp_wait(&slot_full[v_slot], v_round & 1, a.status, kSiteSlotFull))) break;
                if (kSingle && j >= 1 && !(ok = warp_wait(dp_free, (j - 1) & 1, a.status, kSiteSFree))) break;
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tmem + kColDP0 + 64 * sb, sdesc_add(do_desc, (ks >> 2) * (kBM * 128) + (ks & 3) * 32),
                               sdesc_add(v_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32), idesc_sq, ks > 0);
                    mma_commit(&dp_full[sb]);
                    mma_commit(&slot_empty[v_slot]);  // V_j is no longer needed
                }
                __syncwarp();
            }
        }
        // Drain this warp's MMAs before TMEM can be released (immediate in the normal path).
        if (leader) mma_commit(a_final);
        __syncwarp();
        warp_wait(a_final, 0, a.status, kSiteFinal);
    } else if (warp == 2) {
        // Issuer B: dQ += dS_j K_j.
        constexpr uint32_t idesc_dq = idesc_bf16_f32(kBM, DQ, false, true);  // dQ += dS K: 128 x DQ
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            const uint32_t b = j & 1;
            const int k_slot = (2 * j) % NSLOT;
            // B = this CTA's DQ columns of K_j (MN-major: whole 64-column panels from panel dq0 / 64 on)
            const uint64_t kmn_desc =
                sdesc_sw128(slot_addr + k_slot * L::kTileBytes + (dq0 / 64) * (kBN * 128), kBN * 128, 1024);
            if (!(ok = warp_wait(&ds_full[b], (j >> 1) & 1, a.status, kSiteDsFull))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tmem + kColDQ, tmem + kColDS + 32 * b + kk * 8, sdesc_add(kmn_desc, kk * 2048),
                           idesc_dq, (j > 0 || kk > 0));
                mma_commit(&dq_done[b]);
                mma_commit(&slot_empty[k_slot]);  // S_j completed before dS_j was produced
            }
            __syncwarp();
        }
        if (leader) mma_commit(final_bar);
        __syncwarp();
        warp_wait(final_bar, 0, a.status, kSiteFinal);
    } else {
        const int quarter = warp & 3;
        const int g = (warp - kFirstComputeWarp) >> 2;  // key range of every tile
        const int r = quarter * 32 + lane;
        const int row = q_tile * kBM + r;
        const bool valid = row < N;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float c = a.scale_log2;
        // P = 2^(S c - L log2 e); invalid rows get P = 0.
        const float lse2 = valid ? a.lse[(size_t)bh * N + row] * 1.4426950408889634f : INFINITY;
        // D_i = sum_d dO_id O_id for this thread's row: warpgroup g sums columns [g D / kComputeWG,
        // (g + 1) D / kComputeWG), the partial sums meet in shared memory, and every warpgroup adds them in
        // the same order.  With O's tile staged, both operands come from the swizzled shared tiles, whose
        // chunk k of row r sits at the same place in each (columns past the caller's D and rows past N are
        // zeros from the TMA); otherwise from the rows in global memory.
        constexpr int kDCols = D / kComputeWG;
        float delta = 0.f;
        if constexpr (L::kOTile) {
            bool ook = mbar_wait(o_full, 0, a.status, kSiteQ) && mbar_wait(q_full, 0, a.status, kSiteQ);
            if (__all_sync(0xffffffffu, ook)) {
#pragma unroll
                for (int p = g * (kDCols / 64); p < (g + 1) * (kDCols / 64); ++p) {
                    const uint8_t *orow = o_s + p * (kBM * 128) + r * 128;
                    const uint8_t *drow = do_s + p * (kBM * 128) + r * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        // the swizzled position of chunk k: lanes (rows) spread over all 32 banks
                        const uint4 ov = *reinterpret_cast<const uint4 *>(orow + ((k ^ (r & 7)) << 4));
                        const uint4 dv = *reinterpret_cast<const uint4 *>(drow + ((k ^ (r & 7)) << 4));
                        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[t]));
                            const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&dw[t]));
                            delta = fmaf(of.x, df.x, delta);
                            delta = fmaf(of.y, df.y, delta);
                        }
                    }
                }
            }
        } else if (valid) {
            const uint4 *orow = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.o) +
                                                                ((size_t)bh * N + row) * Dr + g * kDCols);
            const uint4 *drow = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.dO) +
                                                                ((size_t)bh * N + row) * Dr + g * kDCols);
#pragma unroll 4
            for (int i = 0; i < kDCols / 8; ++i) {
                if (g * kDCols + 8 * i >= Dr) break;
                const uint4 ov = orow[i], dv = drow[i];
                const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[t]));
                    const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&dw[t]));
                    delta = fmaf(of.x, df.x, delta);
                    delta = fmaf(of.y, df.y, delta);
                }
            }
        }
        delta_s[g * kBM + r] = delta;
        // every compute warp reaches this barrier: nothing before it waits or exits early
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kComputeWG) : "memory");
        delta = 0.f;
#pragma unroll
        for (int t = 0; t < kComputeWG; ++t) delta += delta_s[t * kBM + r];
        if (valid && g == 0 && blockIdx.y == 0) a.delta[(size_t)bh * N + row] = delta;
        // Q rows into TMEM as bf16 pairs, one 64-column panel per warpgroup (row r of a panel is 128 B at
        // r * 128, its 16-byte chunk k stored at k ^ (r % 8)).  Copying Q before summing D_i lets S_0 and dP_0
        // start earlier but measured 6 % slower per key tile over long rows, so D_i comes first.
        {
            bool qok = !QT || mbar_wait(q_full, 0, a.status, kSiteQ);
            if (!__all_sync(0xffffffffu, qok)) qok = false;
            if (QT && qok) {
#pragma unroll
                for (int p = g; p < kPanels; p += kComputeWG) {
                    const uint8_t *panel = q_s + p * (kBM * 128) + r * 128;
                    uint32_t w[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(panel + ((k ^ (r & 7)) << 4));
                        w[4 * k] = x.x;
                        w[4 * k + 1] = x.y;
                        w[4 * k + 2] = x.z;
                        w[4 * k + 3] = x.w;
                    }
                    tmem_st32(tmem + lane_base + kColQ + 32 * p, w);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            warp_arrive(qt_ready);
        }
        const int lim = a.causal ? min(N - 1, row) : N - 1;  // last visible key
        constexpr int kHalf = kBN / kComputeWG;              // columns per thread per tile
        const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(-lse2, -lse2), d2 = f2_pack(delta, delta);
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const uint32_t b = j & 1;
            const uint32_t sb = kSingle ? 0 : b;                        // the S / dP buffer
            const uint32_t sph = kSingle ? (j & 1) : ((j >> 1) & 1);   // its phase for tile j
            ok = mbar_wait(&s_full[sb], sph, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int key0 = j * kBN + g * kHalf;
            const bool need_mask = (key0 + kHalf > N) || (a.causal && key0 + kHalf - 1 > q_tile * kBM);
            // dS[j % 2] was last read by dQ_{j-2}
            if (j >= 2) {
                ok = mbar_wait(&dq_done[b], ((j - 2) >> 1) & 1, a.status, kSiteDqDone);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
            }
            uint32_t dsk[kHalf / 2];
            if constexpr (!kSplitDp) {
                uint32_t sraw[kHalf], praw[kHalf];
                tmem_ld_n<kHalf>(tmem + lane_base + 64 * b + g * kHalf, sraw);
                tmem_ld_n<kHalf>(tmem + lane_base + 128 + 64 * b + g * kHalf, praw);
                tmem_wait_ld();
                // dS / scale = P * (dP - D), on fp32 pairs (f32x2), two scores per instruction
#pragma unroll
                for (int i = 0; i < kHalf; i += 2) {
                    float p0, p1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sraw[i]), __uint_as_float(sraw[i + 1])), c2, nl2), p0, p1);
                    p0 = ex2_approx(p0);
                    p1 = ex2_approx(p1);
                    if (need_mask) {
                        if (key0 + i > lim) p0 = 0.f;
                        if (key0 + i + 1 > lim) p1 = 0.f;
                    }
                    dsk[i / 2] = f2_to_bf16x2(
                        f2_mul(f2_sub(f2_pack(__uint_as_float(praw[i]), __uint_as_float(praw[i + 1])), d2), f2_pack(p0, p1)));
                }
            } else {
                uint32_t sraw[kHalf], praw[kHalf];
                uint64_t p2[kHalf / 2];
                tmem_ld_n<kHalf>(tmem + lane_base + 64 * sb + g * kHalf, sraw);
                tmem_wait_ld();
                if constexpr (kSingle) {
                    // S_j is in registers: S_{j+1} may overwrite the buffer
                    tc_fence_before();
                    warp_arrive(s_free);
                }
                // P = 2^(S c - L log2 e) while dP_j may still be executing, on fp32 pairs (f32x2)
#pragma unroll
                for (int i = 0; i < kHalf; i += 2) {
                    float p0, p1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sraw[i]), __uint_as_float(sraw[i + 1])), c2, nl2), p0, p1);
                    p0 = ex2_approx(p0);
                    p1 = ex2_approx(p1);
                    if (need_mask) {
                        if (key0 + i > lim) p0 = 0.f;
                        if (key0 + i + 1 > lim) p1 = 0.f;
                    }
                    p2[i / 2] = f2_pack(p0, p1);
                }
                ok = mbar_wait(&dp_full[sb], sph, a.status, kSiteSFull);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                tmem_ld_n<kHalf>(tmem + lane_base + kColDP0 + 64 * sb + g * kHalf, praw);
                tmem_wait_ld();
                if constexpr (kSingle) {
                    tc_fence_before();
                    warp_arrive(dp_free);
                }
                // dS / scale = P * (dP - D), two scores per instruction
#pragma unroll
                for (int i = 0; i < kHalf; i += 2)
                    dsk[i / 2] = f2_to_bf16x2(
                        f2_mul(f2_sub(f2_pack(__uint_as_float(praw[i]), __uint_as_float(praw[i + 1])), d2), p2[i / 2]));
            }
            tmem_st_n<kHalf / 2>(tmem + lane_base + kColDS + 32 * b + g * (kHalf / 2), dsk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&ds_full[b]);
        }
        if (ok) {
            ok = mbar_wait(final_bar, 0, a.status, kSiteDq);  // single phase: every MMA has completed
            ok = __all_sync(0xffffffffu, ok);
        }
        // Epilogue: dQ (times the scale) is staged in the Q / dO tiles' shared memory, which no MMA reads any
        // more (every S and dP product completed before the last dS was written), as 128-byte-swizzled
        // panels of 128 rows -- 64 columns in bf16, 32 in fp32 -- and written by TMA bulk stores, which clip
        // rows past N and columns past the caller's D.  (A thread storing its own row to global memory
        // touches a different 128-byte line per lane and instruction, and took ~1.3 us per CTA.)
        static_assert(DQ * 4 <= 4 * D, "staging fits in the Q and dO tiles");
        if (ok) {
            tc_fence_after();
            constexpr int kCols = DQ / kComputeWG;  // this warpgroup's columns of dQ (64 or 96)
            static_assert(kCols % 32 == 0, "32-column TMEM loads");
            const int sw = r & 7;
            uint32_t v[32];
#pragma unroll
            for (int ch = 0; ch < kCols / 32; ++ch) {
                const int col = g * kCols + ch * 32;  // within this CTA's DQ columns
                tmem_ld32(tmem + lane_base + kColDQ + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * a.scale);
                if (a.grad_bf16) {
                    // 32 columns = 4 chunks of a 64-column panel's row
                    uint8_t *prow = smem + (col / 64) * (kBM * 128) + r * 128;
                    const int c0 = (col % 64) / 8;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(prow + (((c0 + c) ^ sw) << 4),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1])),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
                } else {
                    // 32 columns = one 32-column fp32 panel's row
                    uint8_t *prow = smem + (col / 32) * (kBM * 128) + r * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(prow + ((c ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                }
            }
        } else if (lane == 0) {
            epi_abort = 1;
        }
        fence_proxy_async_smem();  // the staged tile is read by the TMA (async proxy)
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kComputeWG) : "memory");
        if (threadIdx.x == 32 * kFirstComputeWarp && !epi_abort) {
            const int n_panels = a.grad_bf16 ? DQ / 64 : DQ / 32;
            const int pw = a.grad_bf16 ? 64 : 32;  // panel width in elements
            for (int p = 0; p < n_panels; ++p)
                if (dq0 + p * pw < Dr)  // a panel wholly past the caller's D is not stored
                    tma_store_3d(&tmap_dq, smem + p * (kBM * 128), dq0 + p * pw, q_tile * kBM, bh);
            tma_store_commit();
            tma_store_wait_read();  // the CTA's shared memory must outlive the stores' reads
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int DQ, bool QT, int NSLOT>
cudaError_t launch_spec(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, const CUtensorMap &to, const CUtensorMap &tdq, cudaStream_t s) {
    using L = DqSmem<D, NSLOT>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    auto kern = bwd_dq_kernel<D, DQ, QT, NSLOT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBM - 1) / kBM) * a.H * a.B, D / DQ);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, tdo, to, tdq, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tdo, const CUtensorMap &to, const CUtensorMap &tdq, cudaStream_t s) {
    switch (kernel_head_dim(a.D)) {
        case 128: return launch_spec<128, 128, true, 8>(a, tq, tk, tv, tdo, to, tdq, s);
        case 192: return launch_spec<192, 192, false, 4>(a, tq, tk, tv, tdo, to, tdq, s);  // 3, 5 slots slower
        case 256: return launch_spec<256, 256, false, 3>(a, tq, tk, tv, tdo, to, tdq, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
