// bwd_dkdv.cu -- second kernel of the atomic-free split backward ("backward
// key-value" of the metal-flash-attention page's pseudocode): one CTA per
// 128-key tile of one (batch, head), iterating over query tiles.
//
//   per query tile i:  S^T = K Q_i^T,  P^T = exp(S^T scale - L_i) (base 2 here),
//                      dV += P^T dO_i,
//                      dP^T = V dO_i^T,  dS^T = P^T * (dP^T - D_i),
//                      dK += dS^T Q_i
//   dK (times the softmax scale, which every dS^T carries and which is
//   applied once here instead of per score) and dV written once after the
//   last query tile.  Four GEMMs per tile, no
//   atomics, no scratch.  Causal: only query tiles on or below the diagonal
//   (queries >= keys) are visited.
//
// GB300 mapping: warp 0 TMA producer (K, V once; 64-row Q_i, dO_i tiles through
// a ring); two tcgen05 issuer warps, warp 1 (also the TMEM allocator) for
// S^T and dP^T and warp 2 for dV and dK, so that one keeps the tensor core
// fed while the other waits on a barrier (an MMA's issue blocks until the
// tensor core accepts it, at its execution rate); warps 3-18 compute: four
// warpgroups, each thread owning one key row (its TMEM lane) and one quarter
// (16 queries) of every tile's columns -- P^T and dS^T are elementwise given the
// queries' L_i and D_i (broadcast from shared memory as float4), so the
// quarters never exchange data, and four compute warps per SM sub-partition
// hide the latencies of the TMEM loads and the exponentials (measured 2.6 %
// faster at D = 128 than two warpgroups of 32 queries).  This kernel serves
// D = 128; D = 64 runs bwd_dkdv_q128.cu, whose 128-query tiles make S^T and
// dP^T N = 128 products.
// The producer warp also copies each query tile's L_i and D_i into a ring of
// kStatSlots shared buffers (4-byte cp.async, zero fill past N, completion
// tracked by the copies' own mbarrier arrivals), so no compute warp waits for
// another to load or publish them.
// TMEM (128 lanes = keys): S^T[b] = [64b, 64b+64), dP^T[b] = [128+64b, ...),
// dV [256, 256+D), dK [256+D, 256+2D), b = i % 2.  The query tile is 64 rows so
// that S^T and dP^T are double-buffered: the tensor core computes tile i+1
// while the compute warps turn tile i into P^T and dS^T.
// P^T (bf16) overwrites S^T[b] and dS^T overwrites dP^T[b]: warpgroup g packs
// its 16 queries into the first 8 columns of its own 16-column range (columns
// [16g, 16g+8)), so no warpgroup writes columns another has yet to read.  They
// feed dV / dK as the TMEM A operand (16-query step kk reads columns 16kk),
// with dO_i / Q_i as MN-major B operands (queries are the reduction).
// tcgen05.mma operations are only ordered among MMAs on the same accumulator (and a commit only tracks
// its own thread's MMAs), so the S^T/dP^T issuer waits for dV_{i-2} (resp.
// dK_{i-2}) to complete before S^T_i (resp. dP^T_i) overwrites that buffer;
// those waits are two tiles old and normally already satisfied, and each
// buffer has its own completion barrier (see dv_done below).  Q_i and dO_i
// slots are released after dK_i, which is issued only after the compute warps
// saw S^T_i and dP^T_i complete.
//
// Wider heads run the same kernel.  At D = 192, dV and dK take 384 columns, so
// S^T and dP^T are single-buffered (NB = 1): S^T_{i+1} waits for dV_i and dP^T_{i+1}
// for dK_i.  At D = 256 dV and dK (256 columns each) fill TMEM, so two CTAs share
// each key tile and split the gradients (VK): the first keeps dV (S^T x 2 + dV),
// the second dK (S^T x 2 + dP^T x 2 + dK); the dV CTA computes no dP^T, so the
// tensor core does 5/4 of the useful products.  (Splitting the columns instead,
// each CTA with half of dV and dK and both computing S^T and dP^T, did 6/4 and
// measured 15 % slower.)
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBN = 128;          // keys per CTA (TMEM lanes)
constexpr int kBQ = kDkdvQRows;   // queries per tile
constexpr int kComputeWG = 4;     // compute warpgroups, one 16-query range of every tile each
constexpr int kFirstComputeWarp = 3;
constexpr int kThreads = 32 * kFirstComputeWarp + 128 * kComputeWG;

enum : int { kSiteKV = 41, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePReady, kSiteDpFull, kSiteDsReady,
             kSiteDone, kSiteFinal, kSiteDrain, kSiteStats, kSiteDvDone, kSiteDkDone };

template <int D, int NSLOT, int kStatSlots>
struct DkdvSmem {
    static constexpr int kKVBytes = kBN * D * 2;
    static constexpr int kTileBytes = kBQ * D * 2;  // one Q_i or dO_i tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKVBytes;
    static constexpr int kSlotOff = 2 * kKVBytes;
    static constexpr int kStatOff = kSlotOff + NSLOT * kTileBytes;  // [kStatSlots][L kBQ | D kBQ] fp32
    static constexpr int kBarOff = kStatOff + kStatSlots * 2 * kBQ * 4;
    // kv_full, slot_full[NSLOT], slot_empty[NSLOT], s_full[2], dp_full[2], p_ready[2], ds_ready[2],
    // stat_full[kStatSlots], stat_empty[kStatSlots], dv_done[2], dk_done[2], final, a_final
    static constexpr int kNumBars = 1 + 2 * NSLOT + 8 + 2 * kStatSlots + 6;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

// D: the contraction width the kernel is built for (64-column panels); DO: the columns of dV and dK one
// CTA accumulates (D here); NB: S^T / dP^T buffers in TMEM (2, or 1 where dV and dK leave no room);
// kStatSlots: query tiles whose L / D are staged ahead.
// VK: the two CTAs of a key tile split the gradients rather than their columns (grid y = 0 keeps all of
// dV, y = 1 all of dK); the dV CTA computes no dP^T, and neither repeats the other's product.
template <int D, int DO, int NB, int NSLOT, int kStatSlots, bool VK>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                    const __grid_constant__ CUtensorMap tmap_dk, const __grid_constant__ CUtensorMap tmap_dv,
                    BwdArgs a) {
    using L = DkdvSmem<D, NSLOT, kStatSlots>;
    constexpr int kPanels = D / 64;
    // Compute warpgroup g owns queries [g kSpan, (g+1) kSpan) of every tile and packs their bf16 P^T /
    // dS^T into the first kSpan / 2 columns of that range: 16-query k-step kk sits at column
    // kSpan (kk / kStepsPerWG) + 8 (kk % kStepsPerWG).
    constexpr int kSpan = kBQ / kComputeWG;
    constexpr int kStepsPerWG = kSpan / 16;
    static_assert(kSpan == 16 || kSpan == 32, "16 or 32 queries per compute thread");
    constexpr uint32_t kTmemCols = 512;
    // TMEM: S^T[b] = [64b, +64), dP^T[b] = [64 NB + 64b, +64), dV, dK (DO columns each)
    // (VK: the CTA's one gradient at 128 NB)
    constexpr uint32_t kColDP = 64 * NB, kColDV = 128 * NB, kColDK = VK ? 128 * NB : 128 * NB + DO;
    static_assert(128 * NB + (VK ? 1 : 2) * DO <= 512, "TMEM budget");
    static_assert(DO % 64 == 0 && D % DO == 0 && (NB == 1 || NB == 2), "dV / dK columns per CTA: whole panels");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *k_s = smem + L::kKOff;
    uint8_t *v_s = smem + L::kVOff;
    uint8_t *slots = smem + L::kSlotOff;
    float *stat_s = reinterpret_cast<float *>(smem + L::kStatOff);  // slot s: L at [2 kBQ s], D after it
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + NSLOT;
    uint64_t *s_full = slot_empty + NSLOT;  // [2]
    uint64_t *dp_full = s_full + 2;         // [2]
    uint64_t *p_ready = dp_full + 2;        // [2]
    uint64_t *ds_ready = p_ready + 2;       // [2]
    uint64_t *stat_full = ds_ready + 2;           // [kStatSlots]: a query tile's L / D landed
    uint64_t *stat_empty = stat_full + kStatSlots;  // [kStatSlots]: every compute warp is done with it
    // dV_i / dK_i complete, one barrier per TMEM buffer b = i % 2: issuer A waits for tile i - 2 while
    // tile i - 1's product may already have completed, and on a single barrier that later phase
    // would carry the parity it waits for.
    uint64_t *dv_done = stat_empty + kStatSlots;  // [2]
    uint64_t *dk_done = dv_done + 2;              // [2]
    uint64_t *final_bar = dk_done + 2;   // issuer B: every dV / dK MMA has completed
    uint64_t *a_final = final_bar + 1;   // issuer A: every S^T / dP^T MMA has completed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    __shared__ int epi_abort;  // a compute warp's wait ran out: the epilogue stores nothing
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    tile_order((a.N + kBN - 1) / kBN, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int k_tile = rank;  // causal: key tile 0 has the most query tiles
    const int N = a.N;
    const int n_q_total = (N + kBQ - 1) / kBQ;
    const int q_begin = a.causal ? (k_tile * kBN) / kBQ : 0;
    const int n_q = n_q_total - q_begin;  // >= 1
    const int do0 = VK ? 0 : blockIdx.y * DO;  // first dV / dK column of this CTA
    const bool role_dv = VK && blockIdx.y == 0;  // VK: this CTA keeps dV only
    const bool role_dk = VK && blockIdx.y == 1;  // VK: this CTA keeps dK only
    const int Dr = a.D;                   // row stride and real columns (<= D; the rest are zeros)

    if (threadIdx.x == 0) {
        epi_abort = 0;
        mbar_init(kv_full, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&dp_full[b], 1);
            mbar_init(&p_ready[b], 4 * kComputeWG);  // one arrive per compute warp
            mbar_init(&ds_ready[b], 4 * kComputeWG);
        }
        for (int t = 0; t < kStatSlots; ++t) {
            mbar_init(&stat_full[t], 32);  // one arrival per producer lane, when its copies have landed
            mbar_init(&stat_empty[t], 4 * kComputeWG);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&dv_done[b], 1);
            mbar_init(&dk_done[b], 1);
        }
        mbar_init(final_bar, 1);
        mbar_init(a_final, 1);
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
        // TMA producer (lane 0): K, V once, then Q_i, dO_i into the ring.  The whole warp: each query
        // tile's L_i, D_i into the stats ring (4-byte copies, 32 consecutive words per instruction).
        if (lane == 0) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            tma_prefetch_desc(&tmap_do);
            mbar_arrive_expect_tx(kv_full, 2 * L::kKVBytes);
#pragma unroll
            for (int p = 0; p < kPanels; ++p) {
                tma_load_3d(k_s + p * (kBN * 128), &tmap_k, kv_full, p * 64, k_tile * kBN, bh);
                tma_load_3d(v_s + p * (kBN * 128), &tmap_v, kv_full, p * 64, k_tile * kBN, bh);
            }
        }
        const float *lse_g = a.lse + (size_t)bh * N;
        const float *del_g = a.delta + (size_t)bh * N;
        int last_round[NSLOT];
#pragma unroll
        for (int s = 0; s < NSLOT; ++s) last_round[s] = -1;
        bool ok = true;
        for (int idx = 0; ok && idx < 2 * n_q; ++idx) {
            const int slot = idx % NSLOT, round = idx / NSLOT;
            if (!(ok = warp_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty))) break;
            if (lane == 0) {
                uint8_t *dst = slots + slot * L::kTileBytes;
                const CUtensorMap *map = (idx & 1) ? &tmap_do : &tmap_q;
                mbar_arrive_expect_tx(&slot_full[slot], L::kTileBytes);
#pragma unroll
                for (int p = 0; p < kPanels; ++p)
                    tma_load_3d(dst + p * (kBQ * 128), map, &slot_full[slot], p * 64,
                                (q_begin + (idx >> 1)) * kBQ, bh);
            }
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (s == slot) last_round[s] = round;
            if (idx & 1) continue;
            // stats of query tile i = idx / 2
            const int i = idx >> 1, ss = i % kStatSlots, sr = i / kStatSlots;
            if (!(ok = warp_wait(&stat_empty[ss], (sr & 1) ^ 1, a.status, kSiteStats))) break;
            // lane l copies words l, l + 32, ... of the slot's [L_i | D_i]: each copy instruction writes 32
            // consecutive words of shared memory (one bank each) from 32 consecutive floats
            const int q0 = (q_begin + i) * kBQ;
            float *dst = stat_s + ss * 2 * kBQ;
#pragma unroll
            for (int e = 0; e < 2 * kBQ / 32; ++e) {
                const int w = 32 * e + lane;
                const bool is_l = e < kBQ / 32;
                const int q = q0 + (is_l ? w : w - kBQ);
                const bool valid = q < N;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst + w)),
                             "l"((is_l ? lse_g : del_g) + (valid ? q : 0)), "r"(valid ? 4 : 0)
                             : "memory");
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&stat_full[ss]))
                         : "memory");
        }
        // Drain: never leave the CTA with a copy still in flight.
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            mbar_wait(kv_full, 0, a.status, kSiteDrain);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
    } else if (warp == 1) {
        // Issuer A: S^T_i = K Q_i^T and dP^T_i = V dO_i^T into buffer i % 2.  The whole warp runs the
        // loop (operands stay warp-uniform); one elected lane issues the MMAs and their commits.
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBN, kBQ, false, false);  // S^T, dP^T: 128 x 64
        const uint64_t k_desc = sdesc_sw128(smem_u32(k_s), 16, 1024);
        const uint64_t v_desc = sdesc_sw128(smem_u32(v_s), 16, 1024);
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = warp_wait(kv_full, 0, a.status, kSiteKV);
        tc_fence_after();
        for (int i = 0; ok && i < n_q; ++i) {
            const int q_slot = (2 * i) % NSLOT, q_round = (2 * i) / NSLOT;
            const int d_slot = (2 * i + 1) % NSLOT, d_round = (2 * i + 1) / NSLOT;
            const uint32_t b = i % NB;
            if (!(ok = warp_wait(&slot_full[q_slot], q_round & 1, a.status, kSiteSlotFull))) break;
            // buffer b last held P^T_{i-NB}, read by dV_{i-NB} (the dK CTA: by the compute warps, done with
            // tile i-NB once dK_{i-NB} was issued)
            if (i >= NB && !(ok = warp_wait(role_dk ? &dk_done[b] : &dv_done[b], ((i - NB) / NB) & 1, a.status,
                                            kSiteDvDone)))
                break;
            tc_fence_after();
            const uint64_t q_desc = sdesc_sw128(slot_addr + q_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tmem + 64 * b, sdesc_add(k_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32),
                           sdesc_add(q_desc, (ks >> 2) * (kBQ * 128) + (ks & 3) * 32), idesc_s, ks > 0);
                mma_commit(&s_full[b]);
            }
            __syncwarp();
            if (role_dv) continue;  // the dV CTA needs no dP^T
            if (!(ok = warp_wait(&slot_full[d_slot], d_round & 1, a.status, kSiteSlotFull))) break;
            // buffer b last held dS^T_{i-NB}, read by dK_{i-NB}
            if (i >= NB && !(ok = warp_wait(&dk_done[b], ((i - NB) / NB) & 1, a.status, kSiteDkDone))) break;
            tc_fence_after();
            const uint64_t do_desc = sdesc_sw128(slot_addr + d_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tmem + kColDP + 64 * b, sdesc_add(v_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32),
                           sdesc_add(do_desc, (ks >> 2) * (kBQ * 128) + (ks & 3) * 32), idesc_s, ks > 0);
                mma_commit(&dp_full[b]);
            }
            __syncwarp();
        }
        // Drain this warp's MMAs before TMEM can be released (immediate in the normal path).
        if (leader) mma_commit(a_final);
        __syncwarp();
        warp_wait(a_final, 0, a.status, kSiteFinal);
    } else if (warp == 2) {
        // Issuer B: dV += P^T dO_i and dK += dS^T Q_i.
        constexpr uint32_t idesc_g = idesc_bf16_f32(kBN, DO, false, true);  // dV, dK: 128 x DO
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = true;
        for (int i = 0; ok && i < n_q; ++i) {
            const uint32_t b = i % NB;
            const int q_slot = (2 * i) % NSLOT, d_slot = (2 * i + 1) % NSLOT;
            // B = this CTA's DO columns of Q_i / dO_i (MN-major: whole 64-column panels from panel do0 / 64 on)
            const uint32_t p0 = (do0 / 64) * (kBQ * 128);
            const uint64_t qmn_desc = sdesc_sw128(slot_addr + q_slot * L::kTileBytes + p0, kBQ * 128, 1024);
            const uint64_t dmn_desc = sdesc_sw128(slot_addr + d_slot * L::kTileBytes + p0, kBQ * 128, 1024);
            if (!role_dk) {
                if (!(ok = warp_wait(&p_ready[b], (i / NB) & 1, a.status, kSitePReady))) break;
                // p_ready only proves S^T_i, hence Q_i, complete: dO_i's copy may still be in flight when the
                // ring is short, so wait for its slot too (normally long since done; the slot cannot refill
                // before this warp's own release after dK_i, so the phase is never two behind)
                if (!(ok = warp_wait(&slot_full[d_slot], ((2 * i + 1) / NSLOT) & 1, a.status, kSiteSlotFull)))
                    break;
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kBQ / 16; ++kk)
                        mma_ts(tmem + kColDV, tmem + 64 * b + (kk / kStepsPerWG) * kSpan + (kk % kStepsPerWG) * 8,
                               sdesc_add(dmn_desc, kk * 2048), idesc_g, (i > 0 || kk > 0));
                    mma_commit(&dv_done[b]);
                    if (role_dv) {
                        // the dV CTA: S^T_i completed before P^T_i was produced, so after dV_i nothing reads
                        // Q_i or dO_i any more
                        mma_commit(&slot_empty[q_slot]);
                        mma_commit(&slot_empty[d_slot]);
                    }
                }
                __syncwarp();
                if (role_dv) continue;
            }
            if (!(ok = warp_wait(&ds_ready[b], (i / NB) & 1, a.status, kSiteDsReady))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_ts(tmem + kColDK,
                           tmem + kColDP + 64 * b + (kk / kStepsPerWG) * kSpan + (kk % kStepsPerWG) * 8,
                           sdesc_add(qmn_desc, kk * 2048), idesc_g, (i > 0 || kk > 0));
                mma_commit(&dk_done[b]);
                // S^T_i and dP^T_i (issuer A) completed before the compute warps produced dS^T_i, so after
                // dK_i nothing reads Q_i or dO_i any more.
                mma_commit(&slot_empty[q_slot]);
                mma_commit(&slot_empty[d_slot]);
            }
            __syncwarp();
        }
        if (leader) mma_commit(final_bar);
        __syncwarp();
        warp_wait(final_bar, 0, a.status, kSiteFinal);
    } else {
        const int quarter = warp & 3;
        const int g = (warp - kFirstComputeWarp) >> 2;  // query range of every tile
        const int r = quarter * 32 + lane;       // key row within the tile (TMEM lane)
        const int key = k_tile * kBN + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float c = a.scale_log2, sc = a.scale;
        constexpr int kHalf = kSpan;  // queries per thread per tile
        bool ok = true;
        for (int i = 0; i < n_q; ++i) {
            const int qt = q_begin + i;
            const int b = i % NB;
            const int ss = i % kStatSlots;
            ok = mbar_wait(&stat_full[ss], (i / kStatSlots) & 1, a.status, kSiteStats);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const float4 *ls4 = reinterpret_cast<const float4 *>(stat_s + ss * 2 * kBQ + g * kHalf);
            const float4 *ds4 = reinterpret_cast<const float4 *>(stat_s + ss * 2 * kBQ + kBQ + g * kHalf);
            const int q0 = qt * kBQ + g * kHalf;  // first query of this thread's half
            // visible iff key <= query (causal), query < N and key < N
            const bool need_mask = (q0 + kHalf > N) || (a.causal && key > q0) || (key >= N);
            const bool any_mask = __any_sync(0xffffffffu, need_mask);

            ok = mbar_wait(&s_full[b], (i / NB) & 1, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // P^T of this thread's queries: bf16 pairs for the dV operand, fp32 pairs kept for dS^T below.
            // The arithmetic runs on fp32 pairs (f32x2), two scores per instruction.
            uint32_t pk[kHalf / 2];
            uint64_t p2[kHalf / 2];
            {
                uint32_t raw[kHalf];
                tmem_ld_n<kHalf>(tmem + lane_base + 64 * b + g * kHalf, raw);
                tmem_wait_ld();
                constexpr float kLog2e = 1.4426950408889634f;
                const uint64_t c2 = f2_pack(c, c), nlog2e2 = f2_pack(-kLog2e, -kLog2e);
#pragma unroll
                for (int q4 = 0; q4 < kHalf / 4; ++q4) {
                    const float4 l4 = ls4[q4];  // natural-log L of four queries
                    float p[4];
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[4 * q4 + 0]), __uint_as_float(raw[4 * q4 + 1])), c2,
                                     f2_mul(f2_pack(l4.x, l4.y), nlog2e2)),
                              p[0], p[1]);
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[4 * q4 + 2]), __uint_as_float(raw[4 * q4 + 3])), c2,
                                     f2_mul(f2_pack(l4.z, l4.w), nlog2e2)),
                              p[2], p[3]);
#pragma unroll
                    for (int t = 0; t < 4; ++t) p[t] = ex2_approx(p[t]);
                    if (any_mask) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int qq = q0 + 4 * q4 + t;
                            if (qq >= N || key >= N || (a.causal && qq < key)) p[t] = 0.f;
                        }
                    }
                    p2[2 * q4] = f2_pack(p[0], p[1]);
                    p2[2 * q4 + 1] = f2_pack(p[2], p[3]);
                    pk[2 * q4] = pack_bf16x2(p[0], p[1]);
                    pk[2 * q4 + 1] = pack_bf16x2(p[2], p[3]);
                }
            }
            tmem_st_n<kHalf / 2>(tmem + lane_base + 64 * b + g * kHalf, pk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&p_ready[b]);
            if (role_dv) {  // the dV CTA computes no dS^T
                warp_arrive(&stat_empty[ss]);
                continue;
            }

            ok = mbar_wait(&dp_full[b], (i / NB) & 1, a.status, kSiteDpFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t raw[kHalf], dsk[kHalf / 2];
                tmem_ld_n<kHalf>(tmem + lane_base + kColDP + 64 * b + g * kHalf, raw);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < kHalf / 4; ++q4) {
                    const float4 d4 = ds4[q4];
                    // dS^T / scale = P^T * (dP^T - D), on fp32 pairs
                    dsk[2 * q4] = f2_to_bf16x2(f2_mul(
                        f2_sub(f2_pack(__uint_as_float(raw[4 * q4 + 0]), __uint_as_float(raw[4 * q4 + 1])),
                               f2_pack(d4.x, d4.y)),
                        p2[2 * q4]));
                    dsk[2 * q4 + 1] = f2_to_bf16x2(f2_mul(
                        f2_sub(f2_pack(__uint_as_float(raw[4 * q4 + 2]), __uint_as_float(raw[4 * q4 + 3])),
                               f2_pack(d4.z, d4.w)),
                        p2[2 * q4 + 1]));
                }
                tmem_st_n<kHalf / 2>(tmem + lane_base + kColDP + 64 * b + g * kHalf, dsk);
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&ds_ready[b]);
            warp_arrive(&stat_empty[ss]);  // this warp has read the tile's L and D
        }
        if (ok) {
            ok = mbar_wait(final_bar, 0, a.status, kSiteDone);
            ok = __all_sync(0xffffffffu, ok);
        }
        // Epilogue: dV and dK (dK times the scale its dS^T operands left out) are staged in the K / V tiles'
        // and the ring's shared memory, which nothing reads any more once every MMA has completed, as
        // 128-byte-swizzled panels of 128 rows (64 bf16 or 32 fp32 columns; dV's panels first), and written
        // by TMA bulk stores that clip rows past N and columns past the caller's D.
        const int n_panels = a.grad_bf16 ? DO / 64 : DO / 32;  // per output
        static_assert((VK ? 1 : 2) * DO * 4 * kBN <= 2 * L::kKVBytes + NSLOT * L::kTileBytes, "staging fits");
        if (ok) {
            tc_fence_after();
            // the first half of the warpgroups writes dV, the second dK; each its share of the D columns
            // (VK: every warpgroup writes its share of the CTA's one gradient, staged from offset 0)
            constexpr int kCols = VK ? DO / kComputeWG : DO / (kComputeWG / 2);
            static_assert(kCols % 32 == 0, "32-column TMEM loads");
            const bool is_dv = VK ? role_dv : g < kComputeWG / 2;
            const int c0 = VK ? g * kCols : (g % (kComputeWG / 2)) * kCols;
            const uint32_t col = (is_dv ? kColDV : kColDK) + c0;
            const float osc = is_dv ? 1.f : sc;  // dK picks up the scale its dS^T operands left out
            uint8_t *stage = smem + ((VK || is_dv) ? 0 : n_panels) * (kBN * 128) + r * 128;
            const int sw = r & 7;
            uint32_t v[32];
#pragma unroll
            for (int ch = 0; ch < kCols / 32; ++ch) {
                tmem_ld32(tmem + lane_base + col + ch * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * osc);
                const int oc = c0 + ch * 32;  // column within this CTA's DO columns
                if (a.grad_bf16) {
                    uint8_t *prow = stage + (oc / 64) * (kBN * 128);
                    const int cb = (oc % 64) / 8;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(prow + (((cb + c) ^ sw) << 4),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1])),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                                     pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
                } else {
                    uint8_t *prow = stage + (oc / 32) * (kBN * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(prow + ((c ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                }
            }
        } else if (lane == 0) {
            epi_abort = 1;
        }
        fence_proxy_async_smem();  // the staged tiles are read by the TMA (async proxy)
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kComputeWG) : "memory");
        if (threadIdx.x == 32 * kFirstComputeWarp && !epi_abort) {
            const int pw = a.grad_bf16 ? 64 : 32;  // panel width in elements
            for (int p = 0; p < n_panels; ++p) {
                if (do0 + p * pw >= Dr) break;  // panels wholly past the caller's D are not stored
                if (!role_dk) tma_store_3d(&tmap_dv, smem + p * (kBN * 128), do0 + p * pw, k_tile * kBN, bh);
                if (!VK) tma_store_3d(&tmap_dk, smem + (n_panels + p) * (kBN * 128), do0 + p * pw, k_tile * kBN, bh);
                if (role_dk) tma_store_3d(&tmap_dk, smem + p * (kBN * 128), do0 + p * pw, k_tile * kBN, bh);
            }
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

template <int D, int DO, int NB, int NSLOT, int STATS, bool VK = false>
cudaError_t launch_spec(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv, cudaStream_t s) {
    using L = DkdvSmem<D, NSLOT, STATS>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    auto kern = bwd_dkdv_kernel<D, DO, NB, NSLOT, STATS, VK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBN - 1) / kBN) * a.H * a.B, VK ? 2 : D / DO);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, tdo, tdk, tdv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv, cudaStream_t s) {
    switch (kernel_head_dim(a.D)) {
        case 128: return launch_spec<128, 128, 2, 8, 4>(a, tq, tk, tv, tdo, tdk, tdv, s);
        case 192: return launch_spec<192, 192, 1, 5, 4>(a, tq, tk, tv, tdo, tdk, tdv, s);
        case 256: return launch_spec<256, 256, 2, 3, 3, true>(a, tq, tk, tv, tdo, tdk, tdv, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
