// bwd_atomic.cu -- a 5-GEMM backward with accumulated dQ, the comparator for
// the atomic-free split backward.  The metal-flash-attention page explains
// the split (one dQ kernel, one dK/dV kernel, 7 GEMMs) by Apple GPUs'
// missing fp32 atomics; the conventional backward instead recomputes S and
// dP once per (key tile, query tile) pair and accumulates dQ across key tiles.
// GB300 has fp32 reductions in L2, so this file builds that design to measure
// the trade-off:
//
//   delta_kernel   D_i = rowsum(dO_i * O_i)
//   bwd_atomic_kernel, one CTA per 128-key tile of one (batch, head), per
//   64-query tile i:   S^T = K Q_i^T,  P^T = 2^(S^T c - L_i),  dV += P^T dO_i,
//                      dP^T = V dO_i^T,  dS^T = P^T * (dP^T - D_i) * scale,
//                      dK += dS^T Q_i,
//                      dQ_i^T = K^T dS^T  (the fifth GEMM, M = D rows of K^T),
//   and dQ_i is added into an fp32 accumulator in global memory with one bulk
//   reduce-add per tile (cp.reduce.async.bulk ... .add.f32: the L2 performs
//   the additions);
//   dq_convert_kernel  dQ = the accumulator in the gradient dtype.
//
// The kernel is bwd_dkdv.cu's pipeline (warp 0 TMA; warp 1 issues S^T, dP^T;
// warp 2 issues dV, dK and dQ^T; warps 3-10 compute, a thread per key row and
// half the tile's queries) with these changes:
// - TMEM (D = 128): S^T[b] [64b, 64b+64) double-buffered, dP^T [128, 192)
//   single-buffered, dQ^T [192, 256), dV [256, 384), dK [384, 512).  dP^T(i+1)
//   therefore waits for dK(i), which read dS^T(i) from those columns.
// - dS^T is also stored to shared memory (MN-major, 128-byte swizzle) as the
//   B operand of dQ^T; K^T is the K tile read MN-major (the same bytes).
// - After dQ^T(i) completes, the compute threads (lane = d, warpgroup = query
//   half) copy it to a [64][D] fp32 staging tile, and one thread issues the
//   bulk reduce-add of the tile's valid rows, waits until the tile has been
//   read, and frees it.
// Head dimension 128 only: dQ^T's M is D, and M = 64 accumulators have
// another TMEM layout.
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBN = 128;          // keys per CTA (TMEM lanes)
constexpr int kBQ = kDkdvQRows;   // queries per tile (64)
constexpr int kComputeWG = 2;     // compute warpgroups, one query half each
constexpr int kFirstComputeWarp = 3;
constexpr int kThreads = 32 * kFirstComputeWarp + 128 * kComputeWG;

enum : int { kSiteKV = 101, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePReady, kSiteDpFull, kSiteDsReady,
             kSiteDone, kSiteFinal, kSiteDrain, kSiteStats, kSiteDvDone, kSiteDkDone, kSiteDqFull, kSiteDqFree,
             kSiteTileFull, kSiteTileFree };

__device__ __forceinline__ void bulk_reduce_add_f32(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int D, int NSLOT>
struct AtomicSmem {
    static constexpr int kKVBytes = kBN * D * 2;
    static constexpr int kTileBytes = kBQ * D * 2;  // one Q_i or dO_i tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKVBytes;
    static constexpr int kSlotOff = 2 * kKVBytes;
    static constexpr int kDsOff = kSlotOff + NSLOT * kTileBytes;  // dS^T, 128 keys x 64 queries bf16
    static constexpr int kDqOff = kDsOff + kBN * kBQ * 2;         // dQ staging, 64 x D fp32
    static constexpr int kStatOff = kDqOff + kBQ * D * 4;         // lse2[2][kBQ], delta[2][kBQ]
    static constexpr int kBarOff = kStatOff + 4 * kBQ * 4;
    // kv_full, slot_full[NSLOT], slot_empty[NSLOT], s_full[2], dp_full, p_ready[2], ds_ready, stats[2],
    // dv_done[2], dk_done, dq_full, dq_free, tile_full, tile_free, final, a_final
    static constexpr int kNumBars = 1 + 2 * NSLOT + 17;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

template <int D, int NSLOT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_atomic_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                      BwdArgs a) {
    using L = AtomicSmem<D, NSLOT>;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kTmemCols = 512;
    constexpr uint32_t kColDP = 128, kColDQ = 192, kColDV = 256, kColDK = 256 + D;
    static_assert(D == 128, "dQ^T uses M = D = 128");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *k_s = smem + L::kKOff;
    uint8_t *v_s = smem + L::kVOff;
    uint8_t *slots = smem + L::kSlotOff;
    uint8_t *ds_s = smem + L::kDsOff;
    float *dq_s = reinterpret_cast<float *>(smem + L::kDqOff);
    float *lse_s = reinterpret_cast<float *>(smem + L::kStatOff);  // [2][kBQ], already times log2(e)
    float *del_s = lse_s + 2 * kBQ;                                 // [2][kBQ]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + NSLOT;
    uint64_t *s_full = slot_empty + NSLOT;  // [2]
    uint64_t *dp_full = s_full + 2;
    uint64_t *p_ready = dp_full + 1;        // [2]
    uint64_t *ds_ready = p_ready + 2;       // dS^T(i) in TMEM and in shared memory
    uint64_t *stats_bar = ds_ready + 1;     // [2]
    // dV_i complete, one barrier per S^T buffer b = i % 2: issuer A waits for tile i - 2 while dV_{i-1}
    // may already have completed, and on a single barrier that later phase would carry the parity it
    // waits for.
    uint64_t *dv_done = stats_bar + 2;      // [2]
    uint64_t *dk_done = dv_done + 2;
    uint64_t *dq_full = dk_done + 1;        // dQ^T(i) complete (it has also read dS^T(i) from shared memory)
    uint64_t *dq_free = dq_full + 1;        // every compute warp has read dQ^T(i) out of TMEM
    uint64_t *tile_full = dq_free + 1;      // the staging tile holds dQ_i
    uint64_t *tile_free = tile_full + 1;    // the bulk reduce-add has read the staging tile
    uint64_t *final_bar = tile_free + 1;    // issuer B: every dV / dK / dQ^T MMA has completed
    uint64_t *a_final = final_bar + 1;      // issuer A: every S^T / dP^T MMA has completed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    tile_order((a.N + kBN - 1) / kBN, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int k_tile = rank;  // causal: key tile 0 has the most query tiles
    const int N = a.N;
    const int n_q_total = (N + kBQ - 1) / kBQ;
    const int q_begin = a.causal ? (k_tile * kBN) / kBQ : 0;
    const int n_q = n_q_total - q_begin;  // >= 1

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_ready[b], 4 * kComputeWG);  // one arrive per compute warp
            mbar_init(&stats_bar[b], 4 * kComputeWG);
        }
        mbar_init(dp_full, 1);
        mbar_init(ds_ready, 4 * kComputeWG);
        mbar_init(&dv_done[0], 1);
        mbar_init(&dv_done[1], 1);
        mbar_init(dk_done, 1);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 4 * kComputeWG);
        mbar_init(tile_full, 4 * kComputeWG);
        mbar_init(tile_free, 1);
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
            int last_round[NSLOT];
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) last_round[s] = -1;
            for (int idx = 0; idx < 2 * n_q; ++idx) {
                const int slot = idx % NSLOT, round = idx / NSLOT;
                if (!mbar_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty)) break;
                uint8_t *dst = slots + slot * L::kTileBytes;
                const CUtensorMap *map = (idx & 1) ? &tmap_do : &tmap_q;
                mbar_arrive_expect_tx(&slot_full[slot], L::kTileBytes);
#pragma unroll
                for (int p = 0; p < kPanels; ++p)
                    tma_load_3d(dst + p * (kBQ * 128), map, &slot_full[slot], p * 64, (q_begin + (idx >> 1)) * kBQ,
                                bh);
#pragma unroll
                for (int s = 0; s < NSLOT; ++s)
                    if (s == slot) last_round[s] = round;
            }
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            mbar_wait(kv_full, 0, a.status, kSiteDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // Issuer A: S^T_i = K Q_i^T into S^T[i % 2], dP^T_i = V dO_i^T into the single dP^T buffer.
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
            const uint32_t b = i & 1;
            if (!(ok = warp_wait(&slot_full[q_slot], q_round & 1, a.status, kSiteSlotFull))) break;
            // S^T[b] last held P^T_{i-2}, read by dV_{i-2}
            if (i >= 2 && !(ok = warp_wait(&dv_done[b], ((i - 2) >> 1) & 1, a.status, kSiteDvDone))) break;
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
            if (!(ok = warp_wait(&slot_full[d_slot], d_round & 1, a.status, kSiteSlotFull))) break;
            // the dP^T columns last held dS^T_{i-1}, read by dK_{i-1}
            if (i >= 1 && !(ok = warp_wait(dk_done, (i - 1) & 1, a.status, kSiteDkDone))) break;
            tc_fence_after();
            const uint64_t do_desc = sdesc_sw128(slot_addr + d_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tmem + kColDP, sdesc_add(v_desc, (ks >> 2) * (kBN * 128) + (ks & 3) * 32),
                           sdesc_add(do_desc, (ks >> 2) * (kBQ * 128) + (ks & 3) * 32), idesc_s, ks > 0);
                mma_commit(dp_full);
            }
            __syncwarp();
        }
        if (leader) mma_commit(a_final);
        __syncwarp();
        warp_wait(a_final, 0, a.status, kSiteFinal);
    } else if (warp == 2) {
        // Issuer B: dV += P^T dO_i, dK += dS^T Q_i, dQ^T_i = K^T dS^T.
        constexpr uint32_t idesc_g = idesc_bf16_f32(kBN, D, false, true);  // dV, dK: 128 x D
        constexpr uint32_t idesc_q = idesc_bf16_f32(D, kBQ, true, true);   // dQ^T: D x 64, both MN-major
        const uint32_t slot_addr = smem_u32(slots);
        // K^T as the MN-major A operand (M = d, contiguous within a 64-column panel; K = key rows)
        const uint64_t kt_desc = sdesc_sw128(smem_u32(k_s), kBN * 128, 1024);
        // dS^T as the MN-major B operand (N = query, one 64-wide panel; K = key rows)
        const uint64_t ds_desc = sdesc_sw128(smem_u32(ds_s), kBN * 128, 1024);
        const bool leader = elect_one();
        bool ok = true;
        for (int i = 0; ok && i < n_q; ++i) {
            const uint32_t b = i & 1;
            const int q_slot = (2 * i) % NSLOT, d_slot = (2 * i + 1) % NSLOT;
            const uint64_t qmn_desc = sdesc_sw128(slot_addr + q_slot * L::kTileBytes, kBQ * 128, 1024);
            const uint64_t dmn_desc = sdesc_sw128(slot_addr + d_slot * L::kTileBytes, kBQ * 128, 1024);
            if (!(ok = warp_wait(&p_ready[b], (i >> 1) & 1, a.status, kSitePReady))) break;
            // p_ready only proves S^T_i, hence Q_i, complete: wait for dO_i's copy as well (normally long
            // since done; its slot cannot refill before this warp's own release after dK_i)
            if (!(ok = warp_wait(&slot_full[d_slot], ((2 * i + 1) / NSLOT) & 1, a.status, kSiteSlotFull))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_ts(tmem + kColDV, tmem + 64 * b + (kk >> 1) * 32 + (kk & 1) * 8,
                           sdesc_add(dmn_desc, kk * 2048), idesc_g, (i > 0 || kk > 0));
                mma_commit(&dv_done[b]);
            }
            __syncwarp();
            if (!(ok = warp_wait(ds_ready, i & 1, a.status, kSiteDsReady))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_ts(tmem + kColDK, tmem + kColDP + (kk >> 1) * 32 + (kk & 1) * 8,
                           sdesc_add(qmn_desc, kk * 2048), idesc_g, (i > 0 || kk > 0));
                mma_commit(dk_done);
                mma_commit(&slot_empty[q_slot]);
                mma_commit(&slot_empty[d_slot]);
            }
            __syncwarp();
            // dQ^T(i) overwrites dQ^T(i-1), which the compute warps must have read
            if (i >= 1 && !(ok = warp_wait(dq_free, (i - 1) & 1, a.status, kSiteDqFree))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ss(tmem + kColDQ, sdesc_add(kt_desc, kk * 2048), sdesc_add(ds_desc, kk * 2048), idesc_q,
                           kk > 0);
                mma_commit(dq_full);
            }
            __syncwarp();
        }
        if (leader) mma_commit(final_bar);
        __syncwarp();
        warp_wait(final_bar, 0, a.status, kSiteFinal);
    } else {
        const int quarter = warp & 3;
        const int g = (warp - kFirstComputeWarp) >> 2;           // query half of every tile
        const int tid = (warp - kFirstComputeWarp) * 32 + lane;  // 0..255; 0..127 load the stats
        const int r = quarter * 32 + lane;  // key row within the tile (TMEM lane); for dQ^T: the column d
        const int key = k_tile * kBN + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float c = a.scale_log2, sc = a.scale;
        const float *lse_g = a.lse + (size_t)bh * N;
        const float *del_g = a.delta + (size_t)bh * N;
        constexpr int kHalf = kBQ / kComputeWG;  // 32 queries per thread per tile
        const bool carries = tid < 2 * kBQ;
        const bool carries_lse = tid < kBQ;
        const int stat_q = carries_lse ? tid : tid - kBQ;
        const bool reducer = tid == 0;  // issues the bulk reduce-add of every staging tile
        float *dq_acc = static_cast<float *>(a.dq);
        auto load_stat = [&](int q_tile_idx) -> float {
            if (!carries) return 0.f;
            const int qi = q_tile_idx * kBQ + stat_q;
            if (carries_lse) return qi < N ? lse_g[qi] * 1.4426950408889634f : INFINITY;
            return qi < N ? del_g[qi] : 0.f;
        };
        auto store_stat = [&](int buf, float v) {
            if (!carries) return;
            if (carries_lse)
                lse_s[buf * kBQ + stat_q] = v;
            else
                del_s[buf * kBQ + stat_q] = v;
        };
        bool ok = true;
        store_stat(0, load_stat(q_begin));
        warp_arrive(&stats_bar[0]);
        for (int i = 0; i < n_q; ++i) {
            const int qt = q_begin + i;
            const int b = i & 1;
            const float nxt = (i + 1 < n_q) ? load_stat(qt + 1) : 0.f;  // prefetch; published at the end
            ok = mbar_wait(&stats_bar[b], (i >> 1) & 1, a.status, kSiteStats);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const float4 *ls4 = reinterpret_cast<const float4 *>(lse_s + b * kBQ + g * kHalf);
            const float4 *ds4 = reinterpret_cast<const float4 *>(del_s + b * kBQ + g * kHalf);
            const int q0 = qt * kBQ + g * kHalf;  // first query of this thread's half
            const bool need_mask = (q0 + kHalf > N) || (a.causal && key > q0) || (key >= N);
            const bool any_mask = __any_sync(0xffffffffu, need_mask);

            ok = mbar_wait(&s_full[b], (i >> 1) & 1, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // P^T row half as bf16 pairs: the dV operand, and (unpacked) the factor of dS^T below.
            uint32_t pk[kHalf / 2];
            {
                uint32_t raw[kHalf];
                tmem_ld32(tmem + lane_base + 64 * b + g * kHalf, raw);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < kHalf / 4; ++q4) {
                    const float4 l4 = ls4[q4];
                    float p[4];
                    p[0] = ex2_approx(fmaf(__uint_as_float(raw[4 * q4 + 0]), c, -l4.x));
                    p[1] = ex2_approx(fmaf(__uint_as_float(raw[4 * q4 + 1]), c, -l4.y));
                    p[2] = ex2_approx(fmaf(__uint_as_float(raw[4 * q4 + 2]), c, -l4.z));
                    p[3] = ex2_approx(fmaf(__uint_as_float(raw[4 * q4 + 3]), c, -l4.w));
                    if (any_mask) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int qq = q0 + 4 * q4 + t;
                            if (qq >= N || key >= N || (a.causal && qq < key)) p[t] = 0.f;
                        }
                    }
                    pk[2 * q4] = pack_bf16x2(p[0], p[1]);
                    pk[2 * q4 + 1] = pack_bf16x2(p[2], p[3]);
                }
            }
            tmem_st16(tmem + lane_base + 64 * b + g * kHalf, pk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&p_ready[b]);

            ok = mbar_wait(dp_full, i & 1, a.status, kSiteDpFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t raw[kHalf], dsk[kHalf / 2];
                tmem_ld32(tmem + lane_base + kColDP + g * kHalf, raw);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < kHalf / 4; ++q4) {
                    const float4 d4 = ds4[q4];
                    const float2 p01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pk[2 * q4]));
                    const float2 p23 =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pk[2 * q4 + 1]));
                    const float d0 = p01.x * (__uint_as_float(raw[4 * q4 + 0]) - d4.x) * sc;
                    const float d1 = p01.y * (__uint_as_float(raw[4 * q4 + 1]) - d4.y) * sc;
                    const float d2 = p23.x * (__uint_as_float(raw[4 * q4 + 2]) - d4.z) * sc;
                    const float d3 = p23.y * (__uint_as_float(raw[4 * q4 + 3]) - d4.w) * sc;
                    dsk[2 * q4] = pack_bf16x2(d0, d1);
                    dsk[2 * q4 + 1] = pack_bf16x2(d2, d3);
                }
                tmem_st16(tmem + lane_base + kColDP + g * kHalf, dsk);
                // dS^T row r, queries [32g, 32g+32) = 16-byte chunks 4g..4g+3 of the 128-byte row, stored at
                // chunk ^ (r % 8) (128-byte swizzle); dQ^T(i-1) has read the previous tile (dq_full(i-1))
                uint4 *row_s = reinterpret_cast<uint4 *>(ds_s + r * 128);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    row_s[(4 * g + u) ^ (r & 7)] = make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
            }
            tmem_wait_st();
            fence_proxy_async_smem();  // the shared-memory dS^T is read by the tensor core
            tc_fence_before();
            warp_arrive(ds_ready);
            if (i + 1 < n_q) {
                store_stat(b ^ 1, nxt);
                warp_arrive(&stats_bar[b ^ 1]);
            }

            // dQ_i: TMEM lane = d, column = query; this warpgroup copies its 32 queries to the staging tile
            ok = mbar_wait(dq_full, i & 1, a.status, kSiteDqFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t qv[kHalf];
            tmem_ld32(tmem + lane_base + kColDQ + g * kHalf, qv);
            tmem_wait_ld();
            tc_fence_before();
            warp_arrive(dq_free);
            if (i >= 1) {
                ok = mbar_wait(tile_free, (i - 1) & 1, a.status, kSiteTileFree);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            }
#pragma unroll
            for (int j = 0; j < kHalf; ++j) dq_s[(g * kHalf + j) * D + r] = __uint_as_float(qv[j]);
            fence_proxy_async_smem();  // the staging tile is read by the bulk copy engine
            warp_arrive(tile_full);
            if (reducer) {
                ok = mbar_wait(tile_full, i & 1, a.status, kSiteTileFull);
                if (ok) {
                    const int rows = min(kBQ, N - qt * kBQ);
                    bulk_reduce_add_f32(dq_acc + ((size_t)bh * N + (size_t)qt * kBQ) * D, dq_s,
                                        (uint32_t)(rows * D * 4));
                    bulk_commit();
                    bulk_wait_read_all();
                    mbar_arrive(tile_free);
                }
            }
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        if (reducer) bulk_wait_all();  // every reduce-add has been performed before the CTA ends
        if (ok) {
            ok = mbar_wait(final_bar, 0, a.status, kSiteDone);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const bool valid = key < N;
            // warpgroup 0 writes dV, warpgroup 1 writes dK
            const uint32_t col = g == 0 ? kColDV : kColDK;
            void *outp = g == 0 ? a.dv : a.dk;
            uint32_t v[32];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                tmem_ld32(tmem + lane_base + col + ch * 32, v);
                tmem_wait_ld();
                if (!valid) continue;
                if (a.grad_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(outp) +
                                                           ((size_t)bh * N + key) * D + ch * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[v4 * 8 + 0]), __uint_as_float(v[v4 * 8 + 1]));
                        w.y = pack_bf16x2(__uint_as_float(v[v4 * 8 + 2]), __uint_as_float(v[v4 * 8 + 3]));
                        w.z = pack_bf16x2(__uint_as_float(v[v4 * 8 + 4]), __uint_as_float(v[v4 * 8 + 5]));
                        w.w = pack_bf16x2(__uint_as_float(v[v4 * 8 + 6]), __uint_as_float(v[v4 * 8 + 7]));
                        dst[v4] = w;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(outp) +
                                                             ((size_t)bh * N + key) * D + ch * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 8; ++v4)
                        dst[v4] = make_float4(__uint_as_float(v[v4 * 4 + 0]), __uint_as_float(v[v4 * 4 + 1]),
                                              __uint_as_float(v[v4 * 4 + 2]), __uint_as_float(v[v4 * 4 + 3]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// D_i = sum_d dO_id O_id, one warp per row (bf16 inputs, fp32 sum).
template <int D>
__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16 *o, const __nv_bfloat16 *dO, float *delta,
                                                    long long rows) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    constexpr int kPer = D / 32;  // elements per lane (4 for D = 128)
    const __nv_bfloat16 *orow = o + row * D + lane * kPer;
    const __nv_bfloat16 *drow = dO + row * D + lane * kPer;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(orow + e));
        const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(drow + e));
        s = fmaf(of.x, df.x, s);
        s = fmaf(of.y, df.y, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) delta[row] = s;
}

// dQ = the fp32 accumulator in the gradient dtype, four elements per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float *acc, void *dq, long long n4, int to_bf16) {
    const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
    if (i >= n4) return;
    const float4 v = reinterpret_cast<const float4 *>(acc)[i];
    if (to_bf16) {
        uint2 w;
        w.x = pack_bf16x2(v.x, v.y);
        w.y = pack_bf16x2(v.z, v.w);
        reinterpret_cast<uint2 *>(dq)[i] = w;
    } else {
        reinterpret_cast<float4 *>(dq)[i] = v;
    }
}

}  // namespace

cudaError_t launch_bwd_atomic(const BwdArgs &a, void *dq_out, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t s) {
    if (a.D != 128) return cudaErrorInvalidValue;
    constexpr int D = 128, NSLOT = 6;
    using L = AtomicSmem<D, NSLOT>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    const long long rows = (long long)a.B * a.H * a.N;
    cudaError_t e = cudaMemsetAsync(a.dq, 0, (size_t)rows * D * sizeof(float), s);
    if (e != cudaSuccess) return e;
    delta_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(a.o),
                                                               static_cast<const __nv_bfloat16 *>(a.dO), a.delta,
                                                               rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kern = bwd_atomic_kernel<D, NSLOT>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBN - 1) / kBN) * a.H * a.B);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, tdo, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long n4 = rows * D / 4;
    dq_convert_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(static_cast<const float *>(a.dq), dq_out, n4,
                                                                   a.grad_bf16);
    return cudaGetLastError();
}

}  // namespace fa
