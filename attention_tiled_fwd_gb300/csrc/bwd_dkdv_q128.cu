// bwd_dkdv_q128.cu -- the dK/dV kernel of the split backward for D = 64, with
// 128-row query tiles.  Same computation as bwd_dkdv.cu ("backward key-value"
// of the metal-flash-attention page's pseudocode): one CTA per 128-key tile
// of one (batch, head), iterating over query tiles,
//
//   S^T = K Q_i^T,  P^T = exp(S^T scale - L_i) (base 2 here),  dV += P^T dO_i,
//   dP^T = V dO_i^T,  dS^T = P^T * (dP^T - D_i),  dK += dS^T Q_i,
//
// dK (times the softmax scale, left out of every dS^T) and dV written once at
// the end; causal: only query tiles on or below the diagonal are visited.
//
// Why a separate kernel: at D = 64 the 64-query tiles of bwd_dkdv.cu make every
// product an N = 64 MMA, which the tensor core runs at about 60 % of its rate
// (a clock64 trace shows ~54 instead of 32 cycles per 128 x 64 x 16 step).
// With 128-query tiles the S^T and dP^T products are N = 128.  TMEM then holds
// S^T twice (2 x 128 columns), dP^T once (128) and dV, dK (64 each):
//   - P^T (bf16) is written over the first half of each warpgroup's own S^T
//     columns and dS^T over the second half, so S^T_{i+2} waits for dK_i (which
//     issuer B issues after dV_i, so its commit covers both);
//   - dP^T is single-buffered: every compute warp loads its dP^T columns into
//     registers first thing and releases the buffer (dp_free), so dP^T_{i+1}
//     runs while the compute warps work on tile i.
// Roles: warp 0 TMA producer (K, V once; 128-row Q_i, dO_i through a ring) and,
// as a whole warp, the L_i / D_i ring (4-byte cp.async, zero fill past N);
// warp 1 issuer A (S^T, dP^T); warp 2 issuer B (dV, dK); warps 3-18 compute:
// four warpgroups, warpgroup g owning queries [32g, 32g+32) of every tile, a
// thread owning one key row (its TMEM lane).
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kD = 64;
constexpr int kBN = 128;          // keys per CTA (TMEM lanes)
constexpr int kBQ = 128;          // queries per tile
constexpr int kComputeWG = 4;
constexpr int kSpan = kBQ / kComputeWG;  // 32 queries per compute thread per tile
constexpr int kFirstComputeWarp = 3;
constexpr int kThreads = 32 * kFirstComputeWarp + 128 * kComputeWG;
constexpr int kComputeWarps = 4 * kComputeWG;
constexpr int kStatSlots = 2;     // query tiles' L / D in flight (1, 3 and 4 slots measured 1-36 % slower)
constexpr int kNSlot = 9;         // Q_i / dO_i ring (8 slots measured 0.3-1.8 % slower at N = 32768, 10 and 11 no faster)

enum : int { kSiteKV = 81, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePReady, kSiteDpFull, kSiteDsReady,
             kSiteDone, kSiteFinal, kSiteDrain, kSiteStats, kSiteDkDone, kSiteDpFree };

struct Q128Smem {
    static constexpr int kKVBytes = kBN * kD * 2;
    static constexpr int kTileBytes = kBQ * kD * 2;  // one Q_i or dO_i tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKVBytes;
    static constexpr int kSlotOff = 2 * kKVBytes;
    static constexpr int kStatOff = kSlotOff + kNSlot * kTileBytes;  // [kStatSlots][L kBQ | D kBQ] fp32
    static constexpr int kBarOff = kStatOff + kStatSlots * 2 * kBQ * 4;
    // kv_full, slot_full[kNSlot], slot_empty[kNSlot], s_full[2], p_ready[2], ds_ready[2], dk_done[2], dp_full,
    // dp_free, stat_full[kStatSlots], stat_empty[kStatSlots], final, a_final
    static constexpr int kNumBars = 1 + 2 * kNSlot + 8 + 2 + 2 * kStatSlots + 2;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_q128_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                         const __grid_constant__ CUtensorMap tmap_dk, const __grid_constant__ CUtensorMap tmap_dv,
                         BwdArgs a) {
    using L = Q128Smem;
    constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S^T[b] = [128b, 128b + 128), dP^T = [256, 384), dV = [384, 448), dK = [448, 512).
    // Warpgroup g's queries sit at columns 32g.. of each 128-column score buffer; its P^T (bf16) goes to
    // [128b + 32g, +16) and its dS^T to [128b + 32g + 16, +16), so 16-query k-step kk of the dV (dK)
    // product reads column 128b + 32 (kk / 2) + 8 (kk % 2) (+ 16).
    constexpr uint32_t kColDP = 256, kColDV = 384, kColDK = 448;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *k_s = smem + L::kKOff;
    uint8_t *v_s = smem + L::kVOff;
    uint8_t *slots = smem + L::kSlotOff;
    float *stat_s = reinterpret_cast<float *>(smem + L::kStatOff);  // slot s: L at [2 kBQ s], D after it
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + kNSlot;
    uint64_t *s_full = slot_empty + kNSlot;  // [2]: S^T_i complete
    uint64_t *p_ready = s_full + 2;          // [2]: P^T_i written
    uint64_t *ds_ready = p_ready + 2;        // [2]: dS^T_i written
    uint64_t *dk_done = ds_ready + 2;        // [2]: dK_i (and dV_i) complete: S^T buffer i % 2 is free
    uint64_t *dp_full = dk_done + 2;         // dP^T_i complete (phase i)
    uint64_t *dp_free = dp_full + 1;         // every compute warp has loaded dP^T_i (phase i)
    uint64_t *stat_full = dp_free + 1;             // [kStatSlots]: a query tile's L / D landed
    uint64_t *stat_empty = stat_full + kStatSlots;  // [kStatSlots]: every compute warp is done with it
    uint64_t *final_bar = stat_empty + kStatSlots;  // issuer B: every dV / dK MMA has completed
    uint64_t *a_final = final_bar + 1;              // issuer A: every S^T / dP^T MMA has completed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    __shared__ int epi_abort;  // a compute warp's wait ran out: the epilogue stores nothing
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    tile_order((a.N + kBN - 1) / kBN, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int k_tile = rank;  // causal: key tile 0 has the most query tiles
    const int N = a.N;
    const int n_q_total = (N + kBQ - 1) / kBQ;
    const int q_begin = a.causal ? k_tile : 0;  // kBQ == kBN
    const int n_q = n_q_total - q_begin;       // >= 1

    if (threadIdx.x == 0) {
        epi_abort = 0;
        mbar_init(kv_full, 1);
        for (int s = 0; s < kNSlot; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_ready[b], kComputeWarps);  // one arrive per compute warp
            mbar_init(&ds_ready[b], kComputeWarps);
            mbar_init(&dk_done[b], 1);
        }
        mbar_init(dp_full, 1);
        mbar_init(dp_free, kComputeWarps);
        for (int t = 0; t < kStatSlots; ++t) {
            mbar_init(&stat_full[t], 32);  // one arrival per producer lane, when its copies have landed
            mbar_init(&stat_empty[t], kComputeWarps);
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
            tma_load_3d(k_s, &tmap_k, kv_full, 0, k_tile * kBN, bh);
            tma_load_3d(v_s, &tmap_v, kv_full, 0, k_tile * kBN, bh);
        }
        const float *lse_g = a.lse + (size_t)bh * N;
        const float *del_g = a.delta + (size_t)bh * N;
        int last_round[kNSlot];
#pragma unroll
        for (int s = 0; s < kNSlot; ++s) last_round[s] = -1;
        bool ok = true;
        for (int idx = 0; ok && idx < 2 * n_q; ++idx) {
            const int slot = idx % kNSlot, round = idx / kNSlot;
            if (!(ok = warp_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty))) break;
            if (lane == 0) {
                const CUtensorMap *map = (idx & 1) ? &tmap_do : &tmap_q;
                mbar_arrive_expect_tx(&slot_full[slot], L::kTileBytes);
                tma_load_3d(slots + slot * L::kTileBytes, map, &slot_full[slot], 0, (q_begin + (idx >> 1)) * kBQ, bh);
            }
#pragma unroll
            for (int s = 0; s < kNSlot; ++s)
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
            for (int s = 0; s < kNSlot; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            mbar_wait(kv_full, 0, a.status, kSiteDrain);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
    } else if (warp == 1) {
        // Issuer A: S^T_i = K Q_i^T into buffer i % 2 and dP^T_i = V dO_i^T into the one dP^T buffer.
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBN, kBQ, false, false);  // 128 x 128
        const uint64_t k_desc = sdesc_sw128(smem_u32(k_s), 16, 1024);
        const uint64_t v_desc = sdesc_sw128(smem_u32(v_s), 16, 1024);
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = warp_wait(kv_full, 0, a.status, kSiteKV);
        tc_fence_after();
        for (int i = 0; ok && i < n_q; ++i) {
            const int q_slot = (2 * i) % kNSlot, q_round = (2 * i) / kNSlot;
            const int d_slot = (2 * i + 1) % kNSlot, d_round = (2 * i + 1) / kNSlot;
            const uint32_t b = i & 1;
            if (!(ok = warp_wait(&slot_full[q_slot], q_round & 1, a.status, kSiteSlotFull))) break;
            // buffer b last held P^T and dS^T of tile i-2, read by its dV and dK products
            if (i >= 2 && !(ok = warp_wait(&dk_done[b], ((i - 2) >> 1) & 1, a.status, kSiteDkDone))) break;
            tc_fence_after();
            const uint64_t q_desc = sdesc_sw128(slot_addr + q_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_ss(tmem + 128 * b, sdesc_add(k_desc, ks * 32), sdesc_add(q_desc, ks * 32), idesc_s, ks > 0);
                mma_commit(&s_full[b]);
            }
            __syncwarp();
            if (!(ok = warp_wait(&slot_full[d_slot], d_round & 1, a.status, kSiteSlotFull))) break;
            // the dP^T buffer last held tile i-1's, which every compute warp has loaded
            if (i >= 1 && !(ok = warp_wait(dp_free, (i - 1) & 1, a.status, kSiteDpFree))) break;
            tc_fence_after();
            const uint64_t do_desc = sdesc_sw128(slot_addr + d_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_ss(tmem + kColDP, sdesc_add(v_desc, ks * 32), sdesc_add(do_desc, ks * 32), idesc_s, ks > 0);
                mma_commit(dp_full);
            }
            __syncwarp();
        }
        // Drain this warp's MMAs before TMEM can be released (immediate in the normal path).
        if (leader) mma_commit(a_final);
        __syncwarp();
        warp_wait(a_final, 0, a.status, kSiteFinal);
    } else if (warp == 2) {
        // Issuer B: dV += P^T dO_i and dK += dS^T Q_i (dO_i, Q_i as MN-major B operands: queries are the
        // reduction).
        constexpr uint32_t idesc_g = idesc_bf16_f32(kBN, kD, false, true);  // 128 x 64
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = true;
        for (int i = 0; ok && i < n_q; ++i) {
            const uint32_t b = i & 1;
            const int q_slot = (2 * i) % kNSlot, d_slot = (2 * i + 1) % kNSlot;
            const uint64_t qmn_desc = sdesc_sw128(slot_addr + q_slot * L::kTileBytes, kBQ * 128, 1024);
            const uint64_t dmn_desc = sdesc_sw128(slot_addr + d_slot * L::kTileBytes, kBQ * 128, 1024);
            if (!(ok = warp_wait(&p_ready[b], (i >> 1) & 1, a.status, kSitePReady))) break;
            // p_ready only proves S^T_i, hence Q_i, complete: wait for dO_i's copy as well (normally long
            // since done; its slot cannot refill before this warp's own release after dK_i)
            if (!(ok = warp_wait(&slot_full[d_slot], ((2 * i + 1) / kNSlot) & 1, a.status, kSiteSlotFull))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_ts(tmem + kColDV, tmem + 128 * b + 32 * (kk >> 1) + 8 * (kk & 1),
                           sdesc_add(dmn_desc, kk * 2048), idesc_g, (i > 0 || kk > 0));
            }
            __syncwarp();
            if (!(ok = warp_wait(&ds_ready[b], (i >> 1) & 1, a.status, kSiteDsReady))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_ts(tmem + kColDK, tmem + 128 * b + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                           sdesc_add(qmn_desc, kk * 2048), idesc_g, (i > 0 || kk > 0));
                // covers dV_i as well (a commit tracks every earlier MMA of this thread)
                mma_commit(&dk_done[b]);
                // S^T_i and dP^T_i completed before the compute warps produced dS^T_i, so after dK_i nothing
                // reads Q_i or dO_i any more.
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
        const int r = quarter * 32 + lane;               // key row within the tile (TMEM lane)
        const int key = k_tile * kBN + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float c = a.scale_log2, sc = a.scale;
        constexpr float kLog2e = 1.4426950408889634f;
        const uint64_t c2 = f2_pack(c, c), nlog2e2 = f2_pack(-kLog2e, -kLog2e);
        bool ok = true;
        for (int i = 0; i < n_q; ++i) {
            const int qt = q_begin + i;
            const uint32_t b = i & 1;
            const int ss = i % kStatSlots;
            ok = mbar_wait(&stat_full[ss], (i / kStatSlots) & 1, a.status, kSiteStats);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const float4 *ls4 = reinterpret_cast<const float4 *>(stat_s + ss * 2 * kBQ + g * kSpan);
            const float4 *ds4 = reinterpret_cast<const float4 *>(stat_s + ss * 2 * kBQ + kBQ + g * kSpan);
            const int q0 = qt * kBQ + g * kSpan;  // first query of this thread's range
            // visible iff key <= query (causal), query < N and key < N
            const bool need_mask = (q0 + kSpan > N) || (a.causal && key > q0) || (key >= N);
            const bool any_mask = __any_sync(0xffffffffu, need_mask);

            ok = mbar_wait(&s_full[b], (i >> 1) & 1, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // P^T of this thread's 32 queries as bf16 pairs: the dV operand, and (unpacked) the factor of dS^T
            uint32_t pk[kSpan / 2];
            {
                uint32_t raw[kSpan];
                tmem_ld32(tmem + lane_base + 128 * b + g * kSpan, raw);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < kSpan / 4; ++q4) {
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
                    pk[2 * q4] = pack_bf16x2(p[0], p[1]);
                    pk[2 * q4 + 1] = pack_bf16x2(p[2], p[3]);
                }
            }
            tmem_st16(tmem + lane_base + 128 * b + g * kSpan, pk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&p_ready[b]);

            ok = mbar_wait(dp_full, i & 1, a.status, kSiteDpFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t raw[kSpan], dsk[kSpan / 2];
                tmem_ld32(tmem + lane_base + kColDP + g * kSpan, raw);
                tmem_wait_ld();
                // dP^T_i is in registers: the next dP^T may overwrite the buffer
                tc_fence_before();
                warp_arrive(dp_free);
#pragma unroll
                for (int q4 = 0; q4 < kSpan / 4; ++q4) {
                    const float4 d4 = ds4[q4];
                    const float2 p01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pk[2 * q4]));
                    const float2 p23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pk[2 * q4 + 1]));
                    // dS^T / scale = P^T * (dP^T - D), on fp32 pairs
                    dsk[2 * q4] = f2_to_bf16x2(f2_mul(
                        f2_sub(f2_pack(__uint_as_float(raw[4 * q4 + 0]), __uint_as_float(raw[4 * q4 + 1])),
                               f2_pack(d4.x, d4.y)),
                        f2_pack(p01.x, p01.y)));
                    dsk[2 * q4 + 1] = f2_to_bf16x2(f2_mul(
                        f2_sub(f2_pack(__uint_as_float(raw[4 * q4 + 2]), __uint_as_float(raw[4 * q4 + 3])),
                               f2_pack(d4.z, d4.w)),
                        f2_pack(p23.x, p23.y)));
                }
                // over the second half of this warpgroup's own S^T_i columns, already read
                tmem_st16(tmem + lane_base + 128 * b + g * kSpan + 16, dsk);
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
        // 128-byte-swizzled panels of 128 rows (one of 64 bf16 or two of 32 fp32 columns per output; dV's
        // first), and written by TMA bulk stores that clip rows past N and columns past the caller's D.
        const int n_panels = a.grad_bf16 ? 1 : 2;  // per output
        const int Dr = a.D;
        if (ok) {
            tc_fence_after();
            // warpgroups 0, 1 write dV (32 columns each), warpgroups 2, 3 write dK
            const bool is_dv = g < 2;
            const int c0 = (g & 1) * 32;
            const float osc = is_dv ? 1.f : sc;  // dK picks up the scale its dS^T operands left out
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + (is_dv ? kColDV : kColDK) + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * osc);
            uint8_t *stage = smem + (is_dv ? 0 : n_panels) * (kBN * 128) + r * 128;
            const int sw = r & 7;
            if (a.grad_bf16) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(stage + (((4 * (g & 1) + c) ^ sw) << 4),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
            } else {
                uint8_t *prow = stage + (g & 1) * (kBN * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(prow + ((c ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            }
        } else if (lane == 0) {
            epi_abort = 1;
        }
        fence_proxy_async_smem();  // the staged tiles are read by the TMA (async proxy)
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kComputeWG) : "memory");
        if (threadIdx.x == 32 * kFirstComputeWarp && !epi_abort) {
            const int pw = a.grad_bf16 ? 64 : 32;  // panel width in elements
            for (int p = 0; p < n_panels; ++p) {
                if (p * pw >= Dr) break;  // a panel wholly past the caller's D is not stored
                tma_store_3d(&tmap_dv, smem + p * (kBN * 128), p * pw, k_tile * kBN, bh);
                tma_store_3d(&tmap_dk, smem + (n_panels + p) * (kBN * 128), p * pw, k_tile * kBN, bh);
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

}  // namespace

cudaError_t launch_bwd_dkdv_q128(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdk,
                                 const CUtensorMap &tdv, cudaStream_t s) {
    using L = Q128Smem;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    if (kernel_head_dim(a.D) != kD) return cudaErrorInvalidValue;
    auto kern = bwd_dkdv_q128_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBN - 1) / kBN) * a.H * a.B);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, tdo, tdk, tdv, a);
    return cudaGetLastError();
}

}  // namespace fa
