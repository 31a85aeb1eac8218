// bwd_dq_k128.cu -- the dQ kernel of the split backward for D = 64, with
// 128-row key tiles.  Same computation as bwd_dq.cu ("backward query" of the
// metal-flash-attention page's pseudocode): one CTA per 128-row query tile of
// one (batch, head), iterating over K/V tiles,
//
//   D_i = sum_d dO_id O_id (written out),
//   S = Q K_j^T,  P = exp(S scale - L) (base 2 here),  dP = dO V_j^T,
//   dS = P * (dP - D),  dQ += dS K_j,
//
// dQ (times the softmax scale, left out of every dS) written once at the end;
// causal: only key tiles up to the diagonal are visited.
//
// Why a separate kernel: at D = 64 the 64-key tiles of bwd_dq.cu make every
// product an N = 64 MMA, which the tensor core runs at about 60 % of its rate.
// With 128-key tiles S and dP are N = 128 products.  TMEM holds S and dP once
// each (128 columns each), dS twice (64 bf16 columns each), dQ (64) and Q, dO
// (32 each, the TMEM A operands of S and dP):
//   - S and dP are single-buffered: every compute warp loads its S and dP
//     columns into registers first thing and releases each buffer (s_free,
//     dp_free), so S_{j+1} and dP_{j+1} run while the compute warps work on
//     tile j;
//   - dS_j goes to dS[j % 2], which the compute warps rewrite only after dQ_{j-2}
//     has read it, so no S or dP product waits for a dQ product.
// (An earlier version wrote dS over S and double-buffered S instead; S_{j+2}
// then waited for dQ_j, and this layout measured 15 % faster: 6.60 -> 5.62 ms
// at B=1 H=32 N=32768.  At D = 128 the same scheme needs S and dP as SS
// products and measured 14 % slower than bwd_dq.cu.)
// Roles: warp 0 TMA producer (Q, dO once; 128-row K_j, V_j through a ring);
// warp 1 issuer A (S, dP); warp 2 issuer B (dQ); warps 3-18 compute: four
// warpgroups, warpgroup g owning keys [32g, 32g+32) of every tile, a thread
// owning one query row (its TMEM lane).
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBM = 128;          // queries per CTA (TMEM lanes)
constexpr int kBN = 128;          // keys per tile
constexpr int kComputeWG = 4;
constexpr int kSpan = kBN / kComputeWG;  // 32 keys per compute thread per tile
constexpr int kFirstComputeWarp = 3;
constexpr int kThreads = 32 * kFirstComputeWarp + 128 * kComputeWG;
constexpr int kComputeWarps = 4 * kComputeWG;

enum : int { kSiteQ = 101, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSiteDsFull, kSiteDq, kSiteFinal, kSiteDrain,
             kSiteDqDone, kSiteQt, kSiteDpFull, kSiteDpFree, kSiteSFree };

constexpr int kD = 64;
constexpr int kNSlot = 8;  // K_j / V_j ring (4 tiles)

struct K128Smem {
    static constexpr int kQBytes = kBM * kD * 2;     // Q and dO: 128 x 64 bf16 each
    static constexpr int kTileBytes = kBN * kD * 2;  // one K_j or V_j tile
    static constexpr int kQOff = 0;
    static constexpr int kDoOff = kQBytes;
    static constexpr int kSlotOff = 2 * kQBytes;
    static constexpr int kOOff = kSlotOff + kNSlot * kTileBytes;  // O's tile (for D_i)
    static constexpr int kDeltaOff = kOOff + kQBytes;  // [kComputeWG][kBM] partial sums of dO * O
    static constexpr int kBarOff = kDeltaOff + kComputeWG * kBM * 4;
    // q_full, slot_full[kNSlot], slot_empty[kNSlot], s_full, s_free, ds_full[2], dq_done[2], dp_full, dp_free,
    // qt_ready, final, a_final, o_full
    static constexpr int kNumBars = 1 + 2 * kNSlot + 2 + 4 + 2 + 4;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_k128_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                       const __grid_constant__ CUtensorMap tmap_o, const __grid_constant__ CUtensorMap tmap_dq,
                       BwdArgs a) {
    using L = K128Smem;
    constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S = [0, 128) and dP = [128, 256), each single-buffered and released as soon as every
    // compute warp has loaded it; dS[b] = [256 + 64b, +64) (bf16, b = j % 2); dQ = [384, 448); Q =
    // [448, 480) and dO = [480, 512), the TMEM A operands of S and dP.  Warpgroup g's keys sit at columns
    // 32g.. of S and dP and its dS at [256 + 64b + 16g, +16), so 16-key step kk of the dQ product reads
    // column 256 + 64b + 8kk.
    constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 384, kColQ = 448, kColDO = 480;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem + L::kQOff;
    uint8_t *do_s = smem + L::kDoOff;
    uint8_t *o_s = smem + L::kOOff;
    uint8_t *slots = smem + L::kSlotOff;
    float *delta_s = reinterpret_cast<float *>(smem + L::kDeltaOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + kNSlot;
    uint64_t *s_full = slot_empty + kNSlot;  // S_j complete (phase j)
    uint64_t *s_free = s_full + 1;           // every compute warp has loaded S_j (phase j)
    uint64_t *ds_full = s_free + 1;          // [2]: dS_j written into dS[j % 2]
    uint64_t *dq_done = ds_full + 2;         // [2]: dQ_j complete: dS[j % 2] is free
    uint64_t *dp_full = dq_done + 2;         // dP_j complete (phase j)
    uint64_t *dp_free = dp_full + 1;         // every compute warp has loaded dP_j (phase j)
    uint64_t *qt_ready = dp_free + 1;        // Q and dO are in TMEM
    uint64_t *final_bar = qt_ready + 1;      // issuer B: every dQ MMA has completed
    uint64_t *a_final = final_bar + 1;       // issuer A: every S / dP MMA has completed
    uint64_t *o_full = a_final + 1;          // O's tile landed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    __shared__ int epi_abort;  // a compute warp's wait ran out: the epilogue stores nothing
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    tile_order((a.N + kBM - 1) / kBM, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int q_tile = (a.N + kBM - 1) / kBM - 1 - rank;  // causal: the last query tile has the most keys
    const int N = a.N;
    const int kv_end = a.causal ? min(N, (q_tile + 1) * kBM) : N;
    const int n_kv = (kv_end + kBN - 1) / kBN;  // >= 1

    if (threadIdx.x == 0) {
        epi_abort = 0;
        mbar_init(q_full, 1);
        for (int s = 0; s < kNSlot; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, kComputeWarps);  // one arrive per compute warp
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ds_full[b], kComputeWarps);
            mbar_init(&dq_done[b], 1);
        }
        mbar_init(dp_full, 1);
        mbar_init(dp_free, kComputeWarps);
        mbar_init(qt_ready, kComputeWarps);
        mbar_init(final_bar, 1);
        mbar_init(a_final, 1);
        mbar_init(o_full, 1);
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
            tma_load_3d(q_s, &tmap_q, q_full, 0, q_tile * kBM, bh);
            tma_load_3d(do_s, &tmap_do, q_full, 0, q_tile * kBM, bh);
            tma_prefetch_desc(&tmap_o);
            mbar_arrive_expect_tx(o_full, L::kQBytes);
            tma_load_3d(o_s, &tmap_o, o_full, 0, q_tile * kBM, bh);
            int last_round[kNSlot];
#pragma unroll
            for (int s = 0; s < kNSlot; ++s) last_round[s] = -1;
            for (int idx = 0; idx < 2 * n_kv; ++idx) {
                const int slot = idx % kNSlot, round = idx / kNSlot;
                if (!mbar_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty)) break;
                const CUtensorMap *map = (idx & 1) ? &tmap_v : &tmap_k;
                mbar_arrive_expect_tx(&slot_full[slot], L::kTileBytes);
                tma_load_3d(slots + slot * L::kTileBytes, map, &slot_full[slot], 0, (idx >> 1) * kBN, bh);
#pragma unroll
                for (int s = 0; s < kNSlot; ++s)
                    if (s == slot) last_round[s] = round;
            }
            // Drain: never leave the CTA with a TMA write still in flight.
#pragma unroll
            for (int s = 0; s < kNSlot; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            mbar_wait(q_full, 0, a.status, kSiteDrain);
            mbar_wait(o_full, 0, a.status, kSiteDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // Issuer A: S_j = Q K_j^T and dP_j = dO V_j^T, TS products (Q, dO from TMEM), each into its one
        // buffer as soon as every compute warp has loaded the previous tile's.
        constexpr uint32_t idesc_sq = idesc_bf16_f32(kBM, kBN, false, false);  // 128 x 128
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = warp_wait(qt_ready, 0, a.status, kSiteQt);
        tc_fence_after();
        for (int j = 0; ok && j < n_kv; ++j) {
            const int k_slot = (2 * j) % kNSlot, k_round = (2 * j) / kNSlot;
            const int v_slot = (2 * j + 1) % kNSlot, v_round = (2 * j + 1) / kNSlot;
            if (!(ok = warp_wait(&slot_full[k_slot], k_round & 1, a.status, kSiteSlotFull))) break;
            // the S buffer last held S_{j-1}, which every compute warp has loaded
            if (j >= 1 && !(ok = warp_wait(s_free, (j - 1) & 1, a.status, kSiteSFree))) break;
            tc_fence_after();
            const uint64_t k_desc = sdesc_sw128(slot_addr + k_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_ts(tmem + kColS, tmem + kColQ + ks * 8, sdesc_add(k_desc, ks * 32), idesc_sq, ks > 0);
                mma_commit(s_full);
            }
            __syncwarp();
            if (!(ok = warp_wait(&slot_full[v_slot], v_round & 1, a.status, kSiteSlotFull))) break;
            // the dP buffer last held dP_{j-1}, which every compute warp has loaded
            if (j >= 1 && !(ok = warp_wait(dp_free, (j - 1) & 1, a.status, kSiteDpFree))) break;
            tc_fence_after();
            const uint64_t v_desc = sdesc_sw128(slot_addr + v_slot * L::kTileBytes, 16, 1024);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_ts(tmem + kColDP, tmem + kColDO + ks * 8, sdesc_add(v_desc, ks * 32), idesc_sq, ks > 0);
                mma_commit(dp_full);
                mma_commit(&slot_empty[v_slot]);  // V_j is no longer needed
            }
            __syncwarp();
        }
        // Drain this warp's MMAs before TMEM can be released (immediate in the normal path).
        if (leader) mma_commit(a_final);
        __syncwarp();
        warp_wait(a_final, 0, a.status, kSiteFinal);
    } else if (warp == 2) {
        // Issuer B: dQ += dS_j K_j (K_j as the MN-major B operand: keys are the reduction).
        constexpr uint32_t idesc_dq = idesc_bf16_f32(kBM, kD, false, true);  // 128 x 64
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            const uint32_t b = j & 1;
            const int k_slot = (2 * j) % kNSlot;
            const uint64_t kmn_desc = sdesc_sw128(slot_addr + k_slot * L::kTileBytes, kBN * 128, 1024);
            if (!(ok = warp_wait(&ds_full[b], (j >> 1) & 1, a.status, kSiteDsFull))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tmem + kColDQ, tmem + kColDS + 64 * b + 8 * kk,
                           sdesc_add(kmn_desc, kk * 2048), idesc_dq, (j > 0 || kk > 0));
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
        // Row stride and real columns: the caller's D (a multiple of 8, at most 64; TMA fills the rest of
        // the 64-column panels with zeros, which add nothing).
        const int Dr = a.D;
        // Q (warpgroup 0) and dO (warpgroup 1) rows into TMEM as bf16 pairs first thing, so that S_0 and dP_0
        // run while D_i is summed (row r of the 64-column panel is 128 B at r * 128, its 16-byte chunk k
        // stored at k ^ (r % 8))
        {
            bool qok = mbar_wait(q_full, 0, a.status, kSiteQ);
            if (!__all_sync(0xffffffffu, qok)) qok = false;
            if (qok && g < 2) {
                const uint8_t *panel = (g == 0 ? q_s : do_s) + r * 128;
                uint32_t w[32];
#pragma unroll
                for (int kc = 0; kc < 8; ++kc) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(panel + ((kc ^ (r & 7)) << 4));
                    w[4 * kc] = x.x;
                    w[4 * kc + 1] = x.y;
                    w[4 * kc + 2] = x.z;
                    w[4 * kc + 3] = x.w;
                }
                tmem_st32(tmem + lane_base + (g == 0 ? kColQ : kColDO), w);
                tmem_wait_st();
            }
            tc_fence_before();
            warp_arrive(qt_ready);
        }
        // D_i = sum_d dO_id O_id for this thread's row, from the staged O and dO tiles (both swizzled alike, so
        // chunk k of row r sits at the same place in each; columns past the caller's D and rows past N are
        // zeros from the TMA): warpgroup g sums columns [16g, 16g + 16); the partial sums meet in shared
        // memory and every warpgroup adds them in the same order.
        float delta = 0.f;
        {
            const bool ook = mbar_wait(o_full, 0, a.status, kSiteQ);
            if (__all_sync(0xffffffffu, ook)) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int off = r * 128 + (((2 * g + i) ^ (r & 7)) << 4);
                    const uint4 ov = *reinterpret_cast<const uint4 *>(o_s + off);
                    const uint4 dv = *reinterpret_cast<const uint4 *>(do_s + off);
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
        delta_s[g * kBM + r] = delta;
        // every compute warp reaches this barrier: nothing before it waits or exits early
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kComputeWG) : "memory");
        delta = 0.f;
#pragma unroll
        for (int t = 0; t < kComputeWG; ++t) delta += delta_s[t * kBM + r];
        if (valid && g == 0) a.delta[(size_t)bh * N + row] = delta;
        const int lim = a.causal ? min(N - 1, row) : N - 1;  // last visible key
        const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(-lse2, -lse2), d2 = f2_pack(delta, delta);
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const uint32_t b = j & 1;
            ok = mbar_wait(s_full, j & 1, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int key0 = j * kBN + g * kSpan;
            const bool need_mask = (key0 + kSpan > N) || (a.causal && key0 + kSpan - 1 > q_tile * kBM);
            uint32_t sraw[kSpan], praw[kSpan], dsk[kSpan / 2];
            tmem_ld32(tmem + lane_base + kColS + g * kSpan, sraw);
            tmem_wait_ld();
            // S_j is in registers: the next S may overwrite the buffer
            tc_fence_before();
            warp_arrive(s_free);
            ok = mbar_wait(dp_full, j & 1, a.status, kSiteDpFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(tmem + lane_base + kColDP + g * kSpan, praw);
            tmem_wait_ld();
            // dP_j is in registers: the next dP may overwrite the buffer
            tc_fence_before();
            warp_arrive(dp_free);
            // dS / scale = P * (dP - D), on fp32 pairs (f32x2), two scores per instruction
#pragma unroll
            for (int i = 0; i < kSpan; i += 2) {
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
            // dS[b] was last read by dQ_{j-2}
            if (j >= 2) {
                ok = mbar_wait(&dq_done[b], ((j - 2) >> 1) & 1, a.status, kSiteDqDone);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
            }
            tmem_st16(tmem + lane_base + kColDS + 64 * b + 16 * g, dsk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&ds_full[b]);
        }
        if (ok) {
            ok = mbar_wait(final_bar, 0, a.status, kSiteDq);  // single phase: every MMA has completed
            ok = __all_sync(0xffffffffu, ok);
        }
        // Epilogue: dQ (times the softmax scale) staged in the Q / dO tiles' shared memory, which no MMA reads
        // any more, as 128-byte-swizzled panels of 128 rows (one of 64 bf16 columns, or two of 32 fp32
        // columns), then written by TMA bulk stores that clip rows past N and columns past the caller's D.
        if (ok) {
            tc_fence_after();
            // this warpgroup's 16 columns of dQ
            uint32_t v[16];
            tmem_ld16(tmem + lane_base + kColDQ + 16 * g, v);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * a.scale);
            const int sw = r & 7;
            if (a.grad_bf16) {
                uint8_t *prow = smem + r * 128;  // chunks 2g, 2g + 1 of the 64-column panel
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    st_shared_v4(prow + (((2 * g + c) ^ sw) << 4),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
            } else {
                uint8_t *prow = smem + (g >> 1) * (kBM * 128) + r * 128;  // chunks 4 (g % 2) .. + 3 of panel g / 2
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(prow + (((4 * (g & 1) + c) ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                                 v[4 * c + 3]);
            }
        } else if (lane == 0) {
            epi_abort = 1;
        }
        fence_proxy_async_smem();  // the staged tile is read by the TMA (async proxy)
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kComputeWG) : "memory");
        if (threadIdx.x == 32 * kFirstComputeWarp && !epi_abort) {
            if (a.grad_bf16) {
                tma_store_3d(&tmap_dq, smem, 0, q_tile * kBM, bh);
            } else {
                tma_store_3d(&tmap_dq, smem, 0, q_tile * kBM, bh);
                if (Dr > 32) tma_store_3d(&tmap_dq, smem + kBM * 128, 32, q_tile * kBM, bh);
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

cudaError_t launch_bwd_dq_k128(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                               const CUtensorMap &tdo, const CUtensorMap &to, const CUtensorMap &tdq,
                               cudaStream_t s) {
    using L = K128Smem;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    if (kernel_head_dim(a.D) != kD) return cudaErrorInvalidValue;
    auto kern = bwd_dq_k128_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBM - 1) / kBM) * a.H * a.B);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, tdo, to, tdq, a);
    return cudaGetLastError();
}

}  // namespace fa
