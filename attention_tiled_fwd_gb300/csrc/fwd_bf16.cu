// fwd_bf16.cu -- bf16 attention forward on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM), one 128-row query tile per CTA, K/V tiles
// streamed by TMA through an mbarrier ring in shared memory.  Used for
// D = 192 and 256 (64-key tiles); D = 64 and 128 run the two-tile kernels of
// fwd_bf16_duo.cu and fwd_bf16_pair.cu (launch_fwd_bf16 below holds the measured choice).
//
// Algorithm ("Learning Metal with FlashAttention", section "FlashAttention";
// metalworking "Flash Attention", kernel anatomy items 1-5; metal-flash-
// attention forward pseudocode):
//   Q tile loaded once and kept; for each K/V tile: S = Q K^T, scaled into
//   the base-2 domain and masked in place, running max m / sum l, P = 2^(S-m),
//   O <- alpha O + P V; after the last tile O /= l and L = m + ln(l) is
//   written.  Causal tiles above the diagonal are never loaded or computed.
//
// GB300 mapping (one CTA = one 128-row query tile of one (batch, head)):
//   warp 0      TMA producer: Q once, then K_j, V_j into an NSLOT-deep ring
//   warp 1      TMEM allocator + tcgen05 issuer A: S_j = Q K_j^T (SS: both
//               operands in shared memory) into one of two S buffers in TMEM
//   warp 2      tcgen05 issuer B: O += P_j V_j (TS: P_j, bf16, in one of two P
//               buffers in TMEM).  Two issuers, because an MMA's issue blocks
//               until the tensor core accepts it, so a single issuer leaves the
//               tensor core idle whenever it waits on a barrier.
//   warps 3-10  softmax, two warpgroups: a thread owns one query row (its TMEM
//               lane) and one half of every S tile's columns.  The row max is
//               thread-local within a half; the two halves of a row combine
//               their maxima through shared memory (one bounded mbarrier
//               round per tile) so both use the same reference max, and add
//               their partial sums once at the end.  P is written back to TMEM
//               as bf16; each half rescales and normalises its half of O.
//               The O correction is lazy: O is rescaled only when the running
//               max grows by more than 2^8 (the "branch-guarded correction"
//               of the metalworking page), otherwise the stale max is kept;
//               the final O / l is the same.
//   TMEM: S0 [0, BN), S1 [BN, 2BN), O [2BN, 2BN + D), P0, P1 (BN/2 each)
//   after O.  For D = 256 the O accumulator spans 256 columns and the PV
//   product is one N = 256 MMA per 16-key step (D-blocking lives in the
//   64-column panels of V and Q).
//   Ordering: tcgen05.mma operations are only ordered among MMAs on the same
//   accumulator, and a commit tracks only its own thread's MMAs, so every TMEM
//   buffer is rewritten only after its previous reader is known complete: the
//   softmax writes P_j into P[j % 2] after waiting for PV_{j-2} (per-buffer
//   barrier pv_done[j % 2]), and issuer A writes S_{j+2} into S[j % 2] after the
//   softmax finished reading S_j.
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBM = 128;
constexpr int kSoftmaxWG = 2;  // softmax warpgroups, one column half each
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kThreads = 32 * kFirstSoftmaxWarp + 128 * kSoftmaxWG;

// Wait-site ids recorded in the status word on a time-out.
enum : int { kSiteQ = 1, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePFull, kSitePV, kSiteFinal, kSiteDrain,
             kSiteXchg };

template <int D, int BN, int NSLOT>
struct FwdSmem {
    static constexpr int kPanels = D / 64;
    static constexpr int kQBytes = kBM * D * 2;
    static constexpr int kSlotBytes = BN * D * 2;
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = kQBytes;
    static constexpr int kXchgOff = kSlotOff + NSLOT * kSlotBytes;  // row-max exchange [2][2][128] + l [2][128]
    static constexpr int kBarOff = kXchgOff + (4 * kBM + 2 * kBM) * 4;
    // barriers: q_full, slot_full[NSLOT], slot_empty[NSLOT], s_full[2], p_full[2], pv_done[2], final, a_final,
    // xchg[2], lx
    static constexpr int kNumBars = 1 + 2 * NSLOT + 2 + 2 + 2 + 1 + 1 + 3;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kBytes = kTmemHolderOff + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment of the base
};

template <int D, int BN, int NSLOT>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, FwdArgs a) {
    using L = FwdSmem<D, BN, NSLOT>;
    constexpr int kPanels = L::kPanels;
    constexpr uint32_t kTmemCols = 512;
    constexpr uint32_t kColS0 = 0, kColS1 = BN, kColO = 2 * BN, kColP0 = 2 * BN + D, kColP1 = kColP0 + BN / 2;
    static_assert(kColP1 + BN / 2 <= 512, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem + L::kQOff;
    uint8_t *slots = smem + L::kSlotOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + NSLOT;
    uint64_t *s_full = slot_empty + NSLOT;
    uint64_t *p_full = s_full + 2;
    uint64_t *pv_done = p_full + 2;     // [2]: PV_j completed (P buffer j % 2 is free again)
    uint64_t *final_bar = pv_done + 2;  // issuer B: every PV MMA has completed (O is final)
    uint64_t *a_final = final_bar + 1;  // issuer A: every S MMA has completed
    uint64_t *xchg = a_final + 1;       // [2]: every softmax thread published its half-row max of a tile
    uint64_t *lx = xchg + 2;         // every softmax thread published its partial row sum
    float *smax = reinterpret_cast<float *>(smem + L::kXchgOff);  // [tile parity][half][row]
    float *lsum = smax + 4 * kBM;                                  // [half][row]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    tile_order((a.N + kBM - 1) / kBM, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int q_tile = (a.N + kBM - 1) / kBM - 1 - rank;  // causal: the last query tile has the most keys
    const int N = a.N;
    const int kv_end = a.causal ? min(N, (q_tile + 1) * kBM) : N;
    const int n_kv = (kv_end + BN - 1) / BN;  // >= 1 because q_tile * kBM < N

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4 * kSoftmaxWG);  // one arrive per softmax warp
            mbar_init(&xchg[b], 4 * kSoftmaxWG);
            mbar_init(&pv_done[b], 1);
        }
        mbar_init(final_bar, 1);
        mbar_init(a_final, 1);
        mbar_init(lx, 4 * kSoftmaxWG);
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
            mbar_arrive_expect_tx(q_full, L::kQBytes);
#pragma unroll
            for (int p = 0; p < kPanels; ++p)
                tma_load_3d(q_s + p * (kBM * 128), &tmap_q, q_full, p * 64, q_tile * kBM, bh);
            int last_round[NSLOT];
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) last_round[s] = -1;
            for (int idx = 0; idx < 2 * n_kv; ++idx) {
                const int slot = idx % NSLOT, round = idx / NSLOT;
                if (!mbar_wait(&slot_empty[slot], (round & 1) ^ 1, a.status, kSiteSlotEmpty)) break;
                uint8_t *dst = slots + slot * L::kSlotBytes;
                const CUtensorMap *map = (idx & 1) ? &tmap_v : &tmap_k;
                mbar_arrive_expect_tx(&slot_full[slot], L::kSlotBytes);
#pragma unroll
                for (int p = 0; p < kPanels; ++p)
                    tma_load_3d(dst + p * (BN * 128), map, &slot_full[slot], p * 64, (idx >> 1) * BN, bh);
#pragma unroll
                for (int s = 0; s < NSLOT; ++s)
                    if (s == slot) last_round[s] = round;
            }
            // Drain: never leave the CTA with a TMA write still in flight.
#pragma unroll
            for (int s = 0; s < NSLOT; ++s)
                if (last_round[s] >= 0) mbar_wait(&slot_full[s], last_round[s] & 1, a.status, kSiteDrain);
            mbar_wait(q_full, 0, a.status, kSiteDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer A: S_j = Q K_j^T
        // The whole warp runs the loop (operands stay warp-uniform); one elected lane issues the MMAs
        // and the commits that track them.
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, BN, false, false);
        const uint64_t q_desc = sdesc_sw128(smem_u32(q_s), 16, 1024);
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = warp_wait(q_full, 0, a.status, kSiteQ);
        tc_fence_after();
        for (int j = 0; ok && j < n_kv; ++j) {
            const int idx = 2 * j, slot = idx % NSLOT, round = idx / NSLOT;
            // S[j % 2] last held S_{j-2}; the softmax has read it once P_{j-2} is published
            if (j >= 2 && !(ok = warp_wait(&p_full[j & 1], ((j - 2) >> 1) & 1, a.status, kSitePFull))) break;
            if (!(ok = warp_wait(&slot_full[slot], round & 1, a.status, kSiteSlotFull))) break;
            tc_fence_after();
            const uint64_t k_desc = sdesc_sw128(slot_addr + slot * L::kSlotBytes, 16, 1024);
            const uint32_t d_s = tmem + ((j & 1) ? kColS1 : kColS0);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;  // 16 bf16 = 32 B step inside the 128-B row
                    mma_ss(d_s, sdesc_add(q_desc, (ks >> 2) * (kBM * 128) + off),
                           sdesc_add(k_desc, (ks >> 2) * (BN * 128) + off), idesc_s, ks > 0);
                }
                mma_commit(&s_full[j & 1]);
                mma_commit(&slot_empty[slot]);
            }
            __syncwarp();
        }
        // Drain this warp's MMAs before TMEM can be released (immediate in the normal path).
        if (leader) mma_commit(a_final);
        __syncwarp();
        warp_wait(a_final, 0, a.status, kSiteFinal);
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA issuer B: O += P_j V_j
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, false, true);
        const uint32_t slot_addr = smem_u32(slots);
        const bool leader = elect_one();
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            if (!(ok = warp_wait(&p_full[j & 1], (j >> 1) & 1, a.status, kSitePFull))) break;
            const int idx = 2 * j + 1, slot = idx % NSLOT, round = idx / NSLOT;
            if (!(ok = warp_wait(&slot_full[slot], round & 1, a.status, kSiteSlotFull))) break;
            tc_fence_after();
            const uint64_t v_desc = sdesc_sw128(slot_addr + slot * L::kSlotBytes, BN * 128, 1024);
            const uint32_t p_t = tmem + ((j & 1) ? kColP1 : kColP0);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tmem + kColO, p_t + kk * 8, sdesc_add(v_desc, kk * 2048), idesc_o, (j > 0 || kk > 0));
                mma_commit(&slot_empty[slot]);
                mma_commit(&pv_done[j & 1]);
            }
            __syncwarp();
        }
        // Every PV MMA has completed before O is read or TMEM released.
        if (leader) mma_commit(final_bar);
        __syncwarp();
        warp_wait(final_bar, 0, a.status, kSiteFinal);
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        constexpr int HB = BN / kSoftmaxWG;  // S columns per thread per tile
        constexpr int HD = D / kSoftmaxWG;   // O columns per thread
        const int quarter = warp & 3;                 // TMEM lanes [32*quarter, 32*quarter + 32)
        const int g = (warp - kFirstSoftmaxWarp) >> 2;  // column half
        const int r = quarter * 32 + lane;
        const int row = q_tile * kBM + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float c = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const uint32_t s_col = ((j & 1) ? kColS1 : kColS0) + g * HB;
            const uint32_t p_col = ((j & 1) ? kColP1 : kColP0) + g * (HB / 2);
            ok = mbar_wait(&s_full[j & 1], (j >> 1) & 1, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // raw scores; the scale is folded into the exponent's FMA below
            uint32_t raw[HB];
#pragma unroll
            for (int ch = 0; ch < HB / 32; ++ch) tmem_ld32(tmem + lane_base + s_col + ch * 32, raw + ch * 32);
            tmem_wait_ld();
            const int key0 = j * BN + g * HB;
            const bool need_mask = (key0 + HB > N) || (a.causal && key0 + HB - 1 > q_tile * kBM);
            if (need_mask) {
                const int lim = a.causal ? min(N - 1, row) : N - 1;  // last visible key
#pragma unroll
                for (int i = 0; i < HB; ++i)
                    if (key0 + i > lim) raw[i] = 0xff800000u;  // -inf
            }
            // row max over this half (scale > 0 commutes with max): four chains of three-input maxima
            float mx[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) mx[u] = __uint_as_float(raw[u]);
#pragma unroll
            for (int i = 4; i + 8 <= HB; i += 8)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mx[u] = fmax3(mx[u], __uint_as_float(raw[i + 2 * u]), __uint_as_float(raw[i + 2 * u + 1]));
#pragma unroll
            for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], __uint_as_float(raw[HB - 4 + u]));
            float mt = c * fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
            // combine with the other half of the row
            smax[((j & 1) * 2 + g) * kBM + r] = mt;
            warp_arrive(&xchg[j & 1]);
            ok = mbar_wait(&xchg[j & 1], (j >> 1) & 1, a.status, kSiteXchg);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            mt = fmaxf(mt, smax[((j & 1) * 2 + (g ^ 1)) * kBM + r]);
            const float m_new = fmaxf(m, mt);
            // Lazy correction: keep the stale max unless the row max grew by > 8 (factor 256).
            const bool need = m_new > m + 8.f;
            const float m_use = need ? m_new : m;
            const float m_base = (m_use == -INFINITY) ? 0.f : m_use;
            const float alpha = need ? ex2_approx(m - m_base) : 1.f;
            // P[j % 2] was last read by PV_{j-2}
            if (j >= 2) {
                ok = mbar_wait(&pv_done[j & 1], ((j >> 1) - 1) & 1, a.status, kSitePV);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
            }
            // P = 2^(s c - m) as bf16 pairs into this tile's P buffer (this half's columns), 16 columns
            // per store; the scaling FMA and the row sum run on fp32 pairs
            const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_base, -m_base);
            uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
            for (int ch = 0; ch < HB / 32; ++ch) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint64_t y2 = f2_fma(f2_pack(__uint_as_float(raw[ch * 32 + 2 * i]),
                                                       __uint_as_float(raw[ch * 32 + 2 * i + 1])), c2, nm2);
                    float y0, y1;
                    f2_unpack(y2, y0, y1);
                    const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                    acc2[i & 1] = f2_add(acc2[i & 1], f2_pack(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tmem + lane_base + p_col + ch * 16, pk);
            }
            float r0, r1, r2, r3;
            f2_unpack(acc2[0], r0, r1);
            f2_unpack(acc2[1], r2, r3);
            l = l * alpha + ((r0 + r1) + (r2 + r3));
            m = m_use;
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                // O must hold P_{j-1} V_{j-1} before it is rescaled (this half's columns).
                ok = mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, a.status, kSitePV);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t ov[32];
#pragma unroll
                for (int ch = 0; ch < HD / 32; ++ch) {
                    const uint32_t oc = kColO + g * HD + ch * 32;
                    tmem_ld32(tmem + lane_base + oc, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(tmem + lane_base + oc, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&p_full[j & 1]);
        }
        if (ok) {
            // O is final once every PV MMA has completed: final_bar has a single phase, committed by
            // issuer B after its last MMA.
            ok = mbar_wait(final_bar, 0, a.status, kSiteFinal);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            lsum[g * kBM + r] = l;
            warp_arrive(lx);
            ok = mbar_wait(lx, 0, a.status, kSiteXchg);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            const float l_row = l + lsum[(g ^ 1) * kBM + r];
            tc_fence_after();
            const float inv_l = 1.f / l_row;
            // row stride and stored columns: the caller's D (at most this kernel's D; the columns past it
            // hold zeros from the TMA's out-of-bounds fill)
            const int Dr = a.D;
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.o) + ((size_t)bh * N + row) * Dr + g * HD;
            uint32_t ov[32];
#pragma unroll
            for (int ch = 0; ch < HD / 32; ++ch) {
                tmem_ld32(tmem + lane_base + kColO + g * HD + ch * 32, ov);
                tmem_wait_ld();
                if (row < N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        if (g * HD + ch * 32 + v4 * 8 >= Dr) break;
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 0]) * inv_l, __uint_as_float(ov[v4 * 8 + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 2]) * inv_l, __uint_as_float(ov[v4 * 8 + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 4]) * inv_l, __uint_as_float(ov[v4 * 8 + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(ov[v4 * 8 + 6]) * inv_l, __uint_as_float(ov[v4 * 8 + 7]) * inv_l);
                        dst[v4] = w;
                    }
                }
            }
            if (row < N && g == 0) a.lse[(size_t)bh * N + row] = (m + __log2f(l_row)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int BN, int NSLOT>
cudaError_t launch_spec(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        cudaStream_t s) {
    using L = FwdSmem<D, BN, NSLOT>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    auto kern = fwd_bf16_kernel<D, BN, NSLOT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBM - 1) / kBM) * a.H * a.B);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &to, cudaStream_t s) {
    switch (kernel_head_dim(a.D)) {
        // measured choice per head dimension: a persistent two-tile kernel wherever its TMEM
        // layout fits (D <= 128; at D = 128 non-causal it measured equal to this kernel at
        // N = 4096 and 5-13 % faster at N = 1024, 2048 and 16384); at D = 64 the variant with an
        // issuer and a P buffer per tile (7 % faster there, 12-15 % slower at D = 128 without P buffers)
        case 64: return launch_fwd_bf16_duo(a, tq, tk, tv, s);
        case 128: return launch_fwd_bf16_pair(a, tq, tk, tv, to, s);
        case 192: return launch_spec<192, 64, fwd_nslot(192)>(a, tq, tk, tv, s);
        case 256: return launch_spec<256, 64, fwd_nslot(256)>(a, tq, tk, tv, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
