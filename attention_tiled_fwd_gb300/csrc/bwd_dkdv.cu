// bwd_dkdv.cu -- second kernel of the atomic-free split backward ("backward
// key-value" of the metal-flash-attention page's pseudocode): one CTA per
// 128-key tile of one (batch, head), iterating over query tiles.
//
//   per query tile i:  S^T = K Q_i^T,  P^T = exp(S^T scale - L_i) (base 2 here),
//                      dV += P^T dO_i,
//                      dP^T = V dO_i^T,  dS^T = P^T * (dP^T - D_i) * scale,
//                      dK += dS^T Q_i
//   dK, dV written once after the last query tile.  Four GEMMs per tile, no
//   atomics, no scratch.  Causal: only query tiles on or below the diagonal
//   (queries >= keys) are visited.
//
// GB300 mapping: warp 0 TMA producer (K, V once; Q_i, dO_i through a ring),
// warp 1 TMEM allocator + tcgen05 issuer, warps 2-5 one key row per thread
// (L_i and D_i of the current query tile are broadcast from shared memory).
// TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D).
// P^T and dS^T (bf16) feed their MMAs as the TMEM A operand, with dO_i / Q_i
// as MN-major B operands (queries are the reduction).
// tcgen05.mma operations are only ordered among MMAs on the same accumulator.
//   D = 64: P^T and dS^T get their own 64 columns each ([384,448), [448,512));
//     the compute warps write them only after S^T_i / dP^T_i completed, and the
//     commits behind those track dV_{i-1} / dK_{i-1}, their previous readers.
//   D = 128: TMEM is full, so P^T is written over the first 64 columns of S^T
//     and dS^T over the first 64 of dP^T, and the issuer waits for dV_{i-1}
//     (resp. dK_{i-1}) to complete before S^T_i (resp. dP^T_i) overwrites them.
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>

namespace fa {
namespace {

constexpr int kBM = 128, kBN = 128;  // query tile, key tile
constexpr int kThreads = 192;

enum : int { kSiteKV = 41, kSiteSlotEmpty, kSiteSlotFull, kSiteSFull, kSitePReady, kSiteDpFull, kSiteDsReady,
             kSiteDone, kSiteFinal, kSiteDrain, kSiteStats, kSiteDvDone, kSiteDkDone };

template <int D, int NSLOT>
struct DkdvSmem {
    static constexpr int kTileBytes = kBM * D * 2;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kSlotOff = 2 * kTileBytes;  // slots hold Q_i, dO_i alternately
    static constexpr int kStatOff = kSlotOff + NSLOT * kTileBytes;  // lse2[2][128], delta[2][128]
    static constexpr int kBarOff = kStatOff + 4 * 128 * 4;
    // kv_full, slot_full[NSLOT], slot_empty[NSLOT], s_full, p_ready, dp_full, ds_ready, final, stats[2],
    // dv_done, dk_done
    static constexpr int kNumBars = 1 + 2 * NSLOT + 9;
    static constexpr int kTmemHolderOff = kBarOff + kNumBars * 8;
    static constexpr int kAlloc = kTmemHolderOff + 16 + 1024;
};

template <int D, int NSLOT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                    BwdArgs a) {
    using L = DkdvSmem<D, NSLOT>;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kTmemCols = 512;
    constexpr bool kSep = 256 + 2 * D + 128 <= 512;  // room for separate P^T and dS^T buffers
    constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    constexpr uint32_t kColP = kSep ? 256 + 2 * D : kColS, kColDS = kSep ? 256 + 2 * D + 64 : kColDP;
    static_assert(256 + 2 * D <= 512, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *k_s = smem + L::kKOff;
    uint8_t *v_s = smem + L::kVOff;
    uint8_t *slots = smem + L::kSlotOff;
    float *lse_s = reinterpret_cast<float *>(smem + L::kStatOff);  // [2][128], already times log2(e)
    float *del_s = lse_s + 256;                                     // [2][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *kv_full = bars;
    uint64_t *slot_full = bars + 1;
    uint64_t *slot_empty = slot_full + NSLOT;
    uint64_t *s_full = slot_empty + NSLOT;  // S^T and dP^T of the tile issued; S^T complete
    uint64_t *p_ready = s_full + 1;
    uint64_t *dp_full = p_ready + 1;
    uint64_t *ds_ready = dp_full + 1;
    uint64_t *final_bar = ds_ready + 1;
    uint64_t *stats_bar = final_bar + 1;  // [2]: the 128 compute threads published a stats buffer
    uint64_t *dv_done = stats_bar + 2;
    uint64_t *dk_done = dv_done + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kTmemHolderOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k_tile = blockIdx.x;  // causal: tile 0 has the most query tiles, launched first
    const int bh = blockIdx.z * a.H + blockIdx.y;
    const int N = a.N;
    const int n_q_total = (N + kBM - 1) / kBM;
    const int q_begin = a.causal ? (k_tile * kBN) / kBM : 0;
    const int n_q = n_q_total - q_begin;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(dp_full, 1);
        mbar_init(ds_ready, 128);
        mbar_init(final_bar, 1);
        mbar_init(&stats_bar[0], 128);
        mbar_init(&stats_bar[1], 128);
        mbar_init(dv_done, 1);
        mbar_init(dk_done, 1);
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
            mbar_arrive_expect_tx(kv_full, 2 * L::kTileBytes);
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
                    tma_load_3d(dst + p * (kBM * 128), map, &slot_full[slot], p * 64, (q_begin + (idx >> 1)) * kBM,
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
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBN, kBM, false, false);  // S^T, dP^T
            constexpr uint32_t idesc_g = idesc_bf16_f32(kBN, D, false, true);     // dV, dK
            const uint32_t k_addr = smem_u32(k_s), v_addr = smem_u32(v_s), slot_addr = smem_u32(slots);
            bool ok = mbar_wait(kv_full, 0, a.status, kSiteKV);
            tc_fence_after();
            for (int i = 0; ok && i < n_q; ++i) {
                const int q_idx = 2 * i, q_slot = q_idx % NSLOT, q_round = q_idx / NSLOT;
                const int d_idx = 2 * i + 1, d_slot = d_idx % NSLOT, d_round = d_idx / NSLOT;
                if (!(ok = mbar_wait(&slot_full[q_slot], q_round & 1, a.status, kSiteSlotFull))) break;
                if (!(ok = mbar_wait(&slot_full[d_slot], d_round & 1, a.status, kSiteSlotFull))) break;
                tc_fence_after();
                const uint32_t qbase = slot_addr + q_slot * L::kTileBytes;
                const uint32_t dbase = slot_addr + d_slot * L::kTileBytes;
                // S^T = K Q_i^T  (its columns last held P^T_{i-1} when P^T aliases S^T)
                if (!kSep && i > 0 && !(ok = mbar_wait(dv_done, (i - 1) & 1, a.status, kSiteDvDone))) break;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * (kBM * 128) + (ks & 3) * 32;
                    mma_ss(tmem + kColS, sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(qbase + off, 16, 1024),
                           idesc_s, ks > 0);
                }
                mma_commit(s_full);
                // dP^T = V dO_i^T  (its columns last held dS^T_{i-1} when dS^T aliases dP^T)
                if (!kSep && i > 0 && !(ok = mbar_wait(dk_done, (i - 1) & 1, a.status, kSiteDkDone))) break;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * (kBM * 128) + (ks & 3) * 32;
                    mma_ss(tmem + kColDP, sdesc_sw128(v_addr + off, 16, 1024), sdesc_sw128(dbase + off, 16, 1024),
                           idesc_s, ks > 0);
                }
                mma_commit(dp_full);
                // dV += P^T dO_i
                if (!(ok = mbar_wait(p_ready, i & 1, a.status, kSitePReady))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBM / 16; ++kk)
                    mma_ts(tmem + kColDV, tmem + kColP + kk * 8, sdesc_sw128(dbase + kk * 2048, kBM * 128, 1024),
                           idesc_g, (i > 0 || kk > 0));
                mma_commit(&slot_empty[d_slot]);
                mma_commit(dv_done);
                // dK += dS^T Q_i
                if (!(ok = mbar_wait(ds_ready, i & 1, a.status, kSiteDsReady))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBM / 16; ++kk)
                    mma_ts(tmem + kColDK, tmem + kColDS + kk * 8, sdesc_sw128(qbase + kk * 2048, kBM * 128, 1024),
                           idesc_g, (i > 0 || kk > 0));
                mma_commit(&slot_empty[q_slot]);
                mma_commit(dk_done);
            }
            mma_commit(final_bar);
            mbar_wait(final_bar, 0, a.status, kSiteFinal);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3;
        const int tid = (warp - 2) * 32 + lane;  // 0..127 for the stats loads
        const int r = quarter * 32 + lane;       // key row within the tile (TMEM lane)
        const int key = k_tile * kBN + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float c = a.scale_log2, sc = a.scale;
        const float *lse_g = a.lse + (size_t)bh * N;
        const float *del_g = a.delta + (size_t)bh * N;
        bool ok = true;
        // stats of query tile q_begin into buffer 0
        {
            const int qi = q_begin * kBM + tid;
            lse_s[tid] = qi < N ? lse_g[qi] * 1.4426950408889634f : INFINITY;
            del_s[tid] = qi < N ? del_g[qi] : 0.f;
            mbar_arrive(&stats_bar[0]);
        }
        for (int i = 0; i < n_q; ++i) {
            const int qt = q_begin + i;
            const int buf = i & 1;
            // prefetch next tile's stats into registers
            float nl = INFINITY, nd = 0.f;
            if (i + 1 < n_q) {
                const int qn = (qt + 1) * kBM + tid;
                if (qn < N) {
                    nl = lse_g[qn] * 1.4426950408889634f;
                    nd = del_g[qn];
                }
            }
            // stats of this tile visible to all compute threads (bounded wait, no named barrier)
            ok = mbar_wait(&stats_bar[buf], (i >> 1) & 1, a.status, kSiteStats);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const float *ls = lse_s + buf * 128;
            const float *ds = del_s + buf * 128;
            const int q0 = qt * kBM;
            // visible iff key <= query (causal) and query < N
            const bool need_mask = (q0 + kBM > N) || (a.causal && key > q0) || (key >= N);
            ok = mbar_wait(s_full, i & 1, a.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // P^T row as bf16 pairs: the MMA operand, and (unpacked) the factor of dS^T below.
            uint32_t pk[kBM / 2];
            const bool any_mask = __any_sync(0xffffffffu, need_mask);
#pragma unroll
            for (int ch = 0; ch < kBM / 32; ++ch) {
                uint32_t raw[32];
                tmem_ld32(tmem + lane_base + kColS + ch * 32, raw);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; t += 2) {
                    const int qc = ch * 32 + t;
                    float p0 = ex2_approx(fmaf(__uint_as_float(raw[t]), c, -ls[qc]));
                    float p1 = ex2_approx(fmaf(__uint_as_float(raw[t + 1]), c, -ls[qc + 1]));
                    if (any_mask) {
                        const int qq = q0 + qc;
                        if (qq >= N || key >= N || (a.causal && qq < key)) p0 = 0.f;
                        if (qq + 1 >= N || key >= N || (a.causal && qq + 1 < key)) p1 = 0.f;
                    }
                    pk[qc / 2] = pack_bf16x2(p0, p1);
                }
            }
#pragma unroll
            for (int ch = 0; ch < kBM / 64; ++ch) tmem_st32(tmem + lane_base + kColP + ch * 32, pk + ch * 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_ready);

            ok = mbar_wait(dp_full, i & 1, a.status, kSiteDpFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < kBM / 32; ++ch) {
                uint32_t raw[32], dsk[16];
                tmem_ld32(tmem + lane_base + kColDP + ch * 32, raw);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; t += 2) {
                    const int qc = ch * 32 + t;
                    const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pk[qc / 2]));
                    const float d0 = pf.x * (__uint_as_float(raw[t]) - ds[qc]) * sc;
                    const float d1 = pf.y * (__uint_as_float(raw[t + 1]) - ds[qc + 1]) * sc;
                    dsk[t / 2] = pack_bf16x2(d0, d1);
                }
                // When aliased: dS^T over dP^T columns [16 ch, 16 ch + 16), already read by chunks <= ch.
                tmem_st16(tmem + lane_base + kColDS + ch * 16, dsk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_ready);
            // Publish the next tile's stats into the other buffer.  Its readers of two tiles ago are
            // done: each of them arrived on this tile's stats barrier only after its last read.
            if (i + 1 < n_q) {
                lse_s[(buf ^ 1) * 128 + tid] = nl;
                del_s[(buf ^ 1) * 128 + tid] = nd;
                mbar_arrive(&stats_bar[buf ^ 1]);
            }
        }
        if (ok) {
            ok = mbar_wait(final_bar, 0, a.status, kSiteDone);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const bool valid = key < N;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which == 0 ? kColDV : kColDK;
                void *outp = which == 0 ? a.dv : a.dk;
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
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int NSLOT>
cudaError_t launch_spec(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, cudaStream_t s) {
    using L = DkdvSmem<D, NSLOT>;
    static_assert(L::kAlloc <= 232448, "shared memory budget");
    auto kern = bwd_dkdv_kernel<D, NSLOT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + kBN - 1) / kBN, a.H, a.B);
    kern<<<grid, kThreads, L::kAlloc, s>>>(tq, tk, tv, tdo, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_spec<64, 8>(a, tq, tk, tv, tdo, s);
        case 128: return launch_spec<128, 4>(a, tq, tk, tv, tdo, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
