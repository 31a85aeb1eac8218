// fa_internal.h -- launch interfaces shared by the C-ABI layer (fa_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

// Spec table of the bf16 forward: query rows per CTA, keys per K/V tile, K/V
// ring depth, keyed by head dimension.  Picked so that the score, P and O
// buffers fit the 512 TMEM columns and the staged tiles fill (but do not
// exceed) shared memory.
//   D = 64, 128: two 128-row query tiles per CTA (fwd_bf16_pair.cu), causal
//                and non-causal, on a persistent grid of one CTA per SM; TMEM
//                per tile S 128 (P over its first 64) + O D columns; shared
//                memory 2 Q tiles + ring.
//   D = 192, 256: one 128-row query tile, two softmax warpgroups splitting
//                the columns (fwd_bf16.cu); TMEM S 2x64 + P 2x32 + O D (one
//                N = D accumulator, D-blocked shared-memory panels).
struct FwdSpec {
    int D, BM, BN, nslot;
};
constexpr FwdSpec kFwdSpecs[] = {
    {64, 256, 128, 4},   // Q 2 x 16 KB + 4 x 16 KB ring (6, 8, 10 slots measured 0-5 % slower; 5, 7, 9 more)
    {128, 256, 128, 4},  // Q 2 x 32 KB + 4 x 32 KB ring + 32 KB staging for O's TMA stores
    {192, 128, 64, 7},   // Q 48 KB + 7 x 24 KB ring (4, 5 slots measured 4-13 % slower)
    {256, 128, 64, 4},   // Q 64 KB + 4 x 32 KB ring (3 slots measured 19 % slower)
};

// Tile rows of the backward kernels' streamed operands (TMA box heights).
constexpr int kDqKRows = 64;    // dQ kernel: 128 query rows per CTA, 64-key K/V tiles
constexpr int kDkdvQRows = 64;  // dK/dV kernel: 128 keys per CTA, 64-query Q/dO tiles

// Work order of a 1-D grid over (tile, batch*head).  Causal launches go by
// tile rank, rank 0 (the most K/V tiles) first, so that the hardware, which
// dispatches CTAs in index order, starts every SM on the longest tiles and
// fills the tail with short ones.  The ranks run across groups of `group`
// heads, one group after the other, so that the K/V (or Q/dO) tiles that a
// group's CTAs stream stay in L2 between the CTAs that read them; a group of
// every head is the plain rank order.  Non-causal tiles are equal, so the
// tiles of one head stay adjacent (they share its K/V in L2).
#ifdef __CUDACC__
__device__ __forceinline__ void tile_order_at(int L, int n_tiles, int n_bh, bool causal, int group, int *rank,
                                              int *bh) {
    if (causal && (group < 1 || group >= n_bh)) {
        *rank = L / n_bh;
        *bh = L % n_bh;
    } else if (causal) {
        const int g = group;
        const int per = n_tiles * g;        // items of a full group
        const int gi = L / per;             // L's group
        const int g0 = gi * g;              // its first head
        const int gs = min(g, n_bh - g0);   // its heads (the last group may have fewer)
        const int in = L - gi * per;
        *rank = in / gs;
        *bh = g0 + in % gs;
    } else {
        *rank = L % n_tiles;
        *bh = L / n_tiles;
    }
}

__device__ __forceinline__ void tile_order(int n_tiles, int n_bh, bool causal, int group, int *rank, int *bh) {
    tile_order_at(blockIdx.x, n_tiles, n_bh, causal, group, rank, bh);
}

// The k-th work item of CTA c in a persistent grid of G CTAs (one per SM): round k of the 1-D work
// order above is dealt out forwards in even rounds and backwards in odd ones, so a CTA that drew a heavy
// item in one round draws a light one in the next.  -1: no item for this CTA in round k.
__device__ __forceinline__ int persistent_work_index(int k, int n_work) {
    const int G = gridDim.x, c = blockIdx.x;
    const int Lw = k * G + ((k & 1) ? G - 1 - c : c);
    return Lw < n_work ? Lw : -1;
}
#endif

struct FwdArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int B, H, N, D;
    float scale;       // softmax scale
    float scale_log2;  // scale * log2(e): scores go straight to the base-2 domain
    int causal;
    int *status;       // device status word (bounded-wait failures)
    int num_sms;       // SMs of the device: the persistent forward runs one CTA per SM
    int head_group;    // heads per group of the causal work order (tile_order_at)
    // The persistent forwards' work counter (two ints, zero between launches: the next item to draw and
    // the CTAs that have stopped drawing; the last of them zeroes both).  Null: the static deal
    // persistent_work_index, used when the whole launch's K/V fits in L2.
    int *work;
};

struct BwdArgs {
    const void *q, *k, *v, *o, *dO;
    const float *lse;
    float *delta;        // written by the dQ kernel, read by the dK/dV kernel
    void *dq, *dk, *dv;  // grad_dtype
    int B, H, N, D;
    float scale, scale_log2;
    int causal;
    int grad_bf16;  // 1: gradients stored as bf16, 0: fp32
    int *status;
    int head_group;  // heads per group of the causal work order (tile_order_at)
};

// 5-GEMM comparator backward (bwd_atomic.cu): a.dq is the fp32 accumulator
// (B*H*N*D floats), dq_out the gradient in grad dtype; D = 128 only.
cudaError_t launch_bwd_atomic(const BwdArgs &a, void *dq_out, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t s);

// Decode (few query rows against a long key range), split over the keys.
constexpr int kNumSms = 152;  // GB300; used only when the device's own SM count cannot be read

struct DecodeArgs {
    const void *q, *k, *v;  // q [B, H, n_q, D]; k, v [B, H, N, D]; bf16
    void *o;                // [B, H, n_q, D] bf16
    float *lse;             // [B, H, n_q]
    float *workspace;       // O, m, l partials of every key chunk (decode_workspace_bytes)
    int B, H, n_q, N, D;
    int splits, chunk;      // key chunks per (batch, head), keys per chunk
    float scale_log2;
    int causal;
};

int decode_max_rows(int D);
// The key-chunk split (and so the workspace size) depends on the device's SM count.
void decode_split(int B, int H, int n_q, int N, int D, int num_sms, int *splits, int *chunk);
size_t decode_workspace_bytes(int B, int H, int n_q, int N, int D, int num_sms);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);

// Fixed scratch of fa_decode_noalloc (static device storage in decode.cu).
constexpr size_t kDecodeScratchBytes = size_t(16) << 20;
// Device address of the current device's scratch; the first call on a device
// looks it up (cudaGetSymbolAddress), later calls return the cached address.
cudaError_t decode_static_scratch(float **ptr);

// Tensor maps for one [B*H, N, D] bf16 tensor, box = {64, rows, 1}, 128-byte swizzle.
struct TmaPair {
    CUtensorMap map;
};

cudaError_t launch_fwd_f32(const FwdArgs &a, cudaStream_t s);
// `to`: O's tensor map (bf16, 64-column boxes of 128 rows, 128-byte swizzle), for the kernels whose
// epilogue stores O by TMA
cudaError_t launch_fwd_bf16(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                            const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t s);
cudaError_t launch_fwd_bf16_pair(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t s);
// fwd_bf16_duo.cu: D = 64, the two-tile persistent forward with one issuer warp and one P buffer per tile
cudaError_t launch_fwd_bf16_duo(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, cudaStream_t s);
// The dQ kernels also take O's tensor map (128-row boxes; its tile is staged for D_i = rowsum(dO * O))
// and dQ's (grad dtype, 128-byte boxes of 128 rows, 128-byte swizzle: the TMA stores of the epilogue).
cudaError_t launch_bwd_dq(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &to,
                          const CUtensorMap &tdq, cudaStream_t s);
// bwd_dq_k128.cu: the dQ kernel for D = 64 with 128-row K / V tiles (TMA boxes of 128 rows)
cudaError_t launch_bwd_dq_k128(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &to,
                               const CUtensorMap &tdq, cudaStream_t s);
// The dK/dV kernels also take dK's and dV's tensor maps (grad dtype, 128-byte boxes of 128 rows, 128-byte
// swizzle: the TMA stores of the epilogue).
// bwd_dkdv_q128.cu: the dK/dV kernel for D = 64 with 128-row Q / dO tiles (TMA boxes of 128 rows)
cudaError_t launch_bwd_dkdv_q128(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdk,
                                 const CUtensorMap &tdv, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                            const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdk,
                            const CUtensorMap &tdv, cudaStream_t s);
cudaError_t launch_selftest_timeout(int *status, int limit_us, cudaStream_t s);

// Head dimension a bf16 kernel is built for: the smallest of 64, 128, 192, 256 that holds D.  Any
// D that is a multiple of 8 (so a row is a whole number of 16-byte units) runs on that kernel: the
// TMA loads a 64-column panel that reaches past D with zeros, which add nothing to a score or an
// output column, and the kernels store only the D real columns (row stride D).
inline int kernel_head_dim(int D) { return D <= 64 ? 64 : D <= 128 ? 128 : D <= 192 ? 192 : 256; }

// K/V ring depth of the forward kernel of width D (a template argument of its launch).
constexpr int fwd_nslot(int D) {
    return D == 64 ? kFwdSpecs[0].nslot : D == 128 ? kFwdSpecs[1].nslot : D == 192 ? kFwdSpecs[2].nslot
                                                                                     : kFwdSpecs[3].nslot;
}

inline int fwd_block_n(int D) {
    for (const auto &sp : kFwdSpecs)
        if (sp.D == D) return sp.BN;
    return 0;
}

}  // namespace fa
