// fwd_f32.cu -- exact fp32 forward on the CUDA cores (FFMA), for callers that
// need fp32 inputs and outputs.
//
// Same tiled algorithm as the tensor-core path ("Learning Metal with
// FlashAttention", section "FlashAttention": running max m, running sum l,
// unnormalised output rescaled by exp(m - m_new) per K/V tile, divided by l
// after the last tile; launch grid (query tile, head, batch)), with the
// base-2 exponent and causal tile skipping of the metalworking "Flash
// Attention" page (kernel anatomy items 3-4).
//
// CTA = 8 warps x 8 query rows = 64 rows; K/V tiles of 32 keys staged in
// shared memory (K rows padded by one float against bank conflicts).  Within
// a tile, lane j scores key j for each of its warp's rows, the row max / sum
// are warp reductions, and lane t owns output columns t, t+32, ...
// Any D that is a multiple of 4 up to 256 runs: the staged tiles are D
// rounded up to a multiple of 32 wide, the extra columns zero (they add
// nothing to a score and their outputs are not stored).
#include "fa_internal.h"
#include <cfloat>
#include <cmath>

namespace fa {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr int kWarps = 8;
constexpr int kBM = kRowsPerWarp * kWarps;  // 64 query rows per CTA
constexpr int kBN = 32;                     // keys per tile (one per lane)

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int DPL>  // head dimension / 32, rounded up (columns per lane)
__global__ void __launch_bounds__(kWarps * 32) fwd_f32_kernel(FwdArgs a) {
    constexpr int DP = DPL * 32;  // staged width
    const int D = a.D;            // row stride and stored columns; D <= DP
    extern __shared__ float sm[];
    float *q_s = sm;                      // [kBM][DP]
    float *k_s = q_s + kBM * DP;          // [kBN][DP + 1]
    float *v_s = k_s + kBN * (DP + 1);    // [kBN][DP]

    int rank, bh;
    tile_order((a.N + kBM - 1) / kBM, a.B * a.H, a.causal, a.head_group, &rank, &bh);
    const int q_tile = (a.N + kBM - 1) / kBM - 1 - rank;  // causal: the last query tile has the most keys
    const int N = a.N;
    const float *q = static_cast<const float *>(a.q) + (size_t)bh * N * D;
    const float *k = static_cast<const float *>(a.k) + (size_t)bh * N * D;
    const float *v = static_cast<const float *>(a.v) + (size_t)bh * N * D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = q_tile * kBM;

    for (int idx = threadIdx.x; idx < kBM * DP; idx += blockDim.x) {
        int r = idx / DP, c = idx % DP;
        q_s[idx] = (row0 + r < N && c < D) ? q[(size_t)(row0 + r) * D + c] : 0.f;
    }

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[r][t] = 0.f;
    }

    const int kv_end = a.causal ? min(N, row0 + kBM) : N;
    const int n_tiles = (kv_end + kBN - 1) / kBN;
    for (int jt = 0; jt < n_tiles; ++jt) {
        const int key0 = jt * kBN;
        __syncthreads();  // previous tile fully consumed (and q_s written on the first pass)
        for (int idx = threadIdx.x; idx < kBN * DP; idx += blockDim.x) {
            int r = idx / DP, c = idx % DP;
            bool ok = key0 + r < N && c < D;
            k_s[r * (DP + 1) + c] = ok ? k[(size_t)(key0 + r) * D + c] : 0.f;
            v_s[r * DP + c] = ok ? v[(size_t)(key0 + r) * D + c] : 0.f;
        }
        __syncthreads();
        const int key = key0 + lane;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int row = row0 + warp * kRowsPerWarp + r;
            const float *qr = q_s + (warp * kRowsPerWarp + r) * DP;
            float s = 0.f;
#pragma unroll 8
            for (int d = 0; d < DP; ++d) s = fmaf(qr[d], k_s[lane * (DP + 1) + d], s);
            s *= a.scale_log2;  // base-2 domain
            if (key >= N || (a.causal && key > row)) s = -INFINITY;
            const float m_new = fmaxf(m[r], warp_max(s));
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = exp2f(m[r] - m_use);
            const float p = exp2f(s - m_use);
            l[r] = l[r] * alpha + warp_sum(p);
            m[r] = m_new;
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[r][t] *= alpha;
#pragma unroll 4
            for (int j = 0; j < kBN; ++j) {
                const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
                for (int t = 0; t < DPL; ++t) acc[r][t] = fmaf(pj, v_s[j * DP + t * 32 + lane], acc[r][t]);
            }
        }
    }

    float *o = static_cast<float *>(a.o) + (size_t)bh * N * D;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = row0 + warp * kRowsPerWarp + r;
        if (row >= N) continue;
        const float inv = 1.f / l[r];
#pragma unroll
        for (int t = 0; t < DPL; ++t)
            if (t * 32 + lane < D) o[(size_t)row * D + t * 32 + lane] = acc[r][t] * inv;
        if (lane == 0) a.lse[(size_t)bh * N + row] = (m[r] + log2f(l[r])) * 0.69314718055994531f;
    }
}

template <int DPL>
cudaError_t launch_dpl(const FwdArgs &a, cudaStream_t s) {
    constexpr int DP = DPL * 32;
    const size_t smem = sizeof(float) * (size_t)(kBM * DP + kBN * (DP + 1) + kBN * DP);
    cudaError_t e = cudaFuncSetAttribute(fwd_f32_kernel<DPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(((a.N + kBM - 1) / kBM) * a.H * a.B);
    fwd_f32_kernel<DPL><<<grid, kWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs &a, cudaStream_t s) {
    switch ((a.D + 31) / 32) {
        case 1: return launch_dpl<1>(a, s);
        case 2: return launch_dpl<2>(a, s);
        case 3: return launch_dpl<3>(a, s);
        case 4: return launch_dpl<4>(a, s);
        case 5: return launch_dpl<5>(a, s);
        case 6: return launch_dpl<6>(a, s);
        case 7: return launch_dpl<7>(a, s);
        case 8: return launch_dpl<8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
