// decode.cu -- attention for a few query rows against a long key/value range
// ("decode": the metalworking "Flash Attention" page notes that one query
// row cannot fill a matrix-engine tile, so implementations ship a separate
// vector kernel).  Same mathematics as the forward: softmax(scale q K^T) V per
// query row, online base-2 softmax, L = m + ln(l); the n_q query rows are the
// last n_q positions, so with causal masking row i sees keys j <= N - n_q + i.
//
// The work is HBM-bound (each K/V byte is used by only n_q <= 16 rows), so it
// runs on the CUDA cores and is split over the key range (split-KV) to put
// enough CTAs on the GPU:
//   decode_partial_kernel  one CTA per (key chunk, head, batch): K/V tiles are
//                          staged into padded shared memory with cp.async
//                          (double-buffered); each warp owns 32 keys of a tile
//                          (lane = key) for every query row, keeps a running
//                          (m, l, O) per row, and the CTA merges its warps into
//                          one partial (m, l, unnormalised O) per row and chunk,
//                          written to the caller's workspace;
//   decode_combine_kernel  one thread per (row, column): merges the chunks'
//                          partials, O = sum_s 2^(m_s - M) O_s / L, and writes
//                          O (bf16) and the natural log-sum-exp.
// Workspace (fp32): O partials [B*H][splits][n_q][D], then m [..][n_q], then
// l [..][n_q].  Every entry is written by the partial kernel before the
// combine kernel reads it (a chunk a row cannot see stores m = -inf, l = 0,
// O = 0), so the workspace needs no clearing.
#include "fa_internal.h"
#include "sm100_ptx.cuh"
#include <cmath>
#include <mutex>

namespace fa {

// Scratch for fa_decode_noalloc: the same partials as the caller's workspace
// of fa_decode, held in the library's own static device storage (one copy per
// device, reserved when the module loads) so that the entry point allocates
// nothing.  Sizes that need more are rejected before launch.
static __device__ __align__(256) float g_decode_scratch[kDecodeScratchBytes / sizeof(float)];

namespace {

template <int D>
struct DecodeCfg {
    static constexpr int kWarps = (D == 256) ? 2 : 4;
    static constexpr int kTile = kWarps * 32;           // keys per stage
    static constexpr int kRow = D + 8;                   // padded bf16 row stride in shared memory
    static constexpr int kMaxQ = (D == 256) ? 8 : 16;    // query rows per launch
    static constexpr int kVec = D / 32;                  // output columns per lane
    static constexpr size_t kSmem = sizeof(float) * kMaxQ * D + 2ull * 2 * kTile * kRow * 2;
};

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, bool valid) {
    // 16-byte global -> shared copy; src-size 0 fills the destination with zeros without reading.
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

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

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::kWarps * 32) decode_partial_kernel(DecodeArgs a) {
    using C = DecodeCfg<D>;
    constexpr int W = C::kWarps, T = C::kTile, R = C::kRow, NQ = C::kMaxQ, V = C::kVec;
    extern __shared__ __align__(16) uint8_t smem[];
    float *q_s = reinterpret_cast<float *>(smem);                                  // [NQ][D], times scale*log2(e)
    __nv_bfloat16 *k_s = reinterpret_cast<__nv_bfloat16 *>(q_s + NQ * D);         // [2][T][R]
    __nv_bfloat16 *v_s = k_s + 2 * T * R;                                          // [2][T][R]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int bh = blockIdx.z * a.H + blockIdx.y;
    const int N = a.N, nq = a.n_q;
    const int key_begin = split * a.chunk;
    const int key_end = min(N, key_begin + a.chunk);
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q) + (size_t)bh * nq * D;
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k) + (size_t)bh * N * D;
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v) + (size_t)bh * N * D;

    for (int i = threadIdx.x; i < nq * D; i += blockDim.x)
        q_s[i] = __bfloat162float(q[i]) * a.scale_log2;

    // stage loader: T rows of K and of V, D*2 bytes each, as 16-byte chunks (rows past the end zero-fill)
    auto load_stage = [&](int st, int key0) {
        constexpr int kChunks = D / 8;
        for (int c = threadIdx.x; c < T * kChunks; c += blockDim.x) {
            const int r = c / kChunks, cc = c % kChunks;
            const int key = key0 + r;
            const bool valid = key < key_end;
            const size_t off = (size_t)(valid ? key : key_begin) * D + cc * 8;
            cp_async16(k_s + (st * T + r) * R + cc * 8, k + off, valid);
            cp_async16(v_s + (st * T + r) * R + cc * 8, v + off, valid);
        }
        cp_async_commit();
    };

    float m[NQ], l[NQ], o[NQ][V];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        m[qi] = -INFINITY;
        l[qi] = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) o[qi][e] = 0.f;
    }

    const int n_tiles = (key_end - key_begin + T - 1) / T;
    if (n_tiles > 0) load_stage(0, key_begin);
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) {
            load_stage(st ^ 1, key_begin + (t + 1) * T);
            cp_async_wait_prev();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();  // stage st (and, on the first pass, q_s) visible to every warp

        const int key = key_begin + t * T + warp * 32 + lane;
        const __nv_bfloat16 *krow = k_s + (st * T + warp * 32 + lane) * R;
        float s[NQ];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) s[qi] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
            const uint4 kv = *reinterpret_cast<const uint4 *>(krow + c * 8);
            const float kf[8] = {bf16lo(kv.x), bf16hi(kv.x), bf16lo(kv.y), bf16hi(kv.y),
                                 bf16lo(kv.z), bf16hi(kv.z), bf16lo(kv.w), bf16hi(kv.w)};
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                if (qi < nq) {
                    const float4 qa = *reinterpret_cast<const float4 *>(q_s + qi * D + c * 8);
                    const float4 qb = *reinterpret_cast<const float4 *>(q_s + qi * D + c * 8 + 4);
                    float acc = s[qi];
                    acc = fmaf(qa.x, kf[0], acc);
                    acc = fmaf(qa.y, kf[1], acc);
                    acc = fmaf(qa.z, kf[2], acc);
                    acc = fmaf(qa.w, kf[3], acc);
                    acc = fmaf(qb.x, kf[4], acc);
                    acc = fmaf(qb.y, kf[5], acc);
                    acc = fmaf(qb.z, kf[6], acc);
                    acc = fmaf(qb.w, kf[7], acc);
                    s[qi] = acc;
                }
            }
        }
        // online softmax per row (scores are already in the base-2 domain)
        float p[NQ];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            p[qi] = 0.f;
            if (qi < nq) {
                const int lim = a.causal ? N - nq + qi : N - 1;  // last visible key of row qi
                const float sv = (key < key_end && key <= lim) ? s[qi] : -INFINITY;
                const float m_new = fmaxf(m[qi], warp_max(sv));
                const float m_base = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = ex2_approx(m[qi] - m_base);
                p[qi] = ex2_approx(sv - m_base);
                l[qi] = l[qi] * alpha + warp_sum(p[qi]);
                m[qi] = m_new;
#pragma unroll
                for (int e = 0; e < V; ++e) o[qi][e] *= alpha;
            }
        }
        // O += P V: lane owns output columns [lane*V, lane*V + V)
        const __nv_bfloat16 *vtile = v_s + (st * T + warp * 32) * R + lane * V;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            float vf[V];
            if constexpr (V == 2) {
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(vtile + j * R);
                vf[0] = bf16lo(w0);
                vf[1] = bf16hi(w0);
            } else if constexpr (V == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(vtile + j * R);
                vf[0] = bf16lo(w.x); vf[1] = bf16hi(w.x); vf[2] = bf16lo(w.y); vf[3] = bf16hi(w.y);
            } else {
                const uint4 w = *reinterpret_cast<const uint4 *>(vtile + j * R);
                vf[0] = bf16lo(w.x); vf[1] = bf16hi(w.x); vf[2] = bf16lo(w.y); vf[3] = bf16hi(w.y);
                vf[4] = bf16lo(w.z); vf[5] = bf16hi(w.z); vf[6] = bf16lo(w.w); vf[7] = bf16hi(w.w);
            }
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                if (qi < nq) {
                    const float pj = __shfl_sync(0xffffffffu, p[qi], j);
#pragma unroll
                    for (int e = 0; e < V; ++e) o[qi][e] = fmaf(pj, vf[e], o[qi][e]);
                }
            }
        }
        __syncthreads();  // every warp is done with stage st before it is refilled
    }

    // merge the warps' states of each row: shared scratch [W][NQ][D + 2] over the (now idle) K stages
    float *mrg = reinterpret_cast<float *>(k_s);
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
            float *dst = mrg + (warp * NQ + qi) * (D + 2);
#pragma unroll
            for (int e = 0; e < V; ++e) dst[lane * V + e] = o[qi][e];
            if (lane == 0) {
                dst[D] = m[qi];
                dst[D + 1] = l[qi];
            }
        }
    }
    __syncthreads();
    const size_t part = ((size_t)bh * a.splits + split) * nq;  // first row of this chunk's partials
    float *part_o = a.workspace;
    float *part_m = part_o + (size_t)a.B * a.H * a.splits * nq * D;
    float *part_l = part_m + (size_t)a.B * a.H * a.splits * nq;
    for (int idx = threadIdx.x; idx < nq * D; idx += blockDim.x) {
        const int qi = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, mrg[(w * NQ + qi) * (D + 2) + D]);
        const float Mb = (M == -INFINITY) ? 0.f : M;
        float O = 0.f, Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float *src = mrg + (w * NQ + qi) * (D + 2);
            const float f = ex2_approx(src[D] - Mb);
            O = fmaf(src[d], f, O);
            Lsum = fmaf(src[D + 1], f, Lsum);
        }
        part_o[(part + qi) * D + d] = O;
        if (d == 0) {
            part_m[part + qi] = M;
            part_l[part + qi] = Lsum;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(DecodeArgs a) {
    const int qi = blockIdx.x, d = threadIdx.x;
    const int bh = blockIdx.z * a.H + blockIdx.y;
    const int nq = a.n_q, S = a.splits;
    const float *part_o = a.workspace;
    const float *part_m = part_o + (size_t)a.B * a.H * S * nq * D;
    const float *part_l = part_m + (size_t)a.B * a.H * S * nq;
    const size_t base = (size_t)bh * S * nq + qi;  // partial of chunk s is base + s * nq
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, part_m[base + (size_t)s * nq]);
    const float Mb = (M == -INFINITY) ? 0.f : M;
    float O = 0.f, Lsum = 0.f;
    for (int s = 0; s < S; ++s) {
        const size_t e = base + (size_t)s * nq;
        const float f = ex2_approx(part_m[e] - Mb);
        O = fmaf(part_o[e * D + d], f, O);
        Lsum = fmaf(part_l[e], f, Lsum);
    }
    const size_t row = (size_t)bh * nq + qi;
    static_cast<__nv_bfloat16 *>(a.o)[row * D + d] = __float2bfloat16_rn(O / Lsum);
    if (d == 0) a.lse[row] = (M + __log2f(Lsum)) * 0.69314718055994531f;
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t s) {
    using C = DecodeCfg<D>;
    auto kp = decode_partial_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    kp<<<dim3(a.splits, a.H, a.B), C::kWarps * 32, C::kSmem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D><<<dim3(a.n_q, a.H, a.B), D, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int decode_max_rows(int D) { return D == 256 ? DecodeCfg<256>::kMaxQ : DecodeCfg<128>::kMaxQ; }

void decode_split(int B, int H, int N, int D, int *splits, int *chunk) {
    const int tile = D == 256 ? DecodeCfg<256>::kTile : DecodeCfg<128>::kTile;
    // aim for kDecodeTargetCtas CTAs in total, each with at least one full stage of keys
    const long long bh = (long long)B * H;
    long long want = (kDecodeTargetCtas + bh - 1) / bh;
    const long long max_splits = (N + tile - 1) / tile;
    if (want > max_splits) want = max_splits;
    if (want < 1) want = 1;
    long long c = (N + want - 1) / want;
    c = (c + tile - 1) / tile * tile;
    *chunk = (int)c;
    *splits = (int)((N + c - 1) / c);
}

size_t decode_workspace_bytes(int B, int H, int n_q, int N, int D) {
    int splits, chunk;
    decode_split(B, H, N, D, &splits, &chunk);
    return sizeof(float) * (size_t)B * H * splits * n_q * (size_t)(D + 2);
}

namespace {
constexpr int kScratchDevices = 64;
float *g_scratch_addr[kScratchDevices];
std::mutex g_scratch_mu;
}  // namespace

cudaError_t decode_static_scratch(float **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        // once per device, with that device current; a failure is returned and retried on the next call
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<float *>(addr);
    }
    *ptr = g_scratch_addr[dev];
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_decode_d<64>(a, s);
        case 128: return launch_decode_d<128>(a, s);
        case 256: return launch_decode_d<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
