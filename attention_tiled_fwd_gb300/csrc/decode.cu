// decode.cu -- attention for a few query rows against a long key/value range
// ("decode": the metalworking "Flash Attention" page notes that one query
// row cannot fill a matrix-engine tile, so implementations ship a separate
// vector kernel).  Same mathematics as the forward: softmax(scale q K^T) V per
// query row, online base-2 softmax, L = m + ln(l); the n_q query rows are the
// last n_q positions, so with causal masking row i sees keys j <= N - n_q + i.
//
// The work is HBM-bound (each K/V byte is used by only n_q <= 16 rows), so it
// runs on the CUDA cores and is split over the key range (split-KV) to put
// enough CTAs on the GPU.  Two partial kernels, one combine:
//   decode_stream_kernel   n_q <= 4 (the common decode case).  No shared-memory
//                          staging: a group of D/16 lanes owns one key at a
//                          time, each lane 16 of its D columns (two 16-byte
//                          pieces, so one load instruction of the warp covers
//                          whole 128-byte row segments); K and V come straight
//                          from HBM with streaming 16-byte loads, double
//                          buffered in registers one step ahead.  q (times
//                          scale*log2 e) stays in registers; a score is a
//                          16-term dot product plus a shuffle reduction inside
//                          the group.  Each group keeps its own online-softmax
//                          state (m, l, O columns) with the branch-guarded
//                          rescale of the forward (O is rescaled only when the
//                          running max grows by more than 2^8), and the groups
//                          and warps are merged once at the end of the chunk;
//   decode_partial_kernel  5 <= n_q <= 16: K/V tiles staged into padded shared
//                          memory with cp.async (double-buffered); each warp
//                          owns 32 keys of a tile (lane = key) for every query
//                          row, keeps a running (m, l, O) per row, and the CTA
//                          merges its warps;
//   decode_combine_kernel  one thread per (row, column): merges the chunks'
//                          partials, O = sum_s 2^(m_s - M) O_s / L, and writes
//                          O (bf16) and the natural log-sum-exp.
// Both partial kernels write one partial (m, l, unnormalised O) per row and
// key chunk to the workspace (fp32): O partials [B*H][splits][n_q][D], then m
// [..][n_q], then l [..][n_q].  Every entry is written by the partial kernel
// before the combine kernel reads it (a chunk a row cannot see stores
// m = -inf, l = 0, O = 0), so the workspace needs no clearing.
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


// ---------------------------------------------------------------- n_q <= 4: streaming kernel
template <int D>
struct StreamCfg {
    static constexpr int kG = D / 16;                 // lanes per key; each lane owns 16 columns
    static constexpr int kKpp = 32 / kG;              // keys a warp covers per sub-step
    static constexpr int kWarps = 4;
    static constexpr int kSub = 2;                    // sub-steps per step (loaded together)
    static constexpr int kStep = kWarps * kKpp * kSub;  // keys per CTA step
};
constexpr int kStreamMaxQ = 4;
// CTAs per SM the launch bounds ask for: registers grow with the rows (q and O columns per row)
__host__ __device__ constexpr int stream_ctas_per_sm(int nq) { return nq == 1 ? 4 : nq == 2 ? 3 : 2; }

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    // read-once data: bypass L1 allocation
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void unpack8(const uint4 w, float *f) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

template <int D, int NQ>
__global__ void __launch_bounds__(StreamCfg<D>::kWarps * 32, stream_ctas_per_sm(NQ))
    decode_stream_kernel(DecodeArgs a) {
    using C = StreamCfg<D>;
    constexpr int G = C::kG, KPP = C::kKpp, W = C::kWarps, SUB = C::kSub, STEP = C::kStep, HALF = D / 2;
    __shared__ float mrg[W][NQ][D + 2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / G, gl = lane % G;
    const int split = blockIdx.x;
    const int bh = blockIdx.z * a.H + blockIdx.y;
    const int N = a.N;
    const int key_begin = split * a.chunk;
    const int key_end = min(N, key_begin + a.chunk);
    const __nv_bfloat16 *kbase = static_cast<const __nv_bfloat16 *>(a.k) + (size_t)bh * N * D;
    const __nv_bfloat16 *vbase = static_cast<const __nv_bfloat16 *>(a.v) + (size_t)bh * N * D;
    // this lane's columns: [8 gl, 8 gl + 8) and [D/2 + 8 gl, D/2 + 8 gl + 8)
    const int c0 = 8 * gl, c1 = HALF + 8 * gl;

    float qf[NQ][16];
    {
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q) + (size_t)bh * NQ * D;
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            unpack8(*reinterpret_cast<const uint4 *>(q + qi * D + c0), qf[qi]);
            unpack8(*reinterpret_cast<const uint4 *>(q + qi * D + c1), qf[qi] + 8);
#pragma unroll
            for (int e = 0; e < 16; ++e) qf[qi][e] *= a.scale_log2;
        }
    }
    float o[NQ][16], m[NQ], l[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        m[qi] = -INFINITY;
        l[qi] = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) o[qi][e] = 0.f;
    }
    // last key row qi may see
    const int lim0 = a.causal ? N - NQ : N - 1;
    const int lim_step = a.causal ? 1 : 0;

    // key of this lane in sub-step u of step t: each warp covers KPP * SUB consecutive keys per step
    auto key_of = [&](int t, int u) { return key_begin + t * STEP + (warp * SUB + u) * KPP + grp; };
    auto load = [&](int t, uint4 (&kb)[SUB][2], uint4 (&vb)[SUB][2]) {
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
            const int key = key_of(t, u);
            if (key < key_end) {
                const size_t row = (size_t)key * D;
                kb[u][0] = ldg_stream(kbase + row + c0);
                kb[u][1] = ldg_stream(kbase + row + c1);
                vb[u][0] = ldg_stream(vbase + row + c0);
                vb[u][1] = ldg_stream(vbase + row + c1);
            } else {
                kb[u][0] = kb[u][1] = vb[u][0] = vb[u][1] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };
    auto compute = [&](int t, const uint4 (&kb)[SUB][2], const uint4 (&vb)[SUB][2]) {
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
            const int key = key_of(t, u);
            float kf[16];
            unpack8(kb[u][0], kf);
            unpack8(kb[u][1], kf + 8);
            float sc[NQ];
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    s0 = fmaf(qf[qi][e], kf[e], s0);
                    s1 = fmaf(qf[qi][e + 1], kf[e + 1], s1);
                }
                sc[qi] = s0 + s1;
            }
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1) {
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) sc[qi] += __shfl_xor_sync(0xffffffffu, sc[qi], off);
            }
            float vf[16];
            unpack8(vb[u][0], vf);
            unpack8(vb[u][1], vf + 8);
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const bool visible = key < key_end && key <= lim0 + qi * lim_step;
                const float s = visible ? sc[qi] : -INFINITY;
                if (s > m[qi] + 8.f) {  // branch-guarded rescale; always taken by the first visible key
                    const float alpha = ex2_approx(m[qi] - s);
                    l[qi] *= alpha;
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[qi][e] *= alpha;
                    m[qi] = s;
                }
                const float p = visible ? ex2_approx(s - m[qi]) : 0.f;
                l[qi] += p;
#pragma unroll
                for (int e = 0; e < 16; ++e) o[qi][e] = fmaf(p, vf[e], o[qi][e]);
            }
        }
    };

    const int n_steps = (key_end - key_begin + STEP - 1) / STEP;
    uint4 ka[SUB][2], va[SUB][2], kb2[SUB][2], vb2[SUB][2];
    if (n_steps > 0) load(0, ka, va);
    for (int t = 0; t < n_steps; t += 2) {
        if (t + 1 < n_steps) load(t + 1, kb2, vb2);
        compute(t, ka, va);
        if (t + 1 < n_steps) {
            if (t + 2 < n_steps) load(t + 2, ka, va);
            compute(t + 1, kb2, vb2);
        }
    }

    // merge the groups of the warp (lanes differing in the group bits), then the warps
#pragma unroll
    for (int off = G; off < 32; off <<= 1) {
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[qi], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[qi], off);
            const float M = fmaxf(m[qi], mo);
            const float Mb = (M == -INFINITY) ? 0.f : M;
            const float fa = ex2_approx(m[qi] - Mb), fb = ex2_approx(mo - Mb);
            l[qi] = l[qi] * fa + lo * fb;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float oo = __shfl_xor_sync(0xffffffffu, o[qi][e], off);
                o[qi][e] = o[qi][e] * fa + oo * fb;
            }
            m[qi] = M;
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                mrg[warp][qi][c0 + e] = o[qi][e];
                mrg[warp][qi][c1 + e] = o[qi][8 + e];
            }
            if (gl == 0) {
                mrg[warp][qi][D] = m[qi];
                mrg[warp][qi][D + 1] = l[qi];
            }
        }
    }
    __syncthreads();
    const size_t part = ((size_t)bh * a.splits + split) * NQ;  // first row of this chunk's partials
    float *part_o = a.workspace;
    float *part_m = part_o + (size_t)a.B * a.H * a.splits * NQ * D;
    float *part_l = part_m + (size_t)a.B * a.H * a.splits * NQ;
    for (int idx = threadIdx.x; idx < NQ * D; idx += blockDim.x) {
        const int qi = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, mrg[w][qi][D]);
        const float Mb = (M == -INFINITY) ? 0.f : M;
        float O = 0.f, Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float f = ex2_approx(mrg[w][qi][D] - Mb);
            O = fmaf(mrg[w][qi][d], f, O);
            Lsum = fmaf(mrg[w][qi][D + 1], f, Lsum);
        }
        part_o[(part + qi) * D + d] = O;
        if (d == 0) {
            part_m[part + qi] = M;
            part_l[part + qi] = Lsum;
        }
    }
}

template <int D, int NQ>
cudaError_t launch_stream(const DecodeArgs &a, cudaStream_t s) {
    decode_stream_kernel<D, NQ><<<dim3(a.splits, a.H, a.B), StreamCfg<D>::kWarps * 32, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D><<<dim3(a.n_q, a.H, a.B), D, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t s) {
    switch (a.n_q) {
        case 1: return launch_stream<D, 1>(a, s);
        case 2: return launch_stream<D, 2>(a, s);
        case 3: return launch_stream<D, 3>(a, s);
        case 4: return launch_stream<D, 4>(a, s);
        default: break;
    }
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

void decode_split(int B, int H, int n_q, int N, int D, int *splits, int *chunk) {
    const long long bh = (long long)B * H;
    if (n_q <= kStreamMaxQ) {
        // Streaming kernel: pick the number of chunks per (batch, head) that minimises
        //   waves(s) * (keys per chunk + fixed cost per CTA),
        // waves(s) = ceil(B*H*s / resident CTAs), the fixed cost counted as 64 keys.
        const int step = D == 256 ? StreamCfg<256>::kStep : D == 128 ? StreamCfg<128>::kStep : StreamCfg<64>::kStep;
        const long long cap = (long long)kNumSms * stream_ctas_per_sm(n_q);
        const long long max_s = (N + step - 1) / step;
        long long best_s = 1;
        double best = 1e300;
        const long long s_hi = max_s < 4 * cap ? max_s : 4 * cap;
        for (long long sp = 1; sp <= s_hi; ++sp) {
            long long c = (N + sp - 1) / sp;
            c = (c + step - 1) / step * step;
            const long long real_s = (N + c - 1) / c;
            if (real_s != sp) continue;  // the same chunk as a smaller count
            const double waves = (double)((bh * sp + cap - 1) / cap);
            const double cost = waves * (double)(c + 64);
            if (cost < best * 0.999) {
                best = cost;
                best_s = sp;
            }
        }
        long long c = (N + best_s - 1) / best_s;
        c = (c + step - 1) / step * step;
        *chunk = (int)c;
        *splits = (int)((N + c - 1) / c);
        return;
    }
    const int tile = D == 256 ? DecodeCfg<256>::kTile : DecodeCfg<128>::kTile;
    // staged kernel: aim for kDecodeTargetCtas CTAs in total, each with at least one full stage of keys
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
    decode_split(B, H, n_q, N, D, &splits, &chunk);
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
