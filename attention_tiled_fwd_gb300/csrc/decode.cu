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
//   decode_stream_kernel   one CTA per (query-row block, key chunk, head,
//                          batch).  No shared-memory staging: a group of D/16
//                          lanes owns one key at a time, each lane 16 of its D
//                          columns (two 16-byte pieces, so each load
//                          instruction of the warp covers whole 128-byte row
//                          segments); K and V come straight from HBM with
//                          streaming 16-byte loads, double-buffered in
//                          registers one step ahead.  The block's query rows
//                          (times scale*log2 e) stay in registers; a score is a
//                          16-term dot product plus a shuffle reduction inside
//                          the group.  Each group keeps its own online-softmax
//                          state (m, l, O columns) with the branch-guarded
//                          rescale of the forward (O is rescaled only when the
//                          running max grows by more than 2^8), and groups and
//                          warps are merged once at the end of the chunk.
//                          Up to 4 rows per CTA (registers); n_q > 4 is cut
//                          into blocks of 4 rows whose CTAs are adjacent in
//                          launch order, so they read each chunk of K/V at
//                          about the same time and share it through L2;
//   decode_combine_kernel  one CTA per (row, head, batch): 8 warps merge the
//                          chunks' partials with an online rescale, lanes
//                          owning D/32 columns; O = sum_s 2^(m_s - M) O_s / L
//                          written as bf16, and the natural log-sum-exp.
// Workspace (fp32): O partials [B*H][splits][n_q][D], then m [..][n_q], then
// l [..][n_q].  Every entry is written by the stream kernel before the
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

constexpr int kMaxRows = 16;      // query rows per call
constexpr int kRowBlock = 4;      // query rows per CTA
constexpr int kCombineWarps = 8;

template <int D>
struct StreamCfg {
    static constexpr int kG = D / 16;                   // lanes per key; each lane owns 16 columns
    static constexpr int kKpp = 32 / kG;                // keys a warp covers per sub-step
    static constexpr int kWarps = 4;
    static constexpr int kSub = 2;                      // sub-steps per step (loaded together)
    static constexpr int kStep = kWarps * kKpp * kSub;  // keys per CTA step
};

// CTAs per SM the launch bounds ask for: registers grow with the rows (q and O columns per row)
__host__ __device__ constexpr int stream_ctas_per_sm(int nq) { return nq == 1 ? 4 : nq == 2 ? 3 : 2; }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

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

// NQ = rows per CTA.  blockIdx.x = split * row_blocks + row block; the block's
// rows are [NQ * rb, NQ * rb + nvalid), nvalid = min(NQ, n_q - NQ * rb); rows
// past nvalid are computed with q = 0 and not stored.
template <int D, int NQ>
__global__ void __launch_bounds__(StreamCfg<D>::kWarps * 32, stream_ctas_per_sm(NQ))
    decode_stream_kernel(DecodeArgs a) {
    using C = StreamCfg<D>;
    constexpr int G = C::kG, KPP = C::kKpp, W = C::kWarps, SUB = C::kSub, STEP = C::kStep, HALF = D / 2;
    __shared__ float mrg[W][NQ][D + 2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / G, gl = lane % G;
    const int row_blocks = (a.n_q + NQ - 1) / NQ;
    const int rb = blockIdx.x % row_blocks;
    const int split = blockIdx.x / row_blocks;
    const int row0 = rb * NQ;
    const int nvalid = min(NQ, a.n_q - row0);
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
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q) + ((size_t)bh * a.n_q + row0) * D;
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            if (qi < nvalid) {
                unpack8(*reinterpret_cast<const uint4 *>(q + qi * D + c0), qf[qi]);
                unpack8(*reinterpret_cast<const uint4 *>(q + qi * D + c1), qf[qi] + 8);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) qf[qi][e] = 0.f;
            }
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
    // last key block row qi may see
    const int lim0 = a.causal ? N - a.n_q + row0 : N - 1;
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
    const size_t part = ((size_t)bh * a.splits + split) * a.n_q + row0;  // this block's first partial row
    float *part_o = a.workspace;
    float *part_m = part_o + (size_t)a.B * a.H * a.splits * a.n_q * D;
    float *part_l = part_m + (size_t)a.B * a.H * a.splits * a.n_q;
    for (int idx = threadIdx.x; idx < nvalid * D; idx += blockDim.x) {
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

// One CTA per (row, head, batch); warp w merges chunks w, w + 8, ... online, then the warps merge.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(DecodeArgs a) {
    constexpr int V = D / 32;  // columns per lane
    __shared__ float sm_o[kCombineWarps][D];
    __shared__ float sm_m[kCombineWarps], sm_l[kCombineWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qi = blockIdx.x;
    const int bh = blockIdx.z * a.H + blockIdx.y;
    const int nq = a.n_q, S = a.splits;
    const float *part_o = a.workspace;
    const float *part_m = part_o + (size_t)a.B * a.H * S * nq * D;
    const float *part_l = part_m + (size_t)a.B * a.H * S * nq;
    const size_t base = (size_t)bh * S * nq + qi;  // partial of chunk s is base + s * nq

    float M = -INFINITY, L = 0.f, O[V];
#pragma unroll
    for (int c = 0; c < V; ++c) O[c] = 0.f;
    for (int s = warp; s < S; s += kCombineWarps) {
        const size_t e = base + (size_t)s * nq;
        const float ms = part_m[e];
        if (ms == -INFINITY) continue;  // a chunk this row cannot see (l = 0, O = 0)
        const float ls = part_l[e];
        const float *os = part_o + e * D + lane * V;
        float ov[V];
        if constexpr (V == 2) {
            const float2 t = *reinterpret_cast<const float2 *>(os);
            ov[0] = t.x;
            ov[1] = t.y;
        } else {
#pragma unroll
            for (int c = 0; c < V; c += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(os + c);
                ov[c] = t.x;
                ov[c + 1] = t.y;
                ov[c + 2] = t.z;
                ov[c + 3] = t.w;
            }
        }
        const float Mn = fmaxf(M, ms);
        const float fo = ex2_approx(M - Mn), fs = ex2_approx(ms - Mn);  // M = -inf gives fo = 0
        L = L * fo + ls * fs;
#pragma unroll
        for (int c = 0; c < V; ++c) O[c] = O[c] * fo + ov[c] * fs;
        M = Mn;
    }
#pragma unroll
    for (int c = 0; c < V; ++c) sm_o[warp][lane * V + c] = O[c];
    if (lane == 0) {
        sm_m[warp] = M;
        sm_l[warp] = L;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float Mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w) Mx = fmaxf(Mx, sm_m[w]);
        const float Mb = (Mx == -INFINITY) ? 0.f : Mx;
        float Ot = 0.f, Lt = 0.f;
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w) {
            const float f = ex2_approx(sm_m[w] - Mb);
            Ot = fmaf(sm_o[w][d], f, Ot);
            Lt = fmaf(sm_l[w], f, Lt);
        }
        const size_t row = (size_t)bh * nq + qi;
        static_cast<__nv_bfloat16 *>(a.o)[row * D + d] = __float2bfloat16_rn(Ot / Lt);
        if (d == 0) a.lse[row] = (Mx + __log2f(Lt)) * 0.69314718055994531f;
    }
}

template <int D, int NQ>
cudaError_t launch_stream(const DecodeArgs &a, cudaStream_t s) {
    const int row_blocks = (a.n_q + NQ - 1) / NQ;
    decode_stream_kernel<D, NQ><<<dim3(a.splits * row_blocks, a.H, a.B), StreamCfg<D>::kWarps * 32, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D><<<dim3(a.n_q, a.H, a.B), kCombineWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t s) {
    switch (a.n_q) {
        case 1: return launch_stream<D, 1>(a, s);
        case 2: return launch_stream<D, 2>(a, s);
        case 3: return launch_stream<D, 3>(a, s);
        default: return launch_stream<D, kRowBlock>(a, s);
    }
}

constexpr int kScratchDevices = 64;
float *g_scratch_addr[kScratchDevices];
std::mutex g_scratch_mu;

}  // namespace

int decode_max_rows(int) { return kMaxRows; }

void decode_split(int B, int H, int n_q, int N, int D, int num_sms, int *splits, int *chunk) {
    // Pick the number of key chunks per (batch, head) that minimises
    //   waves(s) * (keys per chunk + a fixed cost per CTA, counted as 64 keys),
    // waves(s) = ceil(CTAs / resident CTAs), CTAs = B * H * row blocks * s, for a device of num_sms SMs.
    const int rows = n_q < kRowBlock ? n_q : kRowBlock;
    const long long units = (long long)B * H * ((n_q + rows - 1) / rows);
    const int step = D == 256 ? StreamCfg<256>::kStep : D == 128 ? StreamCfg<128>::kStep : StreamCfg<64>::kStep;
    const long long cap = (long long)(num_sms > 0 ? num_sms : kNumSms) * stream_ctas_per_sm(rows);
    const long long max_s = (N + step - 1) / step;
    const long long s_hi = max_s < 4 * cap ? max_s : 4 * cap;
    long long best_s = 1;
    double best = 1e300;
    for (long long sp = 1; sp <= s_hi; ++sp) {
        long long c = (N + sp - 1) / sp;
        c = (c + step - 1) / step * step;
        if ((N + c - 1) / c != sp) continue;  // the same chunk as a smaller count
        const double waves = (double)((units * sp + cap - 1) / cap);
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
}

size_t decode_workspace_bytes(int B, int H, int n_q, int N, int D, int num_sms) {
    int splits, chunk;
    decode_split(B, H, n_q, N, D, num_sms, &splits, &chunk);
    return sizeof(float) * (size_t)B * H * splits * n_q * (size_t)(D + 2);
}

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
