// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// TMA descriptor encoding, and launches on the caller's stream.
//
// Nothing here allocates device memory.  The only device-side state is the
// library's own static storage: the status word below (one int per device),
// which kernels update when a bounded wait runs out, and a ring of work
// counters for the persistent forwards (each zeroed again by the launch that
// used it).
#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm100_ptx.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

namespace fa {

__device__ int g_status_word;

// Work counters (two ints each) of the persistent forwards, handed out in turn, so that launches in
// flight on different streams draw from different counters.
constexpr int kWorkCounters = 1024;
__device__ int g_work_counters[2 * kWorkCounters];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int status_code = 0;  // FA_OK or the fa_status of the failed set-up
    int *status_word = nullptr;
    int num_sms = kNumSms;  // the device's SM count (sizes persistent grids)
    long long l2_bytes = 0;  // the device's L2 size (sizes the groups of the causal work order)
    int *work_counters = nullptr;
    std::atomic<unsigned> work_seq{0};
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device set-up: architecture check and the status word's device address.
int device_state(int *dev_out, DeviceState **st_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    // Bind the device's primary context to the calling thread: a thread that has made no runtime
    // call yet (a worker thread, autograd's backward thread) has no current context, and the
    // tensor-map encoder is a driver call that needs one.
    if (cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FA_ERR_CUDA;
        st.num_sms = prop.multiProcessorCount > 0 ? prop.multiProcessorCount : kNumSms;
        st.l2_bytes = prop.l2CacheSize;
        if (!(prop.major == 10 && prop.minor == 3)) {
            st.status_code = FA_ERR_DEVICE;  // kernels are built for sm_103a only
        } else if (cudaGetSymbolAddress(reinterpret_cast<void **>(&st.status_word), g_status_word) != cudaSuccess ||
                   cudaGetSymbolAddress(reinterpret_cast<void **>(&st.work_counters), g_work_counters) !=
                       cudaSuccess) {
            st.status_code = FA_ERR_CUDA;
        } else {
            st.status_code = FA_OK;
        }
        if (!g_encode && st.status_code == FA_OK) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                st.status_code = FA_ERR_CUDA;
            else
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        st.ready = true;
    }
    *dev_out = dev;
    *st_out = &st;
    return st.status_code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device-accessible (device or managed memory on the current device).
int check_device_ptr(const void *p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_DEVICE_PTR;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return FA_ERR_DEVICE_PTR;
    return FA_OK;
}

int check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (!p) return FA_ERR_NULL;
    for (const void *p : ptrs)
        if (!aligned16(p)) return FA_ERR_ALIGN;
    for (const void *p : ptrs) {
        int rc = check_device_ptr(p);
        if (rc != FA_OK) return rc;
    }
    return FA_OK;
}

int check_shape(int B, int H, int N, int D, float scale) {
    if (B < 1 || H < 1 || N < 1 || D < 1) return FA_ERR_SHAPE;
    if (B > 65535 || H > 65535) return FA_ERR_SHAPE;  // grid y / z limits
    if ((long long)B * H * (long long)N > (1ll << 31) - 1) return FA_ERR_SHAPE;
    if (!std::isfinite(scale)) return FA_ERR_SCALE;
    return FA_OK;
}

// [B*H, N, D] bf16 or fp32 tensor, box {128 bytes of a row, rows, 1}, 128-byte swizzle, zero fill out of
// bounds (loads) and clipping (stores).
int encode_3d(CUtensorMap *map, const void *base, int BH, int N, int D, int box_rows, bool f32) {
    const int elt = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * elt, (cuuint64_t)N * D * elt};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elt), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// [B*H, N, D] bf16 tensor, box {64, rows, 1}, 128-byte swizzle, zero fill out of bounds.
int encode_bf16_3d(CUtensorMap *map, const void *base, int BH, int N, int D, int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

float log2e() { return 1.4426950408889634f; }

// bf16 head dimensions the tensor-core kernels take: a multiple of 8 (whole 16-byte units per row, as
// the TMA needs for the row stride) up to 256; each runs on the kernel of width kernel_head_dim(D).
bool bf16_head_dim_ok(int D) { return D >= 8 && D <= 256 && D % 8 == 0; }

// SM count of the current device for the host-side size queries, which must also answer without a
// usable device (they make no launch): the GB300 count when it cannot be read.
int current_num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        cudaGetLastError();
        return kNumSms;
    }
    return sms > 0 ? sms : kNumSms;
}

// Heads per group of the causal work order (tile_order_at).  A launch streams two [N, D] bf16 operands per
// head (K and V, or Q and dO); while those of every head fit in three quarters of L2 the order is the plain
// rank order over all heads, otherwise a group holds as many heads as fit in a quarter of it (at least
// one), so that its operands stay in L2 while the group's CTAs read them.  (Three eighths, a half, five
// eighths and three quarters of L2 measured 0-3 % slower at B=1 H=32 N=32768 D=64 and N=16384 D=128.)
int causal_head_group(const DeviceState &st, int B, int H, int N, int D) {
    const int n_bh = B * H;
    const double per_head = 4.0 * N * D;
    const double l2 = st.l2_bytes > 0 ? (double)st.l2_bytes : 126.0 * (1 << 20);
    if (per_head * n_bh <= 0.75 * l2) return n_bh;
    return std::max(1, std::min(n_bh, (int)(0.25 * l2 / per_head)));
}

// The persistent forwards draw their blocks from a work counter when the causal order runs by groups of
// heads (only drawing in turn balances such a sequence); with one group they use the static deal.
int *forward_work_counter(DeviceState &st, int head_group, int B, int H, int causal) {
    if (!causal || head_group >= B * H) return nullptr;
    return st.work_counters + 2 * (st.work_seq.fetch_add(1, std::memory_order_relaxed) % kWorkCounters);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" int fa_forward(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N,
                          int D, float scale, int causal, int dtype, void *stream) {
    int rc = check_shape(B, H, N, D, scale);
    if (rc != FA_OK) return rc;
    if (dtype == FA_BF16) {
        if (!bf16_head_dim_ok(D)) return FA_ERR_HEAD_DIM;
    } else if (dtype == FA_F32) {
        if (D % 4 != 0 || D > 256) return FA_ERR_HEAD_DIM;
    } else {
        return FA_ERR_DTYPE;
    }
    rc = check_ptrs({q, k, v, o, lse});
    if (rc != FA_OK) return rc;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;

    // The D = 128 kernel deals its blocks statically, and so keeps the plain rank order over all heads: handing
    // its issuer warp drawn blocks measured 10-15 % slower.  The D = 64 kernel draws them (a work counter) when
    // the order runs by groups; the other kernels launch one CTA per tile, which the hardware hands out in turn.
    const int Dk = dtype == FA_BF16 ? kernel_head_dim(D) : 0;
    const int group = Dk == 128 ? B * H : causal_head_group(*st, B, H, N, D);
    FwdArgs a{q, k, v, o, lse, B, H, N, D, scale, scale * log2e(), causal ? 1 : 0, st->status_word, st->num_sms,
              group, nullptr};
    if (Dk == 64) a.work = forward_work_counter(*st, group, B, H, causal);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == FA_F32) {
        e = launch_fwd_f32(a, s);
    } else {
        CUtensorMap tq, tk, tv, to;
        const int bn = fwd_block_n(kernel_head_dim(D));
        if (encode_bf16_3d(&tq, q, B * H, N, D, 128) != FA_OK || encode_bf16_3d(&tk, k, B * H, N, D, bn) != FA_OK ||
            encode_bf16_3d(&tv, v, B * H, N, D, bn) != FA_OK || encode_bf16_3d(&to, o, B * H, N, D, 128) != FA_OK)
            return FA_ERR_CUDA;
        e = launch_fwd_bf16(a, tq, tk, tv, to, s);
    }
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fa_backward_dq(const void *q, const void *k, const void *v, const void *o, const void *dO,
                              const float *lse, float *delta, void *dq, int B, int H, int N, int D, float scale,
                              int causal, int dtype, int grad_dtype, void *stream) {
    int rc = check_shape(B, H, N, D, scale);
    if (rc != FA_OK) return rc;
    if (dtype != FA_BF16 && dtype != FA_F32) return FA_ERR_DTYPE;
    if (grad_dtype != FA_BF16 && grad_dtype != FA_F32) return FA_ERR_DTYPE;
    if (dtype != FA_BF16) return FA_ERR_DTYPE;  // the split backward runs on bf16 inputs
    if (!bf16_head_dim_ok(D)) return FA_ERR_HEAD_DIM;
    rc = check_ptrs({q, k, v, o, dO, lse, delta, dq});
    if (rc != FA_OK) return rc;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    BwdArgs a{q, k, v, o, dO, lse, delta, dq, nullptr, nullptr, B, H, N, D, scale, scale * log2e(),
              causal ? 1 : 0, grad_dtype == FA_BF16 ? 1 : 0, st->status_word, causal_head_group(*st, B, H, N, D)};
    CUtensorMap tq, tk, tv, tdo, to, tdq;
    // D <= 64 runs the 128-key-tile kernel (its score products are N = 128 MMAs); wider heads the 64-key one
    const int Dk = kernel_head_dim(D);
    const int kv_rows = Dk == 64 ? 128 : kDqKRows;
    if (encode_bf16_3d(&tq, q, B * H, N, D, 128) != FA_OK ||
        encode_bf16_3d(&tk, k, B * H, N, D, kv_rows) != FA_OK ||
        encode_bf16_3d(&tv, v, B * H, N, D, kv_rows) != FA_OK ||
        encode_bf16_3d(&tdo, dO, B * H, N, D, 128) != FA_OK || encode_bf16_3d(&to, o, B * H, N, D, 128) != FA_OK ||
        encode_3d(&tdq, dq, B * H, N, D, 128, grad_dtype == FA_F32) != FA_OK)
        return FA_ERR_CUDA;
    cudaError_t e = Dk == 64
                        ? launch_bwd_dq_k128(a, tq, tk, tv, tdo, to, tdq, reinterpret_cast<cudaStream_t>(stream))
                        : launch_bwd_dq(a, tq, tk, tv, tdo, to, tdq, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fa_backward_dkdv(const void *q, const void *k, const void *v, const void *dO, const float *lse,
                                const float *delta, void *dk, void *dv, int B, int H, int N, int D, float scale,
                                int causal, int dtype, int grad_dtype, void *stream) {
    int rc = check_shape(B, H, N, D, scale);
    if (rc != FA_OK) return rc;
    if (dtype != FA_BF16 && dtype != FA_F32) return FA_ERR_DTYPE;
    if (grad_dtype != FA_BF16 && grad_dtype != FA_F32) return FA_ERR_DTYPE;
    if (dtype != FA_BF16) return FA_ERR_DTYPE;
    if (!bf16_head_dim_ok(D)) return FA_ERR_HEAD_DIM;
    rc = check_ptrs({q, k, v, dO, lse, delta, dk, dv});
    if (rc != FA_OK) return rc;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    BwdArgs a{q, k, v, nullptr, dO, lse, const_cast<float *>(delta), nullptr, dk, dv, B, H, N, D, scale,
              scale * log2e(), causal ? 1 : 0, grad_dtype == FA_BF16 ? 1 : 0, st->status_word,
              causal_head_group(*st, B, H, N, D)};
    CUtensorMap tq, tk, tv, tdo, tdk, tdv;
    // D <= 64 runs the 128-query-tile kernel (its score products are N = 128 MMAs); wider heads the 64-query one
    const int Dk = kernel_head_dim(D);
    const int q_rows = Dk == 64 ? 128 : kDkdvQRows;
    if (encode_bf16_3d(&tq, q, B * H, N, D, q_rows) != FA_OK ||
        encode_bf16_3d(&tk, k, B * H, N, D, 128) != FA_OK || encode_bf16_3d(&tv, v, B * H, N, D, 128) != FA_OK ||
        encode_bf16_3d(&tdo, dO, B * H, N, D, q_rows) != FA_OK ||
        encode_3d(&tdk, dk, B * H, N, D, 128, grad_dtype == FA_F32) != FA_OK ||
        encode_3d(&tdv, dv, B * H, N, D, 128, grad_dtype == FA_F32) != FA_OK)
        return FA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = Dk == 64 ? launch_bwd_dkdv_q128(a, tq, tk, tv, tdo, tdk, tdv, s)
                             : launch_bwd_dkdv(a, tq, tk, tv, tdo, tdk, tdv, s);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fa_backward_atomic(const void *q, const void *k, const void *v, const void *o, const void *dO,
                                  const float *lse, float *delta, void *dq, void *dk, void *dv, float *dq_accum,
                                  size_t dq_accum_bytes, int B, int H, int N, int D, float scale, int causal,
                                  int dtype, int grad_dtype, void *stream) {
    int rc = check_shape(B, H, N, D, scale);
    if (rc != FA_OK) return rc;
    if (dtype != FA_BF16 && dtype != FA_F32) return FA_ERR_DTYPE;
    if (grad_dtype != FA_BF16 && grad_dtype != FA_F32) return FA_ERR_DTYPE;
    if (dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 128) return FA_ERR_HEAD_DIM;
    rc = check_ptrs({q, k, v, o, dO, lse, delta, dq, dk, dv, dq_accum});
    if (rc != FA_OK) return rc;
    if (dq_accum_bytes < (size_t)B * H * N * D * sizeof(float)) return FA_ERR_WORKSPACE;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    BwdArgs a{q, k, v, o, dO, lse, delta, dq_accum, dk, dv, B, H, N, D, scale, scale * log2e(),
              causal ? 1 : 0, grad_dtype == FA_BF16 ? 1 : 0, st->status_word, causal_head_group(*st, B, H, N, D)};
    CUtensorMap tq, tk, tv, tdo;
    if (encode_bf16_3d(&tq, q, B * H, N, D, kDkdvQRows) != FA_OK || encode_bf16_3d(&tk, k, B * H, N, D, 128) != FA_OK ||
        encode_bf16_3d(&tv, v, B * H, N, D, 128) != FA_OK || encode_bf16_3d(&tdo, dO, B * H, N, D, kDkdvQRows) != FA_OK)
        return FA_ERR_CUDA;
    cudaError_t e = launch_bwd_atomic(a, dq, tq, tk, tv, tdo, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

namespace {
int check_decode(int B, int H, int n_q, int N, int D, float scale) {
    int rc = check_shape(B, H, N, D, scale);
    if (rc != FA_OK) return rc;
    if (D != 64 && D != 128 && D != 256) return FA_ERR_HEAD_DIM;
    if (n_q < 1 || n_q > decode_max_rows(D) || n_q > N) return FA_ERR_SHAPE;
    if ((long long)B * H * (long long)n_q > (1ll << 31) - 1) return FA_ERR_SHAPE;
    return FA_OK;
}
}  // namespace

extern "C" int fa_decode_workspace_bytes(int B, int H, int n_q, int N, int D, size_t *bytes) {
    if (!bytes) return FA_ERR_NULL;
    int rc = check_decode(B, H, n_q, N, D, 1.f);
    if (rc != FA_OK) return rc;
    *bytes = decode_workspace_bytes(B, H, n_q, N, D, current_num_sms());
    return FA_OK;
}

extern "C" int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int n_q,
                         int N, int D, float scale, int causal, void *workspace, size_t workspace_bytes,
                         void *stream) {
    int rc = check_decode(B, H, n_q, N, D, scale);
    if (rc != FA_OK) return rc;
    rc = check_ptrs({q, k, v, o, lse, workspace});
    if (rc != FA_OK) return rc;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    if (workspace_bytes < decode_workspace_bytes(B, H, n_q, N, D, st->num_sms)) return FA_ERR_WORKSPACE;
    DecodeArgs a{q, k, v, o, lse, static_cast<float *>(workspace), B, H, n_q, N, D, 0, 0, scale * log2e(),
                 causal ? 1 : 0};
    decode_split(B, H, n_q, N, D, st->num_sms, &a.splits, &a.chunk);
    cudaError_t e = launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

static_assert(kDecodeScratchBytes == FA_DECODE_NOALLOC_SCRATCH_BYTES, "scratch size differs from fa.h");

// fa_decode with the partials in the library's static scratch instead of a
// caller workspace: same validation and kernels, no allocation anywhere.
extern "C" int fa_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                 int n_q, int N, int D, float scale, int causal, void *stream) {
    int rc = check_decode(B, H, n_q, N, D, scale);
    if (rc != FA_OK) return rc;
    if (decode_workspace_bytes(B, H, n_q, N, D, current_num_sms()) > kDecodeScratchBytes)
        return FA_ERR_SCRATCH_LIMIT;
    rc = check_ptrs({q, k, v, o, lse});
    if (rc != FA_OK) return rc;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    if (decode_workspace_bytes(B, H, n_q, N, D, st->num_sms) > kDecodeScratchBytes) return FA_ERR_SCRATCH_LIMIT;
    float *scratch = nullptr;
    if (decode_static_scratch(&scratch) != cudaSuccess) return FA_ERR_CUDA;
    DecodeArgs a{q, k, v, o, lse, scratch, B, H, n_q, N, D, 0, 0, scale * log2e(), causal ? 1 : 0};
    decode_split(B, H, n_q, N, D, st->num_sms, &a.splits, &a.chunk);
    cudaError_t e = launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_SHAPE: return "invalid shape (B, H, N must be >= 1 and within index limits)";
        case FA_ERR_HEAD_DIM: return "head dimension not supported for this dtype / pass";
        case FA_ERR_DTYPE: return "unsupported dtype or grad_dtype";
        case FA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case FA_ERR_SCALE: return "scale is not finite";
        case FA_ERR_CUDA: return "CUDA runtime error";
        case FA_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
        case FA_ERR_DEVICE_PTR: return "pointer is not device-accessible memory";
        case FA_ERR_DEVICE: return "current device is not sm_103 (GB300)";
        case FA_ERR_WORKSPACE: return "workspace smaller than fa_decode_workspace_bytes() requires";
        case FA_ERR_SCRATCH_LIMIT:
            return "sizes need more than FA_DECODE_NOALLOC_SCRATCH_BYTES of scratch; use fa_decode with a workspace";
        default: return "unknown status";
    }
}

extern "C" int fa_device_status(void *stream) {
    int dev;
    DeviceState *st;
    int rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    int word = 0, zero = 0;
    if (cudaMemcpy(&word, st->status_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (word != 0 && cudaMemcpy(st->status_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return FA_ERR_CUDA;
    if (word == 0) return FA_OK;
    return -(word & 0xFFFF);
}

namespace fa {
namespace {
// One warp waits on a barrier that nothing arrives on; the wait is bounded
// and records FA_ERR_TIMEOUT when it runs out.
__global__ void selftest_timeout_kernel(int *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, 99, limit_ns);
    __syncthreads();
}
}  // namespace

cudaError_t launch_selftest_timeout(int *status, int limit_us, cudaStream_t s) {
    selftest_timeout_kernel<<<1, 32, 0, s>>>(status, (unsigned long long)limit_us * 1000ull);
    return cudaGetLastError();
}
}  // namespace fa

extern "C" int fa_selftest_timeout(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 2000000) return FA_ERR_SHAPE;
    int dev;
    DeviceState *st;
    int rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    cudaError_t e = launch_selftest_timeout(st->status_word, limit_us, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

namespace fa {
namespace {
__global__ void selftest_exp2_kernel(const float *x, float *y, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = ex2_fma(x[i]);
}
}  // namespace
}  // namespace fa

extern "C" int fa_selftest_exp2(const float *x, float *y, int n, void *stream) {
    if (n < 1) return FA_ERR_SHAPE;
    int rc = check_ptrs({x, y});
    if (rc != FA_OK) return rc;
    int dev;
    DeviceState *st;
    rc = device_state(&dev, &st);
    if (rc != FA_OK) return rc;
    selftest_exp2_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, y, n);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" int fa_version(void) { return 100; }
