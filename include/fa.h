/*
 * fa.h -- C ABI of libfa: exact scaled-dot-product attention on one GB300
 * (sm_103a), computed tile by tile (FlashAttention style), with the
 * atomic-free split backward.
 *
 * Operation (all entry points):
 *   Per (batch b, head h) slice, Q, K, V, O, dO are N x D matrices and
 *     S = scale * Q K^T,  P = softmax_row(S)  (causal: key j visible to query
 *     row i iff j <= i),  O = P V,  LSE_i = ln sum_j exp(S_ij).
 *   Definition and streaming form: "Learning Metal with FlashAttention",
 *   section "FlashAttention" (per-row softmax over all keys; running max,
 *   running sum and unnormalised output updated per K/V tile; O divided by
 *   the sum after the last tile).  Causal tiles skipped rather than masked,
 *   base-2 exponent: "Flash Attention" (metalworking), kernel anatomy items
 *   3-4.  LSE = m + ln(l) and the split backward (one dQ kernel, one dK/dV
 *   kernel, 7 GEMMs, no atomics): "FlashAttention (Metal port)"
 *   (metal-flash-attention), documentation section and the forward /
 *   backward pseudocode of its performance section.
 *
 * Memory layout and ownership (all entry points):
 *   - q, k, v, o, dO, dq, dk, dv: [B, H, N, D] contiguous, row-major, in
 *     DEVICE memory allocated by the caller, 16-byte aligned.
 *   - lse, delta: [B, H, N] contiguous float32 in device memory.
 *   - The library never allocates, frees or retains caller memory; outputs
 *     are fully overwritten (rows 0..N-1 of every head).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  No entry point
 *     synchronises the host except fa_device_status().
 *   - The library's own state is static device storage: the status word
 *     below, the decode scratch of fa_decode_noalloc, and a ring of 1024
 *     work counters that the D <= 64 causal forward draws its blocks from
 *     when its keys and values exceed three quarters of L2 (each call takes
 *     the next counter, and the launch zeroes it again when it ends).
 *     Calls in flight at the same time on different streams therefore use
 *     different counters; a captured CUDA graph keeps the counter it was
 *     given, so one graph must not be replayed on two streams at once.
 *
 * Errors: every entry point returns FA_OK (0) or a negative fa_status.
 * Arguments are validated before anything is launched; on a validation
 * error nothing is enqueued and no output is touched.  A launch failure
 * reported by the CUDA runtime is returned as FA_ERR_CUDA.  Kernels never
 * trap: every wait inside a kernel is bounded, and a wait that runs out
 * records FA_ERR_TIMEOUT in a device status word which fa_device_status()
 * reads (outputs of that launch are then undefined).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of q/k/v/o/dO (dtype) and of dq/dk/dv (grad_dtype). */
enum fa_dtype {
    FA_F32 = 0,   /* IEEE float32                                      */
    FA_BF16 = 1   /* bfloat16, round-to-nearest-even on every store    */
};

enum fa_status {
    FA_OK = 0,
    FA_ERR_NULL = -1,        /* a required pointer is NULL                              */
    FA_ERR_SHAPE = -2,       /* B, H or N < 1, or B*H*N*D overflows the index range      */
    FA_ERR_HEAD_DIM = -3,    /* D not supported for this dtype / pass (see below)        */
    FA_ERR_DTYPE = -4,       /* unknown dtype / grad_dtype, or an unsupported pairing   */
    FA_ERR_ALIGN = -5,       /* a pointer is not 16-byte aligned                         */
    FA_ERR_SCALE = -6,       /* scale is not finite                                      */
    FA_ERR_CUDA = -7,        /* the CUDA runtime reported an error (launch, attributes)  */
    FA_ERR_TIMEOUT = -8,     /* a bounded in-kernel wait ran out (read by fa_device_status) */
    FA_ERR_DEVICE_PTR = -9,  /* a pointer is not device-accessible memory                */
    FA_ERR_DEVICE = -10,     /* the current device is not sm_103 (GB300)                 */
    FA_ERR_WORKSPACE = -11,  /* a workspace is smaller than its size query requires      */
    FA_ERR_SCRATCH_LIMIT = -12 /* the sizes need more than FA_DECODE_NOALLOC_SCRATCH_BYTES */
};

/*
 * fa_forward -- O = softmax(scale Q K^T) V and LSE (natural log-sum-exp of the
 * scaled scores of each row).
 *   Defined by: "Learning Metal with FlashAttention", section "FlashAttention"
 *   (the attention definition and its streaming form: running max m, running
 *   sum l, O rescaled per K/V tile and divided by l after the last one); the
 *   forward pseudocode of "FlashAttention (Metal port)" (metal-flash-
 *   attention), performance section (L = m + log l written out); tiles above
 *   the causal diagonal skipped, exponent in base 2: "Flash Attention"
 *   (metalworking), kernel anatomy items 1-4.
 *   dtype FA_BF16: D a multiple of 8 in [8, 256]; bf16 inputs, fp32
 *                  accumulation (tcgen05 tensor cores), bf16 O, fp32 LSE.
 *                  Kernels exist for D = 64, 128, 192, 256; any other D runs
 *                  on the next wider one with the extra columns read as
 *                  zeros (the rows keep the caller's stride D).
 *   dtype FA_F32 : D a multiple of 4 in [4, 256]; fp32 inputs and O,
 *                  fp32 FFMA arithmetic throughout, fp32 LSE.
 *   N >= 1 arbitrary (ragged tails are masked).  causal: 0 or non-zero.
 */
FA_API int fa_forward(const void *q, const void *k, const void *v, void *o, float *lse,
               int B, int H, int N, int D, float scale, int causal, int dtype,
               void *stream);

/*
 * fa_backward_dq -- first half of the split backward ("backward query"):
 *   Defined by: "FlashAttention (Metal port)" (metal-flash-attention), the
 *   backward-query pseudocode of its performance section (D = dO * O read as
 *   the row sum; P = exp(S - L) with S the scaled scores), and its
 *   documentation section (dQ and dK/dV as two kernels, 7 GEMMs, no atomics).
 *   delta_i = sum_d dO_id O_id            (written: delta [B,H,N] fp32)
 *   P = exp(S - LSE), dP = dO V^T, dS = P * (dP - delta) * scale,
 *   dQ = dS K                              (written: dq, grad_dtype)
 * o and lse are the outputs of fa_forward on the same q, k, v, scale, causal.
 * Supported: dtype FA_BF16 with D a multiple of 8 in [8, 256] (as for
 * fa_forward); grad_dtype FA_F32 or FA_BF16.
 */
FA_API int fa_backward_dq(const void *q, const void *k, const void *v, const void *o,
                   const void *dO, const float *lse, float *delta, void *dq,
                   int B, int H, int N, int D, float scale, int causal, int dtype,
                   int grad_dtype, void *stream);

/*
 * fa_backward_dkdv -- second half ("backward key-value"), one CTA per K/V
 * tile iterating over query tiles:
 *   Defined by: "FlashAttention (Metal port)" (metal-flash-attention), the
 *   backward-key-value pseudocode of its performance section (delta and L of
 *   every query row read; dS^T carries the softmax scale).
 *   P^T = exp(S^T - LSE), dV = P^T dO, dP^T = V dO^T,
 *   dS^T = P^T * (dP^T - delta) * scale, dK = dS^T Q
 * lse from fa_forward, delta from fa_backward_dq (enqueue this call after it
 * on the same stream, or order the two streams yourself).
 * Supported: dtype FA_BF16 with D a multiple of 8 in [8, 256] (as for
 * fa_forward); grad_dtype FA_F32 or FA_BF16.
 */
FA_API int fa_backward_dkdv(const void *q, const void *k, const void *v, const void *dO,
                     const float *lse, const float *delta, void *dk, void *dv,
                     int B, int H, int N, int D, float scale, int causal, int dtype,
                     int grad_dtype, void *stream);

/*
 * fa_backward_atomic -- the conventional 5-GEMM backward, as a comparator for
 * the split backward above.  "FlashAttention (Metal port)" (metal-flash-
 * attention), documentation section: the split into a dQ kernel and a dK/dV
 * kernel (7 GEMMs, no atomics) is chosen there because Apple GPUs lack fp32
 * atomics; this entry point runs the design that choice replaces.  One pass
 * over key tiles recomputes S^T and dP^T once per (key tile, query tile),
 * writes dK and dV, and accumulates dQ = dS K across key tiles in fp32 (one
 * L2 bulk reduce-add per 64-query tile), then converts it:
 *   delta = rowsum(dO * O)   (written, as fa_backward_dq writes it)
 *   dq, dk, dv               (grad_dtype, same results as the split backward)
 * dq_accum: device workspace owned by the caller, at least B*H*N*D*4 bytes,
 * 16-byte aligned; zeroed and overwritten by the call (FA_ERR_WORKSPACE when
 * smaller).  Supported: dtype FA_BF16, D = 128; grad_dtype FA_F32 or FA_BF16.
 * Enqueues a memset and three kernels on `stream`.
 */
FA_API int fa_backward_atomic(const void *q, const void *k, const void *v, const void *o, const void *dO,
                              const float *lse, float *delta, void *dq, void *dk, void *dv,
                              float *dq_accum, size_t dq_accum_bytes,
                              int B, int H, int N, int D, float scale, int causal, int dtype,
                              int grad_dtype, void *stream);

/*
 * fa_decode -- attention of a few query rows against a long key/value range
 * (decode).  "Flash Attention" (metalworking), section on the technique's
 * boundaries: one query row cannot fill a matrix-engine tile, so decode gets a
 * separate vector kernel; the mathematics is the forward's:
 *   O = softmax(scale q K^T) V per query row, LSE = natural log-sum-exp.
 *   q: [B, H, n_q, D]; k, v: [B, H, N, D]; o: [B, H, n_q, D]; all bf16.
 *   lse: [B, H, n_q] fp32.  1 <= n_q <= N; n_q <= 16;
 *   D in {64, 128, 256}.  The query rows are the LAST n_q positions: with
 *   causal != 0, row i sees keys j <= N - n_q + i; otherwise all N keys.
 *   workspace: device memory owned by the caller, at least
 *   fa_decode_workspace_bytes(...) bytes, 16-byte aligned; it holds the
 *   partial results of the key chunks the work is split into (no clearing
 *   needed; its contents are undefined afterwards).  Two calls that run
 *   concurrently must not share a workspace.
 * Errors as for fa_forward, plus FA_ERR_WORKSPACE when workspace_bytes is too
 * small.  Launches two kernels on `stream`.
 */
FA_API int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int n_q, int N, int D, float scale, int causal,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace fa_decode needs for these sizes (written to *bytes).  The
 * key range is split for the current device's SM count, so the answer is for
 * the device that is current at this call (the GB300's 152 SMs if no device
 * can be queried); call fa_decode on that same device. */
FA_API int fa_decode_workspace_bytes(int B, int H, int n_q, int N, int D, size_t *bytes);

/* Size of the fixed per-device scratch that fa_decode_noalloc works in. */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * fa_decode_noalloc -- fa_decode without a workspace argument.  The attention
 * pages have no counterpart of this entry point: it is a library convenience.
 *
 * Who it is for: callers that cannot allocate device memory, or cannot keep a
 * workspace alive, at the point where they decode -- a plain C host with no
 * device allocator of its own, or a latency-critical loop where a cudaMalloc
 * (which may synchronise the device) or an allocation that fails under a fully
 * committed memory budget is not acceptable.  This call allocates nothing:
 * the key-chunk partials go to a fixed scratch array that the library holds in
 * static device storage, FA_DECODE_NOALLOC_SCRATCH_BYTES per device.
 *
 * Arguments, layout, results and errors are those of fa_decode, minus the
 * workspace; in addition:
 *   - sizes whose fa_decode_workspace_bytes() exceeds
 *     FA_DECODE_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_SCRATCH_LIMIT
 *     before anything is launched (use fa_decode with your own workspace);
 *   - nothing in the scratch needs to start at zero: every entry a call reads
 *     is written by that same call first;
 *   - the first call on each device sets up that device's scratch address
 *     (one cudaGetSymbolAddress with the device current); make that first
 *     call before beginning any stream capture on the device;
 *   - all calls on one device share the one scratch array, so calls that can
 *     overlap in time (different streams without ordering between them, or
 *     different host threads) race on it and give undefined results.  Calls
 *     enqueued on one stream run one after another and are safe.
 */
FA_API int fa_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int n_q, int N, int D, float scale, int causal,
                             void *stream);

/* Static description of a status code (never NULL). */
FA_API const char *fa_status_string(int status);

/*
 * fa_device_status -- synchronises `stream`, then returns and clears the
 * device status word of the current device: FA_OK, or FA_ERR_TIMEOUT if a
 * bounded in-kernel wait ran out since the last call.  Returns FA_ERR_CUDA
 * if the synchronisation itself failed.
 */
FA_API int fa_device_status(void *stream);

/*
 * fa_selftest_timeout -- test hook for the failure path: launches one
 * 32-thread block that waits on a shared-memory barrier nothing arrives on,
 * with a wait bounded by limit_us microseconds (1..2000000); the kernel
 * records FA_ERR_TIMEOUT and returns.  Returns FA_OK if launched.
 */
FA_API int fa_selftest_timeout(int limit_us, void *stream);

/*
 * fa_selftest_exp2 -- test hook: y[i] = 2^x[i] computed on the FMA pipe the
 * way the forward kernel computes a quarter of its softmax exponentials
 * (range split + degree-3 polynomial, relative error < 1e-4 for x >= -125).
 * x, y: n floats of device memory.  Returns FA_OK if launched.
 */
FA_API int fa_selftest_exp2(const float *x, float *y, int n, void *stream);

/* Library version (major*10000 + minor*100 + patch). */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
