/*
 * parallax.h -- C ABI of libparallax.so, the B300 (sm_103a) implementation of
 * the Parallax attention layer (parameterized Local Linear Attention).
 *
 * Operation.  "Parallax: Parameterized Local Linear Attention for Language
 * Modeling" (gist.science technical summary, "Core mechanism") defines the
 * layer output as softmax attention plus a correction: the softmax-weighted
 * KV covariance applied to a per-query probe, with the boundary-amplification
 * factor set to zero.  This library computes, per batch b and head h, over
 * causal keys i <= t, with c = 1/sqrt(d):
 *
 *     s_ti = c q_t.k_i,   lse_t = log sum_i exp(s_ti),   p_ti = exp(s_ti - lse_t)
 *     mu_k = sum_i p_ti k_i,   u_t = P_h (q_t - mu_k),   g_ti = k_i.u_t,
 *     gbar_t = sum_i p_ti g_ti,
 *     o_t = sum_i p_ti (1 + g_ti - gbar_t) v_i
 *         = o^SA_t + Sigma_KV u_t,   Sigma_KV = sum_i p_ti (v_i - mu_v)(k_i - mu_k)^T
 *
 * A zero projector P gives softmax attention exactly (same page,
 * "Significance and claims").
 *
 * Conventions shared by every entry point.
 *  - Pointers marked "device" must point to device memory of the current CUDA
 *    device; the caller allocates and owns every buffer.  The library keeps no
 *    per-call state (it caches one 16-byte status word per device).
 *  - q, k, v, out, dout, dq, dk, dv: contiguous row-major [B][H][T][d] in
 *    `dtype` (PLX_FP32: float, PLX_BF16: bfloat16 bit pattern).  Base pointers
 *    must be 16-byte aligned.
 *  - P, dP: [H][d][d] float32, row-major, u = P . delta  (u[a] = sum_b P[a][b] delta[b]).
 *  - lse: [B][H][T] float32, natural log, scale c included.
 *  - mu_k: [B][H][T][d] float32.
 *  - stream: a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on it; the return code covers argument checks and launch
 *    errors only.  A device-side watchdog (bounded waits inside kernels) is
 *    read back by parallax_last_device_error().
 *  - Supported: d in {64, 128}; T >= 1; B, H >= 1; B*H*T*d < 2^31 (else
 *    PLX_ERR_INVALID_ARG); B*H <= 65535 (else PLX_ERR_UNSUPPORTED: the
 *    kernels index heads by a grid dimension of that size).
 *  - Input range of the bf16 tensor-core kernels: every matrix-multiply
 *    operand is float16 with float32 accumulation.  A bf16 input converts to
 *    f16 exactly when its magnitude lies in [2^-14, 65504] (or is zero);
 *    smaller magnitudes keep an absolute error below 2^-25, and larger ones
 *    SATURATE to +-65504 without any status.  Inputs q, k, v, dout (and rho)
 *    must therefore stay below 65504 in magnitude on that path; the fp32
 *    path (PLX_FP32, or PLX_PATH_SIMT) has no such limit.  The probe u and
 *    the weights p (1 + g - gbar) are rounded to f16 as well (relative
 *    2^-11), so the correction is accurate to about 2^-11 |g|: where
 *    g = k . u reaches 1e3 or more, the output depends on P beyond that
 *    precision, and the fp32 path is the one to use.
 *  - The library never aborts, never prints and never throws across the ABI.
 */
#ifndef PARALLAX_H
#define PARALLAX_H

#include <stddef.h>

#if defined(__GNUC__)
#define PLX_API __attribute__((visibility("default")))
#else
#define PLX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    PLX_OK = 0,
    PLX_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, misaligned base, size overflow */
    PLX_ERR_UNSUPPORTED = 2, /* d not in {64,128}, unknown dtype, device not sm_103 */
    PLX_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    PLX_ERR_TIMEOUT = 4,     /* a device-side bounded wait gave up (see parallax_last_device_error) */
    PLX_ERR_TOO_LARGE = 5    /* problem needs more scratch than parallax_fwd_noalloc's fixed array */
};

/* Element types of q, k, v, out, dout, dq, dk, dv. */
enum { PLX_FP32 = 0, PLX_BF16 = 1 };

/* Kernel families (parallax_set_path). */
enum {
    PLX_PATH_AUTO = 0,  /* bf16 -> tensor-core (tcgen05) kernels where built, fp32 -> SIMT */
    PLX_PATH_SIMT = 1,  /* fp32 FFMA kernels for every dtype (bf16 inputs widened on load) */
    PLX_PATH_TC = 2     /* tensor-core kernels; PLX_ERR_UNSUPPORTED for fp32 */
};

/*
 * Forward.  Writes out [B,H,T,d] (dtype), lse [B,H,T] and mu_k [B,H,T,d]
 * (float32).  Internally allocates its workspace (the probe u and gbar,
 * parallax_fwd_workspace_bytes() bytes) stream-ordered with cudaMallocAsync and
 * frees it before returning; use parallax_fwd_ws() to supply it instead.
 * Inputs q, k, v (device, dtype), P (device, float32) are read only.
 * Returns PLX_OK or an error code; on error nothing has been launched.
 */
PLX_API int parallax_fwd(const void* q, const void* k, const void* v, const float* P,
                 void* out, float* lse, float* mu_k,
                 int B, int H, int T, int d, int dtype, void* stream);

/* Bytes of device workspace the forward needs for these sizes (0 on bad args). */
PLX_API size_t parallax_fwd_workspace_bytes(int B, int H, int T, int d, int dtype);

/* Forward with a caller-supplied device workspace of at least
 * parallax_fwd_workspace_bytes() bytes, 256-byte aligned.  No allocation. */
PLX_API int parallax_fwd_ws(const void* q, const void* k, const void* v, const float* P,
                    void* out, float* lse, float* mu_k, void* workspace,
                    int B, int H, int T, int d, int dtype, void* stream);

/*
 * Forward that allocates nothing.  The paper has no counterpart: this entry
 * point exists for callers that cannot call cudaMalloc.  Examples are a host
 * whose device memory is owned by another allocator (a framework's caching
 * allocator, or a fixed-budget arena), a latency-critical loop where an
 * allocation would synchronise the device, and a plugin that may not allocate
 * after start-up.
 * Same arguments, layouts and results as parallax_fwd.  It computes with the
 * SIMT (fp32 FFMA) forward kernels for both dtypes, whatever
 * parallax_set_path() selects.
 * Its workspace is one static 32 MiB device array inside the library, which
 * every GPU that loads the library holds until the process exits.  Problems
 * whose workspace (B*H*T*d*4 + B*H*T*4 bytes, each rounded up to 256) exceeds
 * 32 MiB return PLX_ERR_TOO_LARGE; nothing is launched.
 * The first call on each device does a one-time set-up: it looks up the
 * array's device address with that device current.  Make that first call
 * before any stream capture.
 * Every call shares the one array.  Calls whose work overlaps on the GPU
 * (several streams, or several host threads on one device) race on it, so
 * the caller must serialise them.  Calls no cudaMalloc, cudaFree or other
 * allocating routine.
 */
PLX_API int parallax_fwd_noalloc(const void* q, const void* k, const void* v, const float* P,
                         void* out, float* lse, float* mu_k,
                         int B, int H, int T, int d, int dtype, void* stream);

/* Bytes of device workspace parallax_bwd needs for these sizes (0 on bad args). */
PLX_API size_t parallax_bwd_workspace_bytes(int B, int H, int T, int d, int dtype);

/*
 * Backward of sum(dout * out) with respect to q, k, v and P.
 * Reads q, k, v, P, lse, mu_k (as written by parallax_fwd on the same inputs)
 * and dout.  The forward output itself is not needed: the row term
 * dout . out is rebuilt from the backward's own fp32 sums, so the rounding of
 * a bf16-stored out does not leak into the gradients.  Writes dq, dk, dv ([B,H,T,d], dtype) and dP ([H,d,d]
 * float32, overwritten, not accumulated; the reduction over b and t runs in a
 * fixed order, so dP is bitwise reproducible).
 * workspace: device, >= parallax_bwd_workspace_bytes(), 256-byte aligned, or
 * NULL to have the library allocate it stream-ordered (cudaMallocAsync) and
 * free it before returning.
 */
PLX_API int parallax_bwd(const void* q, const void* k, const void* v, const float* P,
                 const float* lse, const float* mu_k, const void* dout,
                 void* dq, void* dk, void* dv, float* dP, void* workspace,
                 int B, int H, int T, int d, int dtype, void* stream);

/*
 * Forward and backward of one training step in one call: parallax_fwd's
 * outputs (out, lse, mu_k) and parallax_bwd's (dq, dk, dv, dP), with the
 * same arguments, layouts and errors as those two.  One workspace serves
 * both, so the backward reuses the f16 operand copies of q, k and v that the
 * forward's pass 1 writes (it converts dO only).  Equal, bit for bit, to
 * parallax_fwd followed by parallax_bwd.
 *   workspace: device, >= parallax_fwd_bwd_workspace_bytes(), 256-byte
 *              aligned, or NULL to allocate it stream-ordered.
 */
PLX_API int parallax_fwd_bwd(const void* q, const void* k, const void* v, const float* P, const void* dout,
                     void* out, float* lse, float* mu_k, void* dq, void* dk, void* dv, float* dP,
                     void* workspace, int B, int H, int T, int d, int dtype, void* stream);

/* Bytes of device workspace parallax_fwd_bwd needs (0 on bad args). */
PLX_API size_t parallax_fwd_bwd_workspace_bytes(int B, int H, int T, int d, int dtype);

/*
 * One-pass forward with a given probe: the layer in the form the paper states
 * it ("Parallax: Parameterized Local Linear Attention for Language Modeling",
 * technical summary, "Core mechanism"), with the probe rho supplied by the
 * caller (in the paper it comes from a learned projection of the layer
 * input) instead of formed from mu_k:
 *     o_t = o^SA_t - Sigma_KV,t rho_t,
 *     Sigma_KV,t = sum_i p_ti (v_i - mu_v,t)(k_i - mu_k,t)^T.
 * With rho_t = -P_h (q_t - mu_k,t) it is parallax_fwd's layer.
 *   q, k, v, rho: device, [B][H][T][d] bf16 (PLX_BF16 only; PLX_FP32 returns
 *                 PLX_ERR_UNSUPPORTED).  out: device, [B][H][T][d] bf16.
 *   lse: device, [B][H][T] float32.
 *   workspace: device, >= parallax_fwd_probe_workspace_bytes(), 256-byte
 *              aligned, or NULL to allocate it stream-ordered.
 * One pass over the keys on the tensor cores: S = Q K^T and R = rho K^T on
 * the same K tile, online softmax, two value accumulations.
 */
PLX_API int parallax_fwd_probe(const void* q, const void* k, const void* v, const void* rho,
                       void* out, float* lse, void* workspace,
                       int B, int H, int T, int d, int dtype, void* stream);

/* Bytes of device workspace parallax_fwd_probe needs (0 on bad or unsupported args). */
PLX_API size_t parallax_fwd_probe_workspace_bytes(int B, int H, int T, int d, int dtype);

/*
 * Decode step: one new query per (sequence, head) against a KV cache.
 * The paper's own kernel is a decode kernel ("Parallax: Parameterized Local
 * Linear Attention for Language Modeling", technical summary,
 * "Hardware-aware algorithm"); the layer is the same as parallax_fwd's: the
 * query of sequence b sits at position lens[b] - 1 and attends to keys
 * 0 .. lens[b] - 1, so out[b,h] equals row lens[b] - 1 of parallax_fwd run
 * on the cache with that query in that row.
 *   q:        device, [B][H][d] in dtype, the new queries.
 *   k_cache,
 *   v_cache:  device, [B][H][Lmax][d] in dtype; rows past lens[b] are ignored.
 *   lens:     device, [B] int32, valid keys per sequence (the new token's own
 *             key and value included); values outside [1, Lmax] are clamped
 *             to it.  NULL means every sequence has Lmax keys.
 *   P:        device, [H][d][d] float32.
 *   out:      device, [B][H][d] in dtype.   lse: device, [B][H] float32.
 *   workspace: device, >= parallax_decode_workspace_bytes(), 256-byte
 *             aligned, or NULL to allocate it stream-ordered and free it
 *             before returning.
 * Memory-bound split-KV kernels (fp32 arithmetic for both dtypes): keys are
 * read twice (the softmax statistics, then the weights) and values once.
 * Returns PLX_OK or an error code; on error nothing has been launched.
 */
PLX_API int parallax_decode(const void* q, const void* k_cache, const void* v_cache, const int* lens,
                    const float* P, void* out, float* lse, void* workspace,
                    int B, int H, int Lmax, int d, int dtype, void* stream);

/* Bytes of device workspace parallax_decode needs (0 on bad args). */
PLX_API size_t parallax_decode_workspace_bytes(int B, int H, int Lmax, int d, int dtype);

/*
 * Decode step with a given probe: one new query per (sequence, head) against
 * a KV cache, in the form the paper states the layer ("Parallax:
 * Parameterized Local Linear Attention for Language Modeling", technical
 * summary, "Core mechanism"): o = o^SA - Sigma_KV rho, with the probe rho
 * supplied by the caller.  With r_i = k_i . rho every term is a softmax-
 * weighted sum over the keys,
 *     o = mu_v - sum_i p_i r_i v_i + (sum_i p_i r_i) mu_v,
 * so the keys and values are read once, in one pass, as the paper's own
 * decode kernel runs both branches over one KV stream ("Hardware-aware
 * algorithm").  Row len-1 of parallax_fwd_probe with that row's probe; with
 * rho = -P_h (q - mu_k) it is parallax_decode.
 *   q, rho: device, [B][H][d] bf16 (PLX_BF16 only; PLX_FP32 returns
 *           PLX_ERR_UNSUPPORTED).
 *   k_cache, v_cache: device, [B][H][Lmax][d] bf16.
 *   lens: device int32 [B] (1 <= lens[b] <= Lmax; values outside are
 *         clamped), or NULL for Lmax.  Cache rows at or past lens[b] are
 *         ignored, whatever they hold.
 *   out: device, [B][H][d] bf16.  lse: device, [B][H] float32.
 *   workspace: device, >= parallax_decode_probe_workspace_bytes(), 256-byte
 *              aligned, or NULL to allocate it stream-ordered.
 * Returns PLX_OK, PLX_ERR_INVALID_ARG (null or misaligned pointer, bad
 * sizes), PLX_ERR_UNSUPPORTED or PLX_ERR_CUDA; asynchronous on `stream`.
 */
PLX_API int parallax_decode_probe(const void* q, const void* k_cache, const void* v_cache, const int* lens,
                          const void* rho, void* out, float* lse, void* workspace,
                          int B, int H, int Lmax, int d, int dtype, void* stream);

/* Bytes of device workspace parallax_decode_probe needs (0 on bad or unsupported args). */
PLX_API size_t parallax_decode_probe_workspace_bytes(int B, int H, int Lmax, int d, int dtype);

/*
 * Forward and backward of the layer from HOST buffers, with the copies
 * overlapped with the compute.  The paper has no counterpart: this entry
 * serves callers whose tensors live in host memory.  The heads are split into
 * `chunks` groups (0 = min(H, 8)).  Every group's inputs are copied in on an
 * internal stream, the group's parallax_fwd + parallax_bwd runs on `stream`
 * as soon as its inputs have arrived, and its results are copied out on a
 * second internal stream while later groups compute.  dP_h sums over the
 * batch only, so each group's dP rows are complete within the group, and
 * every group runs exactly the arithmetic of parallax_fwd + parallax_bwd on
 * device copies (dq, whose fp32 accumulation order varies between runs,
 * agrees to its last bit of rounding).
 *   q, k, v, dout: host, [B][H][T][d] in dtype.   P: host, [H][d][d] float32.
 *   out, dq, dk, dv: host, [B][H][T][d] in dtype.   dP: host, [H][d][d] float32.
 *   lse: host, [B][H][T] float32, or NULL (not returned).
 *   mu_k: host, [B][H][T][d] float32, or NULL (not returned).
 * Every pointer must be host memory (PLX_ERR_INVALID_ARG otherwise); use
 * pinned memory (cudaHostAlloc / cudaHostRegister): copies from or to
 * pageable memory are correct but do not overlap.  Device memory (the
 * tensors of all groups plus one workspace for the largest group) is taken
 * stream-ordered on `stream` and freed before returning.  The call is
 * asynchronous: the outputs are complete once `stream` has reached the
 * point where the call was made.  Returns PLX_OK or an error code.
 */
PLX_API int parallax_step_host(const void* q, const void* k, const void* v, const float* P, const void* dout,
                       void* out, float* lse, float* mu_k, void* dq, void* dk, void* dv, float* dP,
                       int chunks, int B, int H, int T, int d, int dtype, void* stream);

/*
 * Synchronizes `stream`, then reads and clears the current device's watchdog
 * word.  Returns PLX_OK, PLX_ERR_TIMEOUT (a bounded wait inside a kernel gave
 * up; the kernel skipped its remaining work and released its resources) or
 * PLX_ERR_CUDA (the synchronize itself failed).  If `detail` is not NULL it
 * receives the raw word (kernel id << 16 | wait site) of the first timeout.
 */
PLX_API int parallax_last_device_error(void* stream, unsigned* detail);

/*
 * Failure-detection hook.  Sets how long a bounded wait inside the
 * tensor-core kernels of the current device may take, in SM clock cycles,
 * before it gives up; cycles <= 0 restores the default (4e9 cycles, about
 * two seconds).  A wait that gives up records (kernel id << 16 | wait site)
 * in the device's status word and raises its CTA's abort flag; every role of
 * the CTA then leaves its loop, waits (with the long bound) for the copies
 * and MMAs it has in flight, releases its TMEM and returns, so the context
 * stays usable and parallax_last_device_error() reports PLX_ERR_TIMEOUT.
 * A short limit makes waits that would have completed time out: it exists
 * to exercise that path in tests, and the outputs of calls made under it
 * are unspecified.  Synchronises the device; applies to kernels launched
 * after it returns.  The setting is kept until changed (reading the status
 * with parallax_last_device_error() does not reset it).
 * Returns PLX_OK, PLX_ERR_UNSUPPORTED (not an sm_103 device) or PLX_ERR_CUDA.
 */
PLX_API int parallax_set_wait_limit(long long cycles);

/* Selects the kernel family for later calls in this process; returns the
 * previous setting, or -1 if `path` is not a PLX_PATH_* value. */
PLX_API int parallax_set_path(int path);

/* Caps the number of CTAs the persistent kernels launch for later calls in
 * this process: pass 2 of the tensor-core forward at d = 128 (one CTA per SM
 * by default) and B2 of the tensor-core backward at d = 64 (two per SM).  0
 * restores the default.  Each CTA of those kernels takes work items from a
 * counter until none are left, so a small cap makes every CTA run many items
 * of mixed lengths: a test hook for their item changes on small problems.
 * Results do not depend on the cap (the items' arithmetic is the same; only
 * which CTA runs an item changes).  Returns the previous cap, or -1 if
 * `ctas` is negative. */
PLX_API int parallax_set_persistent_ctas(int ctas);

/*
 * Launch accounting and per-kernel device timing (tracing).
 * Every kernel launch the library makes is counted.  While timing is enabled,
 * a CUDA event is recorded on the launching stream before and after each
 * launch; parallax_timing_collect() waits for the recorded events and folds
 * their elapsed times into per-kernel totals, which parallax_timing_get()
 * returns by index (name is a static string owned by the library).  Timing
 * assumes one device per process.  Not thread-safe against concurrent calls.
 */
PLX_API unsigned long long parallax_launch_count(void);
PLX_API int parallax_timing_enable(int on);          /* returns the previous setting */
PLX_API int parallax_timing_collect(void);           /* number of kernel names, or -PLX_ERR_CUDA */
PLX_API int parallax_timing_get(int i, const char** name, double* total_ms, long long* launches);
PLX_API void parallax_timing_reset(void);

/* Static description of a status code (never NULL). */
PLX_API const char* parallax_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* PARALLAX_H */
