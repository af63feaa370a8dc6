/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library, libkda.so.
 *
 * The operation. Kimi Delta Attention (KDA) is linear attention with a fixed-size state per
 * (sequence, head): "Inside Kimi K3's Architecture" (maidul-haque blog), section "Kimi Delta
 * Attention: the linear core" -- the delta rule subtracts the value a key currently reads
 * before writing the fresh one, and the forget gate decays each channel separately; "Kimi K3
 * Explained" (researchpapers.dev), "Architecture at a glance" and FAQ "What is Kimi Delta
 * Attention?" -- channel-wise forget gate with a log-decay bounded below through a scaled
 * sigmoid, computed chunkwise on dense tensor-core tiles. Per (sequence, head), with the
 * state S (d_k x d_v, fp32) and natural-log decay g_t (one value per key channel):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t                                      (no scale is applied to q)
 *
 * Conventions shared by every entry point:
 *  - Pointers are device pointers to caller-owned memory. The library never allocates,
 *    frees or keeps a pointer after the call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *    Argument errors are found on the host and returned before anything is launched.
 *    A launch failure returns KDA_ERR_CUDA. Conditions only the device can see (a
 *    cu_seqlens array that is not monotonic, a state slot past the pool end, a pipeline wait
 *    that ran out) are recorded in a per-device error word that kda_check_status() returns.
 *  - Layouts are row-major and dense: q, k, g [B, T, H, d_k]; v, o [B, T, H, d_v];
 *    beta [B, T, H]; states [N, H, d_k, d_v] (fp32, row index = key channel).
 *  - Accuracy is stated for g in [-5, 0] (the scaled-sigmoid bound with constant 5): inputs
 *    outside it are computed, but the bf16 tensor-core path may lose accuracy there.
 *  - Not thread-safe per device error word only: concurrent calls are fine, but
 *    kda_check_status() reports (and clears) errors of every call on that device.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kda_stream_t; /* same type as cudaStream_t */

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad cu_seqlens or slot */
    KDA_ERR_UNSUPPORTED = 2, /* well-formed request this build has no kernel for */
    KDA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_TIMEOUT = 4      /* a device-side pipeline wait gave up (kda_check_status) */
} kda_status;

typedef enum {
    KDA_BF16 = 0, /* q, k, v, g, beta and o are bfloat16 */
    KDA_F32 = 1   /* q, k, v, g, beta and o are float32 */
} kda_dtype;

/*
 * Options of kda_prefill_ex and kda_decode_step_ex. Zero the struct, set struct_size to
 * sizeof(kda_options), then set the fields wanted; all zero means the plain kda_prefill /
 * kda_decode_step. The library reads only the first struct_size bytes, so a caller built
 * against an older, shorter kda_options keeps working (later fields take their defaults).
 */
typedef struct kda_options {
    size_t struct_size; /* sizeof(kda_options) as the caller compiled it */
    float gate_bound;   /* 0: g holds log-decays. > 0 (at most 1e4): g holds gate logits x and
                           the kernels form g = -gate_bound * sigmoid(x), as kda_prefill_gated */
    int qk_l2norm;      /* non-zero: every row of q and of k (d_k values of one token and head)
                           is divided by sqrt(sum of its squares + 1e-6) in the kernels. The pages
                           do not describe this step; the workloads feed q and k as unit vectors */
    /* Indexed state pool (serving with a prefill cache: "How Kimi K3 works", benebsworth, "KDA:
     * a fixed memory instead of a growing bill"). With an index array, the matching state pointer
     * is a pool fp32 [state_pool_size, H, dk, dv] and sequence n uses slot idx[n]: a negative slot
     * means a zero initial state / no final-state write; a slot >= state_pool_size is treated the
     * same way and sets KDA_ERR_INVALID_ARG in the error word (kda_check_status). Slots written by
     * a call must not be read or written by any other sequence of that call. */
    const int32_t *initial_state_indices; /* NULL or int32 [N] on the device */
    const int32_t *final_state_indices;   /* NULL or int32 [N] on the device. Decode: NULL means
                                             the slots of initial_state_indices (in place) */
    int state_pool_size;                  /* slots in the pool; > 0 when an index array is given */
    /* Output gate ("Kimi K3 Explained", researchpapers.dev, "Architecture at a glance": the output
     * gate is an input-dependent full-rank projection). NULL, or that projection's output z with
     * the layout and dtype of o ([B,T,H,dv] prefill, [N,H,dv] decode), 16-byte aligned: o is
     * stored as o * sigmoid(z). The pages name no activation; the sigmoid is the plain reading. */
    const void *out_gate;
} kda_options;

/*
 * kda_prefill -- run the recurrence over whole sequences (chunked prefill).
 *
 * dtype        element type of q, k, v, g, beta and o.
 * B, T, H      batch, tokens per batch row, heads. With cu_seqlens == NULL the call covers
 *              B sequences of T tokens each. With cu_seqlens != NULL, B must be 1 and T is
 *              the total packed token count.
 * dk, dv       key and value head sizes. Supported: dk == dv in {32, 64, 128}.
 * q, k, g      [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H]. g is log(alpha) <= 0.
 * cu_seqlens   NULL, or int32 [n_seqs + 1] on the device: sequence n covers packed rows
 *              cu_seqlens[n] .. cu_seqlens[n+1]-1; must start at 0, be non-decreasing and
 *              end at T (checked on the device; a violation skips the bad sequence and sets
 *              KDA_ERR_INVALID_ARG in the error word). Chunks restart at every sequence start.
 * n_seqs       number of sequences when cu_seqlens != NULL (ignored otherwise; N = B).
 * initial_state  fp32 [N, H, dk, dv] or NULL (zero state).
 * o            output [B, T, H, dv], same dtype as the inputs. Every row is written.
 * final_state  fp32 [N, H, dk, dv] or NULL (not written). May alias initial_state.
 * workspace, workspace_bytes  device scratch, 256-byte aligned, of at least
 *              kda_prefill_workspace_size() bytes; or NULL / 0. Packed bf16 sequences (2 to
 *              4096 of them) use 4 bytes per sequence for a longest-first launch order (a sort of
 *              cu_seqlens by length on the device), which shortens the tail of the launch; the
 *              results are the same without it. A split call uses it for more: when
 *              few long sequences cannot fill the GPU (bf16, dk == dv == 128; packed or not), each
 *              is cut into segments run side by side and joined through the segment transitions
 *              (the state after a segment is linear in the state before it: "Inside Kimi K3's
 *              Architecture", "Kimi Delta Attention: the linear core"); for packed sequences the
 *              segments are planned on the device from cu_seqlens. Without a large enough
 *              workspace the same call runs one pass per sequence, with the same result up to
 *              rounding. The caller owns the workspace; it must not be used by other work on
 *              other streams until this call's work is done.
 * Alignment: all pointers 16-byte aligned. Rows of q, k, v, g, o are contiguous.
 * Paths: bf16 runs the chunked tensor-core kernel (bf16 operands, fp32 accumulation; heads of
 * 32 or 64 channels with the missing channels zero). fp32 with dk == dv in {32, 64} runs a
 * chunked tensor-core kernel in tf32 (operands rounded to tf32, fp32 accumulation and state);
 * fp32 with dk == dv == 128, or with the L2 normalisation or the output gate of kda_prefill_ex,
 * runs the token-by-token recurrence on the CUDA cores in fp32.
 * Returns KDA_OK once the work is queued on `stream`.
 */
KDA_API kda_status kda_prefill(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                       const void *q, const void *k, const void *v, const void *g,
                       const void *beta, const int32_t *cu_seqlens, int n_seqs,
                       const float *initial_state, void *o, float *final_state,
                       void *workspace, size_t workspace_bytes, kda_stream_t stream);

/* Bytes of device workspace kda_prefill can use for a call with these arguments, or 0. Pass the
 * same dtype, B, T, H, dk, dv, cu_seqlens and n_seqs as the call: cu_seqlens is only compared with
 * NULL (never read, so the device pointer may be passed). bf16 only; the split needs dk == dv ==
 * 128, the launch order dk == dv in {32, 64, 128}; the sizes follow the current device's SM count (0
 * SMs when no device is visible).
 * Packed sequences (cu_seqlens != NULL, B == 1): when there are fewer sequences than SMs / H and at
 * least 4096 rows, the split along the sequence planned on the device (the packed rows of q~ in bf16,
 * T * H * 256 bytes, plus three 128 x 128 states per segment and head for at most
 * min(8 n_seqs, n_seqs + SMs / H) segments); otherwise the launch order, 4 bytes per sequence
 * rounded up to 256, for 2 <= n_seqs <= 4096 (0 for a single sequence). Unpacked (cu_seqlens ==
 * NULL, n_seqs ignored): the split along the sequence (0 when the call would not split). The same
 * sizes apply to kda_prefill_gated and kda_prefill_ex. */
KDA_API size_t kda_prefill_workspace_size(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                                          const int32_t *cu_seqlens, int n_seqs);

/* kda_prefill_workspace_size for a GPU with sm_count SMs instead of the current device: host
 * arithmetic only (nothing is queued, no device is needed), the same sizes the call computes with
 * the device's own SM count. 0 for negative sizes or a negative sm_count. */
KDA_API size_t kda_prefill_workspace_size_for(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                                              const int32_t *cu_seqlens, int n_seqs, int sm_count);

/*
 * kda_prefill_split_plan -- how kda_prefill splits B sequences of T tokens and H heads along the
 * sequence (bf16, dk == dv == 128, no cu_seqlens, with the workspace) on a GPU with sm_count SMs;
 * host arithmetic only, nothing is queued and no device is needed. The state after a segment is
 * affine in the state before it ("Inside Kimi K3's Architecture", "Kimi Delta Attention: the
 * linear core": the per-token transition does not depend on the state), so segments run side by
 * side and are joined exactly afterwards. Outputs: *segments = P segments per sequence (0: a
 * single pass; P = min(8, sm_count / (B H), T / 2048) when that is at least 2), *segment_rows =
 * rows per segment (a multiple of 64; the last segment may be shorter; 0 when not split),
 * *workspace_bytes = what kda_prefill_workspace_size returns on such a GPU. Returns
 * KDA_ERR_INVALID_ARG for negative sizes or a NULL output pointer.
 */
KDA_API kda_status kda_prefill_split_plan(int B, int T, int H, int sm_count, int *segments, int *segment_rows,
                                          size_t *workspace_bytes);

/*
 * kda_prefill_ex / kda_decode_step_ex -- kda_prefill / kda_decode_step with options (see
 * kda_options; NULL = none). Returns KDA_ERR_INVALID_ARG for a struct_size below sizeof(size_t)
 * or above 4096, or a gate_bound that is negative, not finite or above 1e4; every other
 * argument and return value as the plain forms.
 */
KDA_API kda_status kda_prefill_ex(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                                  const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const int32_t *cu_seqlens, int n_seqs,
                                  const float *initial_state, void *o, float *final_state,
                                  const kda_options *options, void *workspace, size_t workspace_bytes,
                                  kda_stream_t stream);

KDA_API kda_status kda_decode_step_ex(kda_dtype dtype, int N, int H, int dk, int dv,
                                      const void *q, const void *k, const void *v, const void *g,
                                      const void *beta, float *state, void *o,
                                      const kda_options *options, kda_stream_t stream);

/*
 * kda_backward -- gradients of L = sum(d_o * o) + sum(d_final_state * final_state) through
 * kda_prefill's computation (plain log-decays; no options), with an fp32 state. The pages
 * train the model ("Kimi K3 Explained", researchpapers.dev, "Architecture at a glance") but give
 * no gradient method: this is reverse-mode differentiation of the recurrence (for d = 128 taken
 * of its chunkwise form on 16-token chunks; the result is the same up to rounding).
 * Precision for d = 128: the products run on the tensor cores in tf32. For fp32 inputs every
 * product is taken to fp32 accuracy (split operands, three tf32 products); for bf16 inputs the
 * products with the 128 x 128 states are single tf32 products, and the gradients agree with an
 * exact computation to about 3e-4 relative (Frobenius norm) instead of about 2e-6. d = 32, 64
 * compute on the CUDA cores in fp32.
 *
 * dtype, B, T, H, dk, dv, q, k, v, g, beta, cu_seqlens, n_seqs, initial_state: as kda_prefill.
 * d_o          [B, T, H, dv] in `dtype`: dL/do.
 * d_final_state  fp32 [N, H, dk, dv] or NULL (zero): dL/dS_final.
 * dq, dk, dg   fp32 [B, T, H, dk]; dv fp32 [B, T, H, dv]; dbeta fp32 [B, T, H]: written in full
 *              (dg is with respect to the log-decay g).
 * d_initial_state  fp32 [N, H, dk, dv] or NULL (not written): dL/dS_initial (also without an
 *              initial state: the gradient at the zero state).
 * workspace    device scratch of at least kda_backward_workspace_size() bytes, 16-byte aligned,
 *              owned by the caller: the state at every chunk start (every 16 tokens for d = 128,
 *              every 64 for d = 32, 64), d * d * 4 bytes per head and chunk.
 * Supported: dk == dv in {32, 64, 128}; bf16 or fp32 inputs. Alignment as kda_prefill for the
 * inputs (d_o as o); dq, dk, dv, dg and the state pointers 16-byte aligned, dbeta 4-byte aligned.
 * Errors: KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED for malformed arguments, found on the host
 * before anything is queued (also a workspace that is missing, short or misaligned).
 */
KDA_API kda_status kda_backward(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                                const void *q, const void *k, const void *v, const void *g,
                                const void *beta, const int32_t *cu_seqlens, int n_seqs,
                                const float *initial_state, const void *d_o, const float *d_final_state,
                                float *dq, float *dk_out, float *dv_out, float *dg, float *dbeta,
                                float *d_initial_state, void *workspace, size_t workspace_bytes,
                                kda_stream_t stream);

/* Bytes of workspace kda_backward needs for these sizes (an upper bound for any n_seqs <= max(B, n_seqs)). */
KDA_API size_t kda_backward_workspace_size(kda_dtype dtype, int B, int T, int H, int dk, int dv, int n_seqs);

/*
 * kda_prefill_noalloc -- kda_prefill without a caller workspace and without any allocation: a
 * call that is split along the sequence uses a fixed scratch array compiled into the library
 * (one per device, kda_prefill_noalloc_capacity() bytes, placed when the library's device code
 * is loaded). The pages describe no such call; it exists for callers that cannot hand over
 * device memory. Arguments as kda_prefill, without workspace / workspace_bytes; results
 * identical to kda_prefill with a workspace. Returns KDA_ERR_UNSUPPORTED, before anything is
 * queued, when kda_prefill_workspace_size() for the call exceeds the capacity. Calls that use the
 * scratch are ordered on the device (each waits for the previous one, whatever its stream).
 */
KDA_API kda_status kda_prefill_noalloc(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                                       const void *q, const void *k, const void *v, const void *g,
                                       const void *beta, const int32_t *cu_seqlens, int n_seqs,
                                       const float *initial_state, void *o, float *final_state,
                                       kda_stream_t stream);

/*
 * kda_prefill_debug_dump -- diagnostic with no counterpart on the pages: it exists so that a test
 * can locate a fault of the tensor-core prefill to one stage of the chunkwise form. Runs kda_prefill
 * (bf16, dk == dv == 128, B sequences of T tokens, no cu_seqlens, no options) and, for the first
 * (sequence, head) only, writes the kernel's intermediates of its first dump_chunks chunks of 64
 * tokens to `dump` (fp32, device, 16-byte aligned, dump_chunks * 40960 floats), chunk after chunk:
 *   [0, 8192)       Gam = cumsum of g within the chunk, [token][d_k] (rows past the sequence end
 *                   repeat the last row)
 *   [8192, 12288)   A = strict_lower(Diag(beta) (K exp Gam)(K exp -Gam)^T), [token][token]
 *   [12288, 16384)  T = (I + A)^{-1} Diag(beta) as the kernel's bf16 operand, [token][token]
 *   [16384, 24576)  U = T (V - (K exp Gam) S), [token][d_v]
 *   [24576, 40960)  S at the chunk start, [d_k][d_v]
 * (the quantities of "Kimi Delta Attention: the linear core", maidul-haque blog, in the chunkwise
 * form). o and final_state as kda_prefill. Returns KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED on the
 * host, else KDA_OK once queued.
 */
KDA_API kda_status kda_prefill_debug_dump(int B, int T, int H, const void *q, const void *k, const void *v,
                                          const void *g, const void *beta, const float *initial_state, void *o,
                                          float *final_state, float *dump, int dump_chunks, kda_stream_t stream);

/* Bytes of the fixed scratch array kda_prefill_noalloc uses. */
KDA_API size_t kda_prefill_noalloc_capacity(void);

/*
 * kda_decode_step -- one token of the recurrence for N independent sequences.
 *
 * q, k, g  [N, H, dk]; v [N, H, dv]; beta [N, H]; o [N, H, dv]; all `dtype`.
 * state    fp32 [N, H, dk, dv], read and updated in place (S_{t-1} -> S_t).
 * o        receives o_t = S_t^T q_t.
 * Supported: dk == dv in {32, 64, 128}; pointers 16-byte aligned.
 */
KDA_API kda_status kda_decode_step(kda_dtype dtype, int N, int H, int dk, int dv,
                           const void *q, const void *k, const void *v, const void *g,
                           const void *beta, float *state, void *o, kda_stream_t stream);

/*
 * kda_prefill_gated / kda_decode_step_gated -- kda_prefill / kda_decode_step with the gate given
 * as raw logits x (same layout and dtype as g) instead of log-decays: the kernels form
 * g = -gate_bound * sigmoid(x) per element, the scaled sigmoid whose lower bound makes the decay
 * bounded ("Kimi K3 Explained", researchpapers.dev, "Architecture at a glance"; the workloads'
 * log-decay is -5 sigmoid(N(0,1))). g then lies in (-gate_bound, 0); the accuracy statement for
 * g in [-5, 0] covers gate_bound <= 5. gate_bound must be finite and in (0, 1e4], else
 * KDA_ERR_INVALID_ARG. Every other argument, and the return values, as the plain forms.
 */
KDA_API kda_status kda_prefill_gated(kda_dtype dtype, int B, int T, int H, int dk, int dv,
                                     const void *q, const void *k, const void *v,
                                     const void *gate_logits, const void *beta,
                                     const int32_t *cu_seqlens, int n_seqs,
                                     const float *initial_state, void *o, float *final_state,
                                     float gate_bound, void *workspace, size_t workspace_bytes,
                                     kda_stream_t stream);

KDA_API kda_status kda_decode_step_gated(kda_dtype dtype, int N, int H, int dk, int dv,
                                         const void *q, const void *k, const void *v,
                                         const void *gate_logits, const void *beta, float *state,
                                         void *o, float gate_bound, kda_stream_t stream);

/*
 * kda_check_status -- synchronise `stream`, then read and clear the device error word of the
 * current device. Returns KDA_OK, KDA_ERR_INVALID_ARG (bad cu_seqlens or a state slot past
 * the pool end seen by a kernel), KDA_ERR_TIMEOUT (a bounded pipeline wait gave up; that
 * (sequence, head) is left unfinished) or KDA_ERR_CUDA (the synchronisation itself failed).
 */
KDA_API kda_status kda_check_status(kda_stream_t stream);

/*
 * kda_selftest_wait_timeout -- diagnostic for the library's failure detection (the pages have no
 * counterpart: it exists so that a caller or a test can see a stalled pipeline being reported).
 * Queues on `stream` one small kernel whose thread waits, bounded by `limit_ns` nanoseconds of
 * %globaltimer, on an mbarrier phase that nothing completes -- the same bounded wait that every
 * pipeline wait of the prefill kernel uses -- then records KDA_ERR_TIMEOUT in the device error
 * word and exits normally; the context stays usable. limit_ns must be in [1, 1e9].
 * Returns KDA_OK once queued (the timeout itself is reported by kda_check_status),
 * KDA_ERR_INVALID_ARG for an out-of-range limit, KDA_ERR_CUDA if the launch failed.
 */
KDA_API kda_status kda_selftest_wait_timeout(uint64_t limit_ns, kda_stream_t stream);

/* Static, human-readable name of a status code. */
KDA_API const char *kda_status_string(kda_status status);

/* Detail of the most recent failure in the calling host thread ("" if none). */
KDA_API const char *kda_last_error(void);

/* Library ABI version: major * 10000 + minor * 100 + patch. Version 2 made packed calls to
 * kda_prefill_workspace_size explicit (the cu_seqlens argument). */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
