/*
 * flce.h - C ABI of the GB300 fused linear cross-entropy (FLCE) library.
 *
 * The operation is the loss of a language-model head computed without keeping
 * the [tokens, vocab] logits (Liger-Kernel, "Muse Glimmer" support, section
 * Summary item 1; DeepSeek-V3 support, section Summary: "logits are never
 * materialized", and section Memory: logits replaced by chunked transients and
 * a fixed fp32 weight-gradient accumulator).
 *
 * For rows i = 0..N-1 with hidden states h_i (bf16, length H), the lm-head
 * weight W (bf16, [V, H]) and labels y_i (int64, ignore_index marks rows that
 * do not count):
 *
 *   z_i   = m (h_i W^T)                 m = out_mult, folded into h (Muse Glimmer
 *                                        page, Details / Softcap)
 *   s_i   = T tanh(z_i / T) if T > 0, else z_i        T = softcap (same section)
 *   lse_i = log sum_j exp(s_ij)
 *   loss  = sum over valid rows of (lse_i - s_{i,y_i}) / n_valid   (MEAN)
 *           or the plain sum (SUM); 0 when n_valid = 0
 *   predicted_i   = argmax_j s_ij (lowest index on ties), every row
 *   token_accuracy = #{valid i : predicted_i = y_i} / n_valid, 0 when n_valid = 0
 *                    (Muse Glimmer page, Summary item 2 and Testing Done)
 *   dz_ij = c (softmax(s_i)_j - [j = y_i]) (1 - (s_ij/T)^2 if T > 0),
 *           c = grad_scale / n_valid (MEAN) or grad_scale (SUM), 0 on ignored rows;
 *           dz is rounded to bf16 before the two backward products
 *   grad_h_i = m sum_j dz_ij W_j                      (bf16 output, fp32 accumulate)
 *   grad_W_j += m sum_i dz_ij h_i                     (fp32, ACCUMULATED in place;
 *           the Muse Glimmer and DeepSeek-V3 pages, section Memory, keep this
 *           accumulator in fp32; NULL means a frozen projection, as in the
 *           SpecForge DSpine PR, section Changes)
 *
 * flce_ce_only is the cheap CE-only pass of the SpecForge DSpine PR (section
 * Changes: only the backbone CE during the graph-free accumulation prepass).
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers owned by the caller, except the
 *    host inputs and host results of the *_from_host entry points. The
 *    library allocates no memory and keeps no state between calls except a
 *    launch counter and optional profiling events.
 *  - Row-major layouts: h [N, ld_h] (ld_h >= H), W [V, ld_w] (ld_w >= H),
 *    grad_h [N, H] contiguous, grad_W [V, H] contiguous, labels/predicted/
 *    row_lse [N] contiguous. h, W and the workspace must be 16-byte aligned,
 *    ld_h and ld_w multiples of 8 elements, H a multiple of 8.
 *  - Scalars (loss, token_accuracy) are written to DEVICE memory, so calls
 *    never synchronise the host. They run asynchronously on `stream` (a
 *    cudaStream_t; NULL = legacy default stream).
 *  - The return value is FLCE_OK or a host-detected error, returned before
 *    any launch. Errors found on the device (bad labels, a bounded wait that
 *    gave up, a non-finite row) are OR-ed into a status word in the
 *    workspace; read it with flce_get_status. On a bad label or a timeout the
 *    outputs are unspecified.
 *  - Nothing traps, prints or throws across this boundary.
 *  - The current CUDA device (cudaSetDevice) must be the device that owns
 *    `stream` and every device pointer of the call: the library takes the SM
 *    count, its one-time per-device kernel set-up and (flce_ce_only_noalloc)
 *    its static scratch array from the current device.
 *  - FLCE_ERR_TIMEOUT means a kernel gave up waiting and returned early. Its
 *    own in-flight copies are drained under the same time limit, and if that
 *    drain also runs out, copies may still land after the kernel has exited.
 *    The outputs of such a call, and of work running beside it on the device,
 *    are then undefined: synchronise, read the status, and discard them.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-detected return codes. */
#define FLCE_OK 0
#define FLCE_ERR_ARG 1          /* null pointer, bad size, negative softcap, bad reduction */
#define FLCE_ERR_ALIGN 2        /* pointer or row stride not 16-byte aligned, H % 8 != 0 */
#define FLCE_ERR_WORKSPACE 3    /* workspace smaller than flce_workspace_size() */
#define FLCE_ERR_UNSUPPORTED 4  /* device is not sm_103, or a tensor map cannot be encoded */
#define FLCE_ERR_CUDA 5         /* a CUDA runtime call or launch failed */
/* Device-detected bits of the status word (flce_get_status). */
#define FLCE_ERR_LABEL 16       /* a label is neither ignore_index nor in [0, V) */
#define FLCE_ERR_TIMEOUT 32     /* a bounded pipeline wait gave up; the kernel returned early */
#define FLCE_ERR_NONFINITE 64   /* a row's log-sum-exp is not finite (inf or NaN in h or W, or
                                   logits beyond fp32 range); that row's predicted token is -1
                                   and its loss and gradients are not meaningful; the other rows
                                   are unaffected */

/* Modes for flce_workspace_size. */
#define FLCE_MODE_CE_ONLY 0
#define FLCE_MODE_FORWARD 1
#define FLCE_MODE_FORWARD_BACKWARD 2
#define FLCE_MODE_CROSS_ENTROPY 3   /* flce_cross_entropy on materialised logits */
#define FLCE_MODE_FORWARD_BACKWARD_HOST 4  /* flce_forward_backward_from_host */
#define FLCE_MODE_CE_ONLY_HOST 5           /* flce_ce_only_from_host */

#define FLCE_REDUCTION_MEAN 0
#define FLCE_REDUCTION_SUM 1
#define FLCE_REDUCTION_NONE 2       /* flce_cross_entropy only: per-row losses, per-row upstream grads */

/* Element types of materialised logits (flce_cross_entropy). */
#define FLCE_DTYPE_BF16 0
#define FLCE_DTYPE_F32 1

/* Flags (flce_params.flags). */
#define FLCE_FLAG_SIMT_GEMM 1        /* debug: plain fp32-FMA GEMMs instead of tcgen05 */
#define FLCE_FLAG_TEST_STALL 2       /* test hook: the forward GEMM's loader issues no copies,
                                        so its bounded waits run out (FLCE_ERR_TIMEOUT) */
#define FLCE_FLAG_KMAJOR_BWD 4       /* cross-check: feed the backward GEMMs explicit transposes
                                        (W^T, dz^T, h^T) instead of MN-major tiles */
#define FLCE_FLAG_RECOMPUTE 8        /* low-memory backward: keep no logits; per vocab slab of
                                        vocab_slab columns, recompute z = m h W^T on the tensor
                                        cores and form bf16 dlogits in the GEMM epilogue's
                                        registers, then run both backward GEMMs on the slab.
                                        Transient O(C * vocab_slab + C * H); 8NHV flops, not 6NHV */
#define FLCE_FLAG_TILE128 16         /* every bf16 tensor-core GEMM on 128 x 256 CTA tiles
                                        with two TMEM accumulators. By default each GEMM takes
                                        256 x 256 tiles (two M = 128 MMAs per K step sharing one
                                        B slice) unless its tile count is too small for them to
                                        fill the SMs evenly */
#define FLCE_FLAG_TILE256 32         /* cross-check: 256 x 256 CTA tiles for every bf16 GEMM
                                        that has them, whatever the tile count */
#define FLCE_FLAG_F32_3PASS 128     /* fp32 operands (FLCE_DTYPE_F32): every product as three tf32
                                        products, hi*hi + hi*lo + lo*hi with hi = x rounded to tf32
                                        and lo = x - hi, for about fp32 accuracy (the default fp32
                                        path multiplies in tf32, a 10-bit mantissa); 3x the tensor
                                        work, 128 x 256 tiles, and hi / lo copies of W, W^T, h_c,
                                        h_c^T, dz and dz^T in the workspace */
#define FLCE_FLAG_CTA_PAIR 64        /* the bf16 GEMMs that take 256 x 256 tiles compute each on a
                                        pair of CTAs (a cluster of two SMs, tcgen05 cta_group::2):
                                        each SM holds 128 rows, so its accumulator is double-
                                        buffered and the epilogue overlaps the next tile's MMAs */
#define FLCE_FLAG_VP_STORED 256      /* vocab shards (flce_vp_forward / flce_vp_backward): the
                                        forward keeps the shard's capped logits in the workspace
                                        (fp16, relative to each 32-column group's max, as the
                                        fused backward stores them) and the backward forms
                                        dlogits from them instead of recomputing the logits:
                                        6 N H V_k tensor flops per shard instead of 8, and
                                        O(N * V_k) workspace (the logits of all N rows; dlogits
                                        one chunk at a time). The two calls take the same params
                                        and the same workspace, which nothing else may use in
                                        between */

typedef struct flce_params {
  int64_t n_rows;        /* N >= 0 */
  int64_t hidden;        /* H > 0, multiple of 8 */
  int64_t vocab;         /* V > 0, < 2^31 */
  int64_t ld_h;          /* row stride of h in elements (0 => H) */
  int64_t ld_w;          /* row stride of W in elements (0 => H) */
  float softcap;         /* T >= 0; 0 => no softcap */
  float out_mult;        /* m, the output multiplier folded into h */
  int64_t ignore_index;  /* rows with this label do not count (default -100) */
  int32_t reduction;     /* FLCE_REDUCTION_MEAN (default) or FLCE_REDUCTION_SUM */
  float grad_scale;      /* g: upstream dL/dloss multiplying every gradient (default 1) */
  int64_t chunk_rows;    /* rows per chunk C (0 => 8192); at most 32768; rounded up to 128 */
  int32_t flags;         /* FLCE_FLAG_* */
  int64_t timeout_ns;    /* limit of each bounded device wait (0 => 2 s) */
  int64_t vocab_slab;    /* FLCE_FLAG_RECOMPUTE: vocab columns per slab (0 => 16384);
                            rounded up to 256 */
  int32_t dtype;         /* element type of h, W and grad_h: FLCE_DTYPE_BF16 (default) or
                            FLCE_DTYPE_F32 (fp32 operands and fp32 grad_h; the products are
                            tf32 products - 10-bit mantissas, fp32 accumulation - unless
                            FLCE_FLAG_F32_3PASS asks for fp32 accuracy; not with
                            FLCE_FLAG_RECOMPUTE or FLCE_FLAG_SIMT_GEMM) */
} flce_params;

/* Fills the defaults: softcap 0, out_mult 1, ignore_index -100, MEAN,
 * grad_scale 1, chunk_rows 0, flags 0, timeout 0; sizes and strides 0. */
void flce_default_params(flce_params* p);

/* Bytes of device workspace a call needs. mode is FLCE_MODE_*; need_grad_h and
 * need_grad_W (0/1) matter for FORWARD_BACKWARD only. Depends on C, H and V
 * but not on N beyond min(N, C): the transient memory is O(C * V).
 * Returns 0 for invalid parameters. */
size_t flce_workspace_size(const flce_params* p, int mode, int need_grad_h, int need_grad_W);

/* Rows per chunk that a call with these arguments uses: chunk_rows rounded up
 * to a multiple of 128 (at most 32768 and at most N rounded up), or, when
 * chunk_rows is 0, the library's choice: 8192, except for the stored-logits
 * bf16 backward, which takes the multiple of 256 from 8192 to 10240 whose
 * chunks fill the tensor-core GEMMs' waves best on 152 SMs (8192 on ties).
 * Returns 0 for invalid parameters. */
int64_t flce_chunk_rows(const flce_params* p, int mode, int need_grad_h, int need_grad_W);

/* CE-only pass: loss and (optionally) token_accuracy, no gradients, no saved
 * state. loss: device float scalar; token_accuracy: device float scalar or NULL. */
int flce_ce_only(const flce_params* p, const void* h, const void* W, const int64_t* labels,
                 float* loss, float* token_accuracy,
                 void* workspace, size_t workspace_bytes, void* stream);

/* CE-only pass that allocates nothing and takes no workspace: for callers that
 * cannot allocate device memory where they need the loss (code inside an
 * allocator's callbacks, hooks that run while a framework's allocator is
 * locked, embeddings that forbid device allocations after start-up). The pages
 * have no counterpart of this entry point; it exists only for such callers.
 * Same computation and outputs as flce_ce_only; device_status (device int32,
 * nullable) receives the call's status word (0, FLCE_ERR_LABEL, FLCE_ERR_TIMEOUT).
 * Scratch is a fixed 64 MiB device array inside the library, reserved on every
 * GPU that loads it until the process exits. chunk_rows = 0 picks the largest
 * chunk (8192 down to 128 rows) that fits; FLCE_ERR_WORKSPACE means the
 * vocabulary (or the given chunk_rows) needs more than 64 MiB. The first call
 * on a device looks up the array's address and should come before any stream
 * capture. All calls share the array: calls that overlap on the GPU race, so
 * serialise them. No call allocates device memory. */
int flce_ce_only_noalloc(const flce_params* p, const void* h, const void* W, const int64_t* labels,
                         float* loss, float* token_accuracy, int32_t* device_status, void* stream);

/* Forward: as flce_ce_only, plus optional per-row outputs predicted [N]
 * (int64, argmax for every row) and row_lse [N] (fp32 log-sum-exp of s_i).
 * With predicted NULL (here, in flce_forward_backward and in flce_ce_only) the
 * forward epilogue skips the argmax and keeps only what token_accuracy needs:
 * whether each row's label is its first maximum. The accuracy is the same,
 * bit for bit. */
int flce_forward(const flce_params* p, const void* h, const void* W, const int64_t* labels,
                 float* loss, float* token_accuracy, int64_t* predicted, float* row_lse,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Forward + backward: the forward outputs plus grad_h (bf16 [N, H], written;
 * NULL => not computed) and grad_W (fp32 [V, H], ACCUMULATED: grad_W += dL/dW;
 * NULL => frozen W, skipped). */
int flce_forward_backward(const flce_params* p, const void* h, const void* W,
                          const int64_t* labels, float* loss, float* token_accuracy,
                          int64_t* predicted, void* grad_h, float* grad_W,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Forward + backward with the inputs in HOST memory: h_host (bf16, rows of
 * ld_h elements) and labels_host (int64 [N]) are host pointers; page-locked
 * memory lets the copies overlap the kernels, pageable memory works but the
 * copies then serialise. The labels are copied first (the prologue counts them
 * all); h then goes over one chunk at a time on `copy_stream` into two staging
 * buffers in the workspace, the copy of chunk k + 1 running under the kernels
 * of chunk k on `stream`, ordered by events that the call creates and
 * releases. loss_host and token_accuracy_host (nullable) are HOST floats,
 * written by copies on `stream` at the end: read them after synchronising
 * `stream`. W, predicted, grad_h and grad_W are device pointers as in
 * flce_forward_backward. copy_stream may equal stream (the copies then do not
 * overlap). h is bf16, or fp32 with p->dtype = FLCE_DTYPE_F32;
 * FLCE_ERR_UNSUPPORTED with FLCE_FLAG_SIMT_GEMM or FLCE_FLAG_KMAJOR_BWD. Workspace: flce_workspace_size(p,
 * FLCE_MODE_FORWARD_BACKWARD_HOST, ...), which adds two chunks of h and N
 * labels to the FORWARD_BACKWARD size. The host buffers must stay valid and
 * unchanged until `stream` has finished the call's work. The call creates and
 * releases CUDA events, so it is not meant for stream capture. */
int flce_forward_backward_from_host(const flce_params* p, const void* h_host, const void* W,
                                   const int64_t* labels_host, float* loss_host, float* token_accuracy_host,
                                   int64_t* predicted, void* grad_h, float* grad_W, void* workspace,
                                   size_t workspace_bytes, void* stream, void* copy_stream);

/* CE-only pass with h and labels in HOST memory, staged as in
 * flce_forward_backward_from_host; loss_host and token_accuracy_host (nullable)
 * are host floats, valid once `stream` has finished. Workspace:
 * flce_workspace_size(p, FLCE_MODE_CE_ONLY_HOST, 0, 0). */
int flce_ce_only_from_host(const flce_params* p, const void* h_host, const void* W, const int64_t* labels_host,
                           float* loss_host, float* token_accuracy_host, void* workspace, size_t workspace_bytes,
                           void* stream, void* copy_stream);

/* Cross-entropy on logits that are already materialised, [N, V] with row
 * stride ld_logits (>= V) in bf16 or fp32 (logits_dtype): the non-fused branch
 * the Liger-Kernel "Muse Glimmer" page tests next to the fused path (Testing
 * Done: the non-fused softcap branch; Details / Softcap: T tanh(logits m / T)),
 * and what DeepSeek-V3's lce_forward does when logits are kept (Summary).
 * Same per-row definition as the fused path with z = m * logits (p->hidden is
 * ignored). reduction: MEAN, SUM, or NONE (per-row losses; loss = their sum;
 * the gradient of sum_i row_scale_i * l_i, row_scale NULL = all ones).
 * Outputs (all device, nullable except loss): token_accuracy, predicted [N],
 * row_loss [N] (0 on ignored rows), grad_logits (dL/dlogits, logits' dtype,
 * [N, ld_logits]; may alias logits to overwrite them in place).
 * Workspace: flce_workspace_size(p, FLCE_MODE_CROSS_ENTROPY, 0, 0). */
int flce_cross_entropy(const flce_params* p, const void* logits, int logits_dtype, int64_t ld_logits,
                       const int64_t* labels, float* loss, float* token_accuracy, int64_t* predicted,
                       float* row_loss, const float* row_scale, void* grad_logits,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Multiplies a gradient by a device scalar and converts it: y_k = scale * x_k
 * for k < n, rounded to y_dtype (bf16 with round to nearest even). This is the
 * upstream factor of an autograd backward (the chain rule through the loss):
 * the fused entry points take grad_scale as a host float, but a caller that
 * computes the gradients during the forward, as the pages' fused
 * linear-cross-entropy functions do, learns the factor only afterwards, as a
 * device scalar. x, y: device arrays of n elements of x_dtype / y_dtype
 * (FLCE_DTYPE_*), in any alignment (16-byte aligned ones take the vector
 * path); y may be x itself (in place) when the dtypes match, and must not
 * overlap it otherwise. scale: device float, or NULL for 1.
 * Returns FLCE_ERR_ARG for n < 0, an unknown dtype, a NULL array with n > 0
 * or an overlap that is not exact in-place; FLCE_ERR_UNSUPPORTED off sm_103. */
int flce_scale_gradient(const void* x, int x_dtype, void* y, int y_dtype, int64_t n, const float* scale,
                        void* stream);

/* ---------------------------------------------------------------- vocab-parallel
 * The head's weight split by vocabulary rows over S shards, one per GPU (or run
 * one after another on one GPU): shard k holds W's rows for vocab ids
 * [o_k, o_{k+1}), 0 = o_0 < o_1 < ... < o_S = vocab_total, and sees all N rows
 * of h and all labels (global vocab ids). This is the vocabulary-sharded form of
 * the fused head for the distributed (DDP / FSDP) runs of the SpecForge DSpine
 * PR (section Validation); each shard keeps its transients chunked as on the
 * Liger-Kernel DeepSeek-V3 page (section Memory). One step is:
 *   1. every shard: flce_vp_forward, its per-row partials (4 x N floats);
 *   2. exchange: every shard obtains all S partial sets in shard order,
 *      [S][4][N] (an all-gather: 16 bytes per row and shard cross GPUs);
 *   3. every shard: flce_vp_backward, which merges them in shard order into the
 *      loss, token accuracy, predicted tokens and lse (bit-identical on every
 *      shard), then adds its own rows of grad_W and its part of grad_h, which
 *      the caller sums over the shards (an all-reduce) and rounds.
 * The backward recomputes the shard's logits per vocab slab, as
 * FLCE_FLAG_RECOMPUTE does, so only the partials cross shards and no logits
 * are kept between the calls: 8 N H V_k tensor flops per shard, transient
 * memory O(C * vocab_slab + N). With FLCE_FLAG_VP_STORED the forward keeps
 * them in the workspace instead (6 N H V_k flops, O(N * V_k) memory). bf16 operands only (FLCE_ERR_UNSUPPORTED for
 * fp32, FLCE_FLAG_SIMT_GEMM and FLCE_FLAG_KMAJOR_BWD).
 * In both calls p->vocab is V_k, the shard's row count, and W_shard is
 * [V_k, ld_w]; labels are checked against [0, vocab_total) (FLCE_ERR_LABEL).
 * Partials, row i (float words, field stride N): [0] max of s over the shard,
 * [1] sum of exp(s - max), [2] argmax as the bit pattern of an int32 global
 * vocab id (the lowest on ties), [3] s at the label if the label is in the
 * shard, else 0. */

/* Workspace bytes of flce_vp_forward (backward = 0) or flce_vp_backward
 * (backward = 1; need_grad_h / need_grad_W as that call will have them). The
 * backward's includes 4 bytes of lse per row (all N rows). With
 * FLCE_FLAG_VP_STORED both calls need the same size, which holds the kept
 * logits (about N * V_k * 2.1 bytes, and C * V_k * 2 for one chunk's
 * dlogits). 0 if invalid. */
size_t flce_vp_workspace_size(const flce_params* p, int backward, int need_grad_h, int need_grad_W);

/* Forward of one shard: writes partials [4][N] (device). FLCE_ERR_ARG when
 * [vocab_offset, vocab_offset + V_k) is not inside [0, vocab_total), and for
 * FLCE_FLAG_VP_STORED with FLCE_FLAG_RECOMPUTE or FLCE_FLAG_KMAJOR_BWD. */
int flce_vp_forward(const flce_params* p, int64_t vocab_offset, int64_t vocab_total, const void* h,
                    const void* W_shard, const int64_t* labels, float* partials, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Backward of one shard, given every shard's partials all_partials [S][4][N]
 * (device) and the host table shard_offsets [S + 1] (S <= 64; FLCE_ERR_ARG if
 * it is not increasing from 0 to vocab_total or does not contain this shard).
 * Writes loss and token_accuracy (device floats; token_accuracy, predicted
 * [N] int64 and row_lse [N] nullable) exactly as flce_forward would for the
 * whole vocabulary, up to the order of the fp32 merge. grad_h_partial: fp32
 * [N, H], ACCUMULATED (+= this shard's m dz_k W_k); summed over all shards it
 * is grad_h. grad_W_shard: fp32 [V_k, H], ACCUMULATED. Either may be NULL. */
int flce_vp_backward(const flce_params* p, int64_t vocab_offset, int64_t vocab_total, int n_shards,
                     const int64_t* shard_offsets, const float* all_partials, const void* h, const void* W_shard,
                     const int64_t* labels, float* loss, float* token_accuracy, int64_t* predicted,
                     float* row_lse, float* grad_h_partial, float* grad_W_shard, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Synchronises `stream` and returns (in *status) the device status word of the
 * last call that used this workspace: 0, or an OR of FLCE_ERR_LABEL,
 * FLCE_ERR_TIMEOUT and FLCE_ERR_NONFINITE.
 * Return value: FLCE_OK or FLCE_ERR_ARG / FLCE_ERR_CUDA. */
int flce_get_status(const void* workspace, void* stream, int32_t* status);

/* Static text for a return code or status bit set. Never NULL. */
const char* flce_status_string(int code);

/* Number of kernels this library has launched in this process. */
int64_t flce_launch_count(void);

/* Per-kernel timing with CUDA events recorded on the launching stream around
 * each launch. flce_profile_begin(1) starts collecting (clears old records),
 * flce_profile_begin(0) stops. flce_profile_read synchronises the recorded
 * events and fills, for kernel ids 0..n-1, the launch count and the summed
 * milliseconds; it returns the number of kernel ids (FLCE_NUM_KERNELS). */
#define FLCE_NUM_KERNELS 17
int flce_profile_begin(int enable);
int flce_profile_read(int64_t* launches, double* total_ms, int n);
const char* flce_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H */
