/*
 * lce.h -- C ABI of the GB300 (sm_103a) fused chunked linear + cross-entropy
 * library (liblce_gb300.so).
 *
 * The operation. Given hidden states H[N,D], the LM-head weight W[V,D] and
 * labels y[N], the library computes the logits Z = H W^T chunk by chunk on
 * chip, the per-row log-sum-exp lse_i, the mean loss over non-ignored rows
 *     loss = sum_{valid i} (lse_i - Z[i, y_i]) / N_valid,
 * and the analytic gradients
 *     G[i,j] = (exp(Z[i,j] - lse_i) - 1[j = y_i]) * dloss / N_valid  (0 for ignored rows)
 *     dH = G W,   dW = G^T H,
 * without ever holding the full [N,V] logits or G in device memory.
 * Sources: "Arquitectura interna de Unsloth y optimizacion en Triton", section 3
 * "Fused Cross Entropy" (token blocks, on-chip logits, online log-sum-exp, the
 * softmax - onehot gradient, backpropagation into X and W_vocab); "Unsloth
 * Architecture: Manual Triton Backpropagation, Fused Cross-Entropy, and 80% VRAM
 * Cut", pillar 1 "Fused Chunked Cross-Entropy Loss" (chunks of tokens, the
 * per-row loss -z_{i,y_i} + log sum_j exp z_ij and the gradient p - 1[j = y_i]);
 * "Unsloth Kernel Architecture: Custom Triton Backpropagation and QLoRA Memory
 * Scaling", section 1 "Fused Cross-Entropy Loss with Logit Streaming" (vocab
 * blocks streamed per row with a running max and running sum).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device,
 *    row-major and contiguous, and 16-byte aligned. H and W are bf16
 *    (IEEE bfloat16, 2 bytes), y is int64, lse / dW / loss / dloss are fp32,
 *    dH is bf16.
 *  - D must be a multiple of 8 (16-byte rows for the tensor-memory copies);
 *    N, V and chunk are otherwise arbitrary (ragged tails are masked).
 *  - The caller owns every buffer, including the workspace (ws, ws_bytes) of at
 *    least lce_workspace_size() bytes. The library allocates no device memory.
 *    The workspace extent is O(chunk * V) plus O(N) bytes.
 *  - All work is enqueued on `stream`; no entry point synchronises the host.
 *    (The gradient phase runs part of its kernels on a stream the library owns,
 *    forked from and joined back to `stream` through events, so every call is
 *    ordered after earlier work on `stream` and before later work on it, and it
 *    can be captured in a CUDA graph. Several host threads may call the library
 *    at once, each with its own buffers.)
 *    Argument errors are returned before anything is enqueued. Errors found on
 *    the device (labels outside [0,V) that are not ignore_index, a bounded wait
 *    that ran out) are recorded in the workspace and returned by
 *    lce_read_status(), which synchronises the stream.
 *  - Rows whose label is ignore_index (usually -100) add nothing to the loss and
 *    get zero dH rows. Labels outside [0,V) other than ignore_index are treated
 *    the same way and flag LCE_ERR_LABEL_RANGE. With no valid row at all the
 *    loss is 0 and dH, dW are 0.
 *  - Results are deterministic: two calls with the same inputs give the same
 *    bits (fixed reduction orders, no floating-point atomics).
 *  - The kernels are built for sm_103a only; other devices get
 *    LCE_ERR_UNSUPPORTED.
 */
#ifndef LCE_GB300_H
#define LCE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lce_status {
    LCE_OK = 0,
    LCE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, D % 8 != 0, chunk <= 0 */
    LCE_ERR_ALIGNMENT = 2,     /* a pointer not 16-byte aligned */
    LCE_ERR_WORKSPACE = 3,     /* ws_bytes < lce_workspace_size() */
    LCE_ERR_LABEL_RANGE = 4,   /* device: some label outside [0,V) and != ignore_index */
    LCE_ERR_TIMEOUT = 5,       /* device: a bounded pipeline wait ran out; outputs invalid */
    LCE_ERR_CUDA = 6,          /* a CUDA runtime call failed */
    LCE_ERR_UNSUPPORTED = 7    /* current device is not sm_103, or an option combination
                                  the library does not offer (fp16 with reduction NONE) */
} lce_status;

/* Same type as cudaStream_t. NULL means the legacy default stream. */
typedef struct CUstream_st *lce_stream_t;

/* Bytes of workspace the calls below need for these sizes (enough for all three
 * calls). Writes *bytes; returns LCE_ERR_INVALID_ARG for bad sizes. */
lce_status lce_workspace_size(int64_t N, int64_t D, int64_t V, int64_t chunk, size_t *bytes);

/* Bytes of workspace lce_forward (and lce_forward_ex / _opt) needs: the header,
 * the per-row losses (4 N bytes), the chunk's target logits and its (max, sum)
 * partial per 128-column slab (8 chunk ceil(V/128) bytes); no chunk buffer, since
 * the forward stores no logits. At most lce_workspace_size(). */
lce_status lce_forward_workspace_size(int64_t N, int64_t D, int64_t V, int64_t chunk,
                                      size_t *bytes);

/* Forward: loss (device scalar, fp32) and lse[N] (device, fp32).
 * Work: 2*N*D*V flops on the tensor cores, chunk rows at a time. The workspace
 * needs lce_forward_workspace_size() bytes. */
lce_status lce_forward(const void *H, const void *W, const int64_t *y,
                       int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                       float *loss, float *lse,
                       void *ws, size_t ws_bytes, lce_stream_t stream);

/* Backward from a saved lse[N]: recomputes each chunk's logits (2*N*D*V flops),
 * forms G in bf16 and writes dH[N,D] (bf16, overwritten) and dW[V,D] (fp32,
 * overwritten) with 4*N*D*V more flops. dloss is a device fp32 scalar (the
 * upstream gradient of the mean loss); NULL means 1. */
lce_status lce_backward(const void *H, const void *W, const int64_t *y, const float *lse,
                        const float *dloss, void *dH, float *dW,
                        int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                        void *ws, size_t ws_bytes, lce_stream_t stream);

/* Fused forward + backward without the recompute (6*N*D*V flops): writes loss,
 * lse, dH (bf16) and dW (fp32). dloss as in lce_backward (NULL means 1). */
lce_status lce_fwd_bwd(const void *H, const void *W, const int64_t *y, const float *dloss,
                       int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                       float *loss, float *lse, void *dH, float *dW,
                       void *ws, size_t ws_bytes, lce_stream_t stream);

/* Reductions of the loss (a library option; the pages use the mean):
 *  MEAN: loss = sum over valid rows / N_valid (device scalar); G = (p - onehot) * dloss / N_valid.
 *  SUM:  loss = sum over valid rows (device scalar); G = (p - onehot) * dloss.
 *  NONE: loss[N] = per-row losses (0 for ignored rows); dloss is NULL (all 1) or a
 *        device vector dloss[N], and row i of G is (p_i - onehot_i) * dloss[i].
 * The _ex entry points take one of these; the entry points above are MEAN. */
enum { LCE_REDUCTION_MEAN = 0, LCE_REDUCTION_SUM = 1, LCE_REDUCTION_NONE = 2 };

lce_status lce_forward_ex(const void *H, const void *W, const int64_t *y,
                          int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                          int reduction, float *loss, float *lse,
                          void *ws, size_t ws_bytes, lce_stream_t stream);
lce_status lce_backward_ex(const void *H, const void *W, const int64_t *y, const float *lse,
                           const float *dloss, void *dH, float *dW,
                           int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                           int reduction, void *ws, size_t ws_bytes, lce_stream_t stream);
lce_status lce_fwd_bwd_ex(const void *H, const void *W, const int64_t *y, const float *dloss,
                          int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                          int reduction, float *loss, float *lse, void *dH, float *dW,
                          void *ws, size_t ws_bytes, lce_stream_t stream);

/* Variants with option flags (the _ex entry points are these with flags = 0):
 *  LCE_ACCUMULATE_DW  add this call's dW into the existing contents of dW (fp32)
 *                     instead of overwriting it;
 *  LCE_ACCUMULATE_DH  add dH into the existing contents of dH (the sum is formed
 *                     in fp32 and rounded once), e.g. to accumulate gradients
 *                     over micro-batches or over several losses sharing H;
 *  LCE_INPUT_FP16     H, W (and dH) are fp16 instead of bf16 (the pages name both
 *                     formats). The chunk buffer then holds fp16 values; because
 *                     dloss / N_valid would push G below fp16's range, G is stored
 *                     as (p - onehot) * 2^14 and the gradient GEMMs apply
 *                     dloss / (N_valid * 2^14) to their fp32 accumulators. Reduction
 *                     NONE (a per-row dloss of unknown range inside G) returns
 *                     LCE_ERR_UNSUPPORTED with fp16;
 *  LCE_FROZEN_W       W is not trained (a frozen LM head, as in LoRA / QLoRA
 *                     fine-tuning, the setting of "Unsloth Kernel Architecture:
 *                     Custom Triton Backpropagation and QLoRA Memory Scaling"; the
 *                     worked example of "Step 2" computes d_hidden only): dW is not
 *                     computed and not written, and may be NULL; the gradient phase
 *                     is the dH contraction alone (4NDV flops per step instead of
 *                     6NDV). Not with LCE_ACCUMULATE_DW (LCE_ERR_INVALID_ARG).
 *  LCE_LOW_MEMORY     one chunk buffer instead of two. By default (more than one
 *                     chunk, chunk a multiple of 8, dW computed) the workspace
 *                     holds two [chunk, V] chunk buffers and the chunks go in pairs:
 *                     both chunks' G stay in the buffers and one dW contraction
 *                     runs over the pair (K = two chunks' rows), which halves the
 *                     fp32 read-modify-write of dW; the logits and dH are still
 *                     computed one chunk at a time. With this flag every chunk has
 *                     its own dW contraction (about half the workspace, slower).
 *                     Either way the results meet the same tolerances and are
 *                     deterministic; the two schedules differ in the rounding
 *                     order of dW and of split dH contractions.
 * With LCE_ACCUMULATE_DH, LCE_FROZEN_W or LCE_LOW_MEMORY the workspace is
 * lce_workspace_size_opt(..., flags) bytes (the accumulation needs the chunk's dH in
 * fp32; the frozen-W gradient splits its dH contraction differently and keeps one
 * chunk buffer); otherwise it is lce_workspace_size(), which
 * lce_workspace_size_opt(..., 0) equals. lce_forward_opt takes LCE_INPUT_FP16 (and
 * ignores LCE_LOW_MEMORY: the forward keeps no chunk buffer). Other arguments and
 * outputs as for the _ex entry points. */
enum {
    LCE_ACCUMULATE_DW = 1,
    LCE_ACCUMULATE_DH = 2,
    LCE_INPUT_FP16 = 4,
    LCE_FROZEN_W = 8,
    LCE_LOW_MEMORY = 16,
    LCE_FLAGS_ALL = 31
};
lce_status lce_workspace_size_opt(int64_t N, int64_t D, int64_t V, int64_t chunk, int flags,
                                  size_t *bytes);
lce_status lce_forward_opt(const void *H, const void *W, const int64_t *y,
                           int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                           int reduction, int flags, float *loss, float *lse,
                           void *ws, size_t ws_bytes, lce_stream_t stream);
lce_status lce_backward_opt(const void *H, const void *W, const int64_t *y, const float *lse,
                            const float *dloss, void *dH, float *dW,
                            int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                            int reduction, int flags, void *ws, size_t ws_bytes,
                            lce_stream_t stream);
lce_status lce_fwd_bwd_opt(const void *H, const void *W, const int64_t *y, const float *dloss,
                           int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                           int reduction, int flags, float *loss, float *lse, void *dH, float *dW,
                           void *ws, size_t ws_bytes, lce_stream_t stream);

/* Token-sharded batches (rows split over several calls, e.g. one per GPU, with W
 * replicated): the mean loss over the valid rows of ALL shards. Rows are
 * independent except for the normaliser N_valid, so each shard
 *  1. counts its valid rows with lce_count_valid (labels in [0, V) other than
 *     ignore_index, the rule every call uses) into a device int64,
 *  2. sums the counts of all shards (an all-reduce; not part of this library),
 *  3. calls lce_fwd_bwd_sharded with that total: the call is lce_fwd_bwd_opt
 *     with reduction MEAN, except that the mean divides by *n_valid_total
 *     instead of this call's own count. Its loss is then this shard's share
 *     sum_{valid i here}(lse_i - z_{i,y_i}) / N_total, and G's rows carry
 *     dloss / N_total;
 *  4. sums loss and dW over the shards (all-reduces); dH and lse are per row.
 * The summed loss and dW are those of one call over the whole batch; dH rows are
 * that call's rows. ("Unsloth Architecture: Manual Triton Backpropagation,
 * Fused Cross-Entropy, and 80% VRAM Cut", pillar 1, normalises the loss by the
 * number of counted tokens; the pages run on one GPU and describe no sharding.)
 * n_valid_total is a device int64 below 2^31; flags as for lce_fwd_bwd_opt;
 * the workspace is lce_workspace_size_opt(..., flags) bytes. lce_count_valid
 * needs no workspace; y is 16-byte aligned, n_valid 8-byte aligned. */
lce_status lce_count_valid(const int64_t *y, int64_t N, int64_t V, int64_t ignore_index,
                           int64_t *n_valid, lce_stream_t stream);
lce_status lce_fwd_bwd_sharded(const void *H, const void *W, const int64_t *y, const float *dloss,
                               const int64_t *n_valid_total, int64_t N, int64_t D, int64_t V,
                               int64_t ignore_index, int64_t chunk, int flags, float *loss,
                               float *lse, void *dH, float *dW, void *ws, size_t ws_bytes,
                               lce_stream_t stream);

/* Cross-entropy over logits the caller already has (no projection): the
 * streaming row kernel of "Unsloth Kernel Architecture: Custom Triton
 * Backpropagation and QLoRA Memory Scaling", section 1 (a row of logits
 * streamed in vocabulary blocks with a running max and a running sum of
 * exponentials). Z is [N][ld] row-major, bf16 (z_dtype = 0), fp32 (z_dtype = 1)
 * or fp16 (z_dtype = 2), ld >= V and a multiple of 8 (bf16, fp16) or 4 (fp32)
 * elements. Writes lse[N] and
 * the loss under `reduction` (as above); when dZ is not NULL it also writes
 * dZ = (softmax(Z) - onehot(y)) * scale in Z's dtype, with the same layout
 * (dZ == Z computes the gradient in place). Work: one read of Z, plus one write
 * with dZ, for V up to 524288 (bf16, fp16) / 262144 (fp32); larger rows take a second
 * read. Bound by HBM bandwidth. The workspace is lce_ce_logits_workspace_size(N)
 * bytes; device status as for lce_forward. */
lce_status lce_ce_logits_workspace_size(int64_t N, size_t *bytes);
lce_status lce_ce_logits(const void *Z, int z_dtype, int64_t ld, const int64_t *y,
                         int64_t N, int64_t V, int64_t ignore_index, int reduction,
                         const float *dloss, float *loss, float *lse, void *dZ,
                         void *ws, size_t ws_bytes, lce_stream_t stream);

/* The final RMSNorm in front of the LM head ("Unsloth Architecture: Manual
 * Triton Backpropagation, Fused Cross-Entropy, and 80% VRAM Cut", pillar 3
 * "Fused RMSNorm & SwiGLU Kernels"): per row of X [N][D] (bf16, row-major),
 *   H = X * r * gamma,  r = 1 / sqrt(mean(X^2) + eps),  gamma [D] bf16.
 * D must be a multiple of 8 and at most 8192; pointers 16-byte aligned.
 *
 * lce_rmsnorm_forward: writes H [N][D] bf16 and, if rstd is not NULL, r [N] fp32.
 * No workspace.
 *
 * lce_rmsnorm_backward: for the upstream gradient dH [N][D] (bf16, or fp32 when
 * dh_fp32 = 1) writes dX [N][D] bf16 and dgamma [D] fp32:
 *   dX = r * (gamma * dH) - X * r^3 * (sum_i gamma_i dH_i X_i) / D,
 *   dgamma = sum over rows of dH * X * r.
 * (The page prints the first line with gamma outside the sum, which is exact
 * only for a uniform gamma; this is the exact derivative.) r is recomputed from
 * X (nothing else is kept from the forward). The workspace is
 * lce_rmsnorm_backward_workspace_size(D) bytes (the dgamma partials); results
 * are deterministic. Bound by HBM bandwidth. */
lce_status lce_rmsnorm_forward(const void *X, const void *gamma, int64_t N, int64_t D, float eps,
                               void *H, float *rstd, lce_stream_t stream);
lce_status lce_rmsnorm_backward_workspace_size(int64_t D, size_t *bytes);
lce_status lce_rmsnorm_backward(const void *X, const void *gamma, const void *dH, int dh_fp32,
                                int64_t N, int64_t D, float eps, void *dX, float *dgamma,
                                void *ws, size_t ws_bytes, lce_stream_t stream);

/* RMSNorm + LM head + cross-entropy, forward and backward in one call: the
 * chunked path of lce_fwd_bwd_ex applied to H = RMSNorm(X), returning the
 * gradients of the pre-norm X and of gamma instead of dH. Per chunk the rows
 * are normalised into a buffer of one chunk's rows (of a pair's, when the chunks
 * go in pairs as on the loss path), the chunk's dH is kept in fp32 and fed to the
 * RMSNorm backward at once, so neither H nor dH exists for all N rows. Outputs:
 * loss and lse as for lce_fwd_bwd_ex (reduction MEAN / SUM / NONE), dX [N][D]
 * bf16, dgamma [D] fp32, dW [V][D] fp32 (overwritten). The workspace is
 * lce_norm_workspace_size(N, D, V, chunk) bytes: that of lce_workspace_size plus
 * the normalised rows (bf16), the chunk's fp32 dH where the loss path's
 * workspace holds none, and the dgamma partials. Device status as for
 * lce_fwd_bwd. */
lce_status lce_norm_workspace_size(int64_t N, int64_t D, int64_t V, int64_t chunk, size_t *bytes);
lce_status lce_norm_fwd_bwd(const void *X, const void *gamma, float eps, const void *W,
                            const int64_t *y, const float *dloss, int64_t N, int64_t D, int64_t V,
                            int64_t ignore_index, int64_t chunk, int reduction, float *loss,
                            float *lse, void *dX, float *dgamma, float *dW, void *ws,
                            size_t ws_bytes, lce_stream_t stream);
/* The same with option flags: LCE_FROZEN_W (a frozen LM head: dW is not
 * computed and may be NULL; dX and dgamma as above; one chunk buffer) and
 * LCE_LOW_MEMORY (one chunk buffer, one dW contraction per chunk). The workspace
 * is lce_norm_workspace_size_opt(..., flags) bytes; lce_norm_workspace_size and
 * lce_norm_fwd_bwd are these with flags = 0. Other flags: LCE_ERR_INVALID_ARG. */
lce_status lce_norm_workspace_size_opt(int64_t N, int64_t D, int64_t V, int64_t chunk, int flags,
                                       size_t *bytes);
lce_status lce_norm_fwd_bwd_opt(const void *X, const void *gamma, float eps, const void *W,
                                const int64_t *y, const float *dloss, int64_t N, int64_t D,
                                int64_t V, int64_t ignore_index, int64_t chunk, int reduction,
                                int flags, float *loss, float *lse, void *dX, float *dgamma,
                                float *dW, void *ws, size_t ws_bytes, lce_stream_t stream);

/* Synchronises `stream`, then returns the device-side status recorded in the
 * workspace by the last call that used it (LCE_OK, LCE_ERR_LABEL_RANGE or
 * LCE_ERR_TIMEOUT; a timeout wins over a label error) and clears it. Returns
 * LCE_ERR_CUDA if the stream reports an error. */
lce_status lce_read_status(const void *ws, lce_stream_t stream);

/* Self-test of the bounded waits (a library diagnostic; the pages have no
 * counterpart). Clears the first 1024 bytes of ws (a workspace header), then
 * runs one warp that waits, with the wait the pipelines use, on an mbarrier
 * nothing signals: after limit_us microseconds (1 .. 2000000) the wait gives up,
 * records the timeout in the header and the kernel returns.
 * lce_read_status(ws) then returns LCE_ERR_TIMEOUT and the stream stays usable. */
lce_status lce_selftest_wait_timeout(void *ws, size_t ws_bytes, int64_t limit_us,
                                     lce_stream_t stream);

/* Static string for a status code. */
const char *lce_status_string(lce_status s);

/* Library version as 10000*major + 100*minor + patch. */
int lce_version(void);

/* Number of kernel launches the last lce_* call on this host thread enqueued. */
int lce_last_launch_count(void);

/* Optional per-kernel timing for profiling (off by default). When enabled, every
 * kernel launch of the calls above is bracketed by two CUDA events recorded on
 * the call's stream. lce_profile_read() waits for the recorded events, adds the
 * elapsed times of every completed launch of one kernel kind to its running
 * totals and returns them; lce_profile_reset() clears the totals. Host-side
 * state only (the events are created by the library on the current device).
 * Kinds: */
enum {
    LCE_KERNEL_LOGITS = 0,   /* chunk logits GEMM with the log-sum-exp / G epilogue */
    LCE_KERNEL_GRAD = 1,     /* dH + dW gradient GEMM tiles */
    LCE_KERNEL_MERGE = 2,    /* slab merge (lse, row loss), G rescale, H-chunk transpose */
    LCE_KERNEL_OTHER = 3,    /* label scan, loss finalisation, dH combination */
    LCE_KERNEL_NORM = 4,     /* RMSNorm forward / backward row kernels, dgamma reduction */
    LCE_KERNEL_PHASE = 5,    /* the second chunk of a pair (two chunk buffers): its dH tiles
                                beside one dW contraction over both chunks of the pair */
    LCE_KERNEL_DH = 6,       /* the first chunk of a pair: its dH tiles, with the second
                                chunk's logits tiles on the CTA pairs they leave free */
    LCE_KERNEL_KINDS = 7
};
lce_status lce_profile_enable(int on);
lce_status lce_profile_read(int kind, double *total_ms, int64_t *launches);
void lce_profile_reset(void);

/* lce_forward for callers that cannot allocate device memory. The pages have no
 * counterpart: this is a library convenience. Some callers have no allocator to
 * hand (a plugin inside another runtime that owns all device memory), may not
 * call cudaMalloc on their hot path (it synchronises the device), or run with a
 * device-memory budget fixed at start-up; they cannot provide a workspace.
 * This call takes the same arguments as lce_forward minus the workspace and
 * uses a 64 MiB array built into the library instead (held on every GPU that
 * loads the library until the process exits). It allocates nothing.
 *  - Sizes whose lce_forward_workspace_size() exceeds 64 MiB return
 *    LCE_ERR_WORKSPACE before anything is enqueued; a smaller chunk may fit
 *    (the Llama-3-sized head, N = 16384, V = 128256, needs ~8.3 MB at chunk 1024).
 *  - Every call looks up the array's address on the current device (one
 *    cudaGetSymbolAddress, a host-side lookup), so a device reset leaves no
 *    stale address behind. The first lookup on a device may load the library's
 *    device code: make the first call before any stream capture.
 *  - Every call shares the array, which keeps the last call's contents; each
 *    call clears what must start at zero on its stream. Calls that overlap on
 *    the GPU race on the array: order them on one stream.
 *  - Device-side status (labels out of range, a bounded wait that ran out) is
 *    recorded in the shared array: lce_noalloc_read_status(stream) synchronises
 *    the stream and returns (and clears) it, as lce_read_status does for a
 *    workspace. Read it before the next call on the device overwrites it. */
lce_status lce_forward_noalloc(const void *H, const void *W, const int64_t *y,
                               int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                               int64_t chunk, float *loss, float *lse, lce_stream_t stream);
lce_status lce_noalloc_read_status(lce_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LCE_GB300_H */
