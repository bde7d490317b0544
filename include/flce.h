/*
 * flce.h -- fused LM-head projection + cross-entropy on one GB300 (sm_103a).
 *
 * The library computes, for hidden rows H [N,D], LM-head weight W [V,D] and
 * targets y [N] (ignore_index marks rows that do not count):
 *
 *   z_n    = H_n W^T                                   (never stored)
 *   LSE_n  = log sum_v exp(z_nv)
 *   loss   = sum_{valid n} (LSE_n - z_{n,y_n}) / max(count, 1)
 *   dZ     = grad_loss / max(count, 1) * valid * (softmax(z) - onehot(y))   (never stored whole)
 *   dH     = dZ W,   dW = dZ^T H
 *
 * The loss and its gradient are the ones stated in the Trillion Labs note on
 * Fused Linear Cross-Entropy ("Cross Entropy를 다시 보면": loss = -z(y) +
 * log sum exp z, dL/dz = softmax(z) - 1[j = y]) and in the PyTorch 2.13
 * LinearCrossEntropyLoss chapter ("먼저 수식에서 없앨 수 있는 tensor를 찾는다":
 * dZ = softmax(Z) - one_hot(target), dH = dZ W, dW = dZ^T H). The mean runs
 * over non-ignored rows with the count clamped to one (the note's chunked
 * cross-entropy listing). The forward is the blockwise linear-log-sum-exp of
 * "Cut Your Losses in Large-Vocabulary Language Models" (Sec. 4.2, Alg. 2)
 * with the target logit gathered as in its indexed matmul (Sec. 4.1, Alg. 1);
 * the backward recomputes logit tiles and forms softmax = exp(z - LSE) without
 * renormalising (Sec. 4.3, Alg. 3 and 4). The full [N,V] logits and dlogits
 * are never allocated.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, owned
 *    by the caller. The library never allocates or frees device memory.
 *  - H and W are bf16 (IEEE bfloat16 bit patterns, 2 bytes each), 16-byte
 *    aligned, with D a multiple of 8 (row pitch of 16 bytes for TMA).
 *  - Outputs lse, loss, dH, dW are fp32. dH and dW must be 16-byte aligned.
 *  - ws is a caller-owned device workspace of at least
 *    flce_workspace_bytes(p) bytes, 256-byte aligned. It holds the status
 *    word, per-tile LSE partials, the per-row LSE when the caller passes no
 *    lse buffer, and two bf16 staging buffers for bounded chunks of dZ
 *    (at most 8192 x 10240 each). Its size grows with N + V, never with
 *    N * V (the vocabulary-sorting and ignored-row-compaction flags below add
 *    a copy of W and of the valid rows; problems of more than 8192 rows also
 *    hold one vocabulary chunk's fp32 dW for flce_forward_backward_adamw). The forward-only calls need only
 *    flce_forward_workspace_bytes(p) bytes of it.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising. Errors found on the
 *    host are returned before anything is launched. Errors found by the GPU
 *    (a target outside [0,V) that is not ignore_index, a wait that ran out)
 *    are recorded in the workspace's status word: such rows are treated as
 *    ignored so all outputs stay finite, and flce_get_device_status reports
 *    the error.
 *  - Results are deterministic: the same inputs give bit-identical outputs.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, bad flag or threshold */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 2,/* ws_bytes < flce_workspace_bytes(p) */
  FLCE_ERR_BAD_TARGET = 3,         /* (device) a target outside [0,V) that is not ignore_index */
  FLCE_ERR_UNSUPPORTED = 4,        /* shape or alignment the kernels do not take (D % 8, 16-B alignment) */
  FLCE_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
  FLCE_ERR_TIMEOUT = 6             /* (device) a bounded wait inside a kernel ran out */
} flce_status;

/* Problem description. Tile and chunk sizes are chosen by the library. */
typedef struct {
  int64_t n_rows;        /* N: token rows (>= 0)                           */
  int64_t hidden;        /* D: hidden size (>= 8, multiple of 8)           */
  int64_t vocab;         /* V: vocabulary size (>= 1, < 2^31)              */
  int64_t ignore_index;  /* rows whose target equals this are ignored (-100) */
  float filter_eps;      /* gradient filter threshold; 0 = off (default).
                            With eps > 0, a 128-row x 256-column tile of the
                            unscaled gradient softmax - onehot whose entries
                            are all below eps in magnitude is left out of dW,
                            and a 256-row x 256-column block whose entries
                            are all below eps is left out of dH (Cut
                            Cross-Entropy, Sec. 4.3 "Gradient filtering" and
                            Alg. 4; the paper uses 2^-12).                   */
  uint32_t flags;        /* 0, or FLCE_FLAG_* bits below                   */
} flce_problem;

/* Test hook: every bounded wait inside the GEMM kernels gives up after about
 * a microsecond, so the timeout path runs and FLCE_ERR_TIMEOUT is recorded.
 * Outputs are then undefined, except that a forward whose GEMM gave up
 * writes NaN as its loss (mean and sum reductions). */
#define FLCE_FLAG_TEST_SHORT_WAITS 0x1u

/* With filter_eps > 0: apply the filter to one gradient only, as the
 * "CCE-FullC" and "CCE-FullE" variants of Cut Cross-Entropy (Table 1, and
 * Sec. 5.3 on pretraining) do. FULL_DW computes dW (the classifier gradient)
 * without filtering and filters dH; FULL_DH does the opposite. */
#define FLCE_FLAG_FILTER_FULL_DW 0x2u
#define FLCE_FLAG_FILTER_FULL_DH 0x4u

/* Remove ignored rows before the backward, as Cut Cross-Entropy suggests
 * for masked data (App. B, "removing ignored tokens"). The forward still
 * computes the LSE of every row. The backward then runs on the valid rows
 * only: their H rows, targets and LSE are gathered into the workspace, and
 * dH is scattered back, with exact zeros on ignored rows. The launch sizes
 * depend on the valid count, so with this flag flce_forward_backward and
 * flce_backward_ex synchronise `stream` once to read it. The workspace
 * grows by about 6*N*D + 28*N bytes. */
#define FLCE_FLAG_COMPACT_IGNORED 0x8u

/* Vocabulary sorting of Cut Cross-Entropy (Sec. 4.3, "Vocabulary sorting"):
 * the backward visits the vocabulary in order of decreasing average logit,
 * so that ids of similar average share a 256-id block and the gradient
 * filter (filter_eps > 0) finds more blocks it can leave out.
 *   The average logit of id v is the mean of z_nv (+ b_v) over the
 *   non-ignored rows, 0 when no row is valid. It is formed as
 *   W_v . mean(H over valid rows) (+ b_v), the same value by linearity,
 *   in fp32; ids of equal average keep their id order.
 *   The backward runs on a copy of W with its rows in that order (kept in
 *   the workspace, which grows by at most V*D*2 + 29*V + 8*N + 1028*D bytes) and
 *   writes dW and d(bias) back to the caller's buffers in id order. With
 *   filtering off the results equal those of the unsorted backward up to
 *   fp32 summation order. The forward ignores the flag.
 *   flce_get_vocab_order reads back the order and the averages. */
#define FLCE_FLAG_SORT_VOCAB 0x10u

/* Bytes of device workspace every compute call below (flce_forward,
 * flce_forward_backward, flce_forward_ex, flce_backward_ex) needs for
 * problem *p (0 if p is NULL or invalid). Pure host arithmetic; needs no GPU. */
size_t flce_workspace_bytes(const flce_problem* p);

/* The smaller workspace the forward-only calls (flce_forward,
 * flce_forward_ex) accept: the status word, the LSE partials and the loss
 * sums, without the backward's staging chunks (about 40 MiB instead of
 * 357 MiB for N = 8192, V = 151552). A workspace of flce_workspace_bytes(p)
 * bytes serves every call. Pure host arithmetic. */
size_t flce_forward_workspace_bytes(const flce_problem* p);

/* Forward: per-row LSE (all rows, ignored ones included) and the mean loss.
 *   H    bf16 [N,D]   W bf16 [V,D]   y int64 [N]
 *   lse  fp32 [N] out (required)     loss fp32 [1] out
 * Follows "Cut Your Losses in Large-Vocabulary Language Models", Sec. 4.1-4.2
 * (Alg. 1 and 2), with the loss of the Trillion Labs note. */
flce_status flce_forward(const flce_problem* p, const void* H, const void* W, const int64_t* y, float* lse,
                         float* loss, void* ws, size_t ws_bytes, void* stream);

/* Forward and backward in one call, for an upstream gradient grad_loss of the
 * scalar loss (1 for a plain loss.backward()); gradients are computed in the
 * same call, as the PyTorch 2.13 chapter describes for scalar reductions
 * ("scalar reduction에서는 forward가 gradient까지 계산한다").
 *   lse  fp32 [N] out, or NULL (then kept in ws)   loss fp32 [1] out
 *   dH   fp32 [N,D] out (overwritten)              dW fp32 [V,D] out (overwritten)
 * Follows "Cut Your Losses in Large-Vocabulary Language Models", Sec. 4.3 and
 * Alg. 4, with gradient sign and mean of the Trillion Labs note. */
flce_status flce_forward_backward(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                  float grad_loss, float* lse, float* loss, float* dH, float* dW, void* ws,
                                  size_t ws_bytes, void* stream);

/* Data parallelism over rows: each process (one per GPU) holds its own rows
 * H, y and the whole W, and the ranks together take the mean over the valid
 * rows of ALL ranks. The pages name the exchange this needs: data
 * parallelism all-reduces the weight gradient (the FORGE explainer, on what
 * its fused update cannot cover), and the PyTorch 2.13 chapter lists
 * sharding the LM head across devices among its open items. One step:
 *   1. flce_count_valid on every rank, then a sum of the counts over the
 *      ranks (the caller's all-reduce, e.g. NCCL on the same stream);
 *   2. flce_forward_backward_global with that sum;
 *   3. a sum over the ranks of the loss and of dW (the caller's
 *      all-reduce); dH and lse stay per rank, since each rank owns its rows.
 *
 * flce_count_valid: *count (device int64) = the number of this rank's targets
 * in [0, V) that are not ignore_index (the rows a mean counts; bad targets
 * are not counted). Enqueued on `stream`; y and count 8-byte aligned.
 * FLCE_ERR_INVALID_ARGUMENT on a bad problem or pointer. */
flce_status flce_count_valid(const flce_problem* p, const int64_t* y, int64_t* count, void* stream);

/* flce_forward_backward with the mean taken over *count_global (device
 * int64, read on `stream` after the caller's all-reduce; the sum of every
 * rank's flce_count_valid) instead of this call's own count:
 *   loss = sum over this rank's valid rows of (LSE_n - z_{n,y_n}) / max(count_global, 1),
 *          this rank's share of the global mean (the shares sum to it);
 *   dH, dW = grad_loss / max(count_global, 1) * (the same sums as
 *          flce_forward_backward), so dW is this rank's contribution and the
 *          sum of dW over the ranks is the gradient of the global mean.
 * Every other argument, output and error is as in flce_forward_backward;
 * count_global must be 8-byte aligned. */
flce_status flce_forward_backward_global(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                         const int64_t* count_global, float grad_loss, float* lse, float* loss,
                                         float* dH, float* dW, void* ws, size_t ws_bytes, void* stream);

/* Reductions of the per-row losses for the general entry points below. */
#define FLCE_REDUCTION_MEAN 0 /* sum over valid rows / max(count, 1) */
#define FLCE_REDUCTION_SUM 1  /* sum over valid rows */
#define FLCE_REDUCTION_NONE 2 /* one loss per row, 0 on ignored rows */

/* General forward: optional bias and a choice of reduction, as in the
 * PyTorch 2.13 chapter's F.linear_cross_entropy(input, weight, target,
 * linear_bias, ignore_index, reduction). Logits are z = H W^T + bias.
 *   bias  fp32 [V] or NULL
 *   lse   fp32 [N] out (required; the backward below takes it)
 *   loss  fp32 out: [1] for MEAN and SUM, [N] for NONE
 * No gradient is computed; pair it with flce_backward_ex. */
flce_status flce_forward_ex(const flce_problem* p, int32_t reduction, const void* H, const void* W, const float* bias,
                            const int64_t* y, float* lse, float* loss, void* ws, size_t ws_bytes, void* stream);

/* General backward: recomputes the logits from H, W (and bias) and the LSE
 * of flce_forward_ex, and forms dZ = s_n * (softmax - onehot) with s_n from
 * the upstream gradient (Cut Cross-Entropy, Sec. 4.3 and Alg. 4, whose
 * gradient is scaled per row by the backpropagated gradient of the loss).
 *   grad   fp32 DEVICE pointer: [1] for MEAN (s_n = g / count) and SUM
 *          (s_n = g), [N] for NONE (s_n = grad[n])
 *   dH fp32 [N,D], dW fp32 [V,D] out (overwritten)
 *   dbias  fp32 [V] out (overwritten) or NULL; d(bias)_v = sum_n dZ_nv
 * With NONE, s_n multiplies G before it is rounded to bf16. */
flce_status flce_backward_ex(const flce_problem* p, int32_t reduction, const void* H, const void* W,
                             const float* bias, const int64_t* y, const float* lse, const float* grad, float* dH,
                             float* dW, float* dbias, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, returns the device status word of the most recent
 * call that used `ws` (FLCE_OK, FLCE_ERR_BAD_TARGET or FLCE_ERR_TIMEOUT; the
 * first in that order that is set wins, timeout over bad target) and clears it. */
flce_status flce_get_device_status(void* ws, void* stream);

/* Hyper-parameters of one AdamW step (decoupled weight decay, bias-corrected
 * moments, the form torch.optim.AdamW computes), read by the kernels from
 * device memory so that a captured CUDA graph picks up each step's values. */
typedef struct {
  float lr;
  float beta1;         /* in [0, 1) */
  float beta2;         /* in [0, 1) */
  float eps;           /* > 0 */
  float weight_decay;
  int32_t step;        /* t >= 1: the step being taken (bias corrections 1 - beta^t) */
} flce_adamw_hparams;

/* flce_forward_backward with W's AdamW update fused into its gradient, as
 * the FORGE explainer describes ("FORGE: Fused On-Register Gradient
 * Elimination for Memory-Efficient LLM Training", Sec. 2): each finished
 * dW tile, still in the tensor cores' accumulator, updates its rows of the
 * fp32 master weights and moments, writes their bf16 copy, and is dropped.
 * dW never reaches memory.
 *   w_master, adam_m, adam_v: device fp32 [V,D], read and updated in place.
 *   w_out: device bf16 [V,D], receives the updated weights rounded to
 *     nearest; it must not overlap W, which the same call still reads.
 *   hp: device pointer to this step's hyper-parameters. A step below 1, a
 *     beta outside [0, 1), eps <= 0 or a non-finite lr / weight_decay leave
 *     the master weights and moments unchanged and make
 *     flce_get_device_status report FLCE_ERR_INVALID_ARGUMENT.
 *   Other arguments and results as flce_forward_backward (dH, LSE, loss).
 *   With n_rows <= 8192 (one row chunk) each dW tile is complete after one
 *   contraction and is applied straight from the accumulator. With more rows
 *   the vocabulary chunks run one after another, each chunk's dW is summed
 *   over the row chunks in a Vc x D fp32 buffer of the workspace, and its
 *   AdamW step runs as soon as it is complete: no more than one chunk's
 *   gradient (at most 10240 x D) exists at a time. n_rows must be >= 1.
 *   The gradient of a tile is final only when the whole batch is in it: a
 *   data-parallel run that must all-reduce dW cannot use this entry point
 *   (the page says the same of FORGE). Combines with filtering, sorting and
 *   ignored-row compaction. Workspace: flce_workspace_bytes(p). */
flce_status flce_forward_backward_adamw(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                        float grad_loss, float* lse, float* loss, float* dH, float* w_master,
                                        float* adam_m, float* adam_v, void* w_out, const flce_adamw_hparams* hp,
                                        void* ws, size_t ws_bytes, void* stream);

/* One AdamW step on n elements outside the LM-head call: the two-phase
 * counterpart of flce_forward_backward_adamw (for example after
 * flce_forward_backward), with the same arithmetic as its fused epilogue,
 * so the two give the same bits for the same gradient. grad (fp32 [n], e.g. dW)
 * updates w_master, adam_m and adam_v (fp32 [n]) in place; w_out (bf16 [n],
 * may be NULL) receives the new weights rounded to nearest. hp is a device
 * pointer as above. ws is any workspace of this library (256-byte aligned,
 * at least 256 bytes): the step's constants and the status word go in its
 * header, so it must not be in use by another call on another stream.
 * grad, w_master, adam_m, adam_v 16-byte aligned and w_out 8-byte aligned,
 * else FLCE_ERR_UNSUPPORTED. */
flce_status flce_adamw_step(const flce_adamw_hparams* hp, const float* grad, float* w_master, float* adam_m,
                            float* adam_v, void* w_out, int64_t n, void* ws, void* stream);

/* Static, human-readable name of a status code. */
const char* flce_status_string(flce_status s);

/* Statistic of the most recent backward (flce_forward_backward or
 * flce_backward_ex) that used `ws` with filtering on: the fraction of 128x256
 * gradient tiles that were skipped. Synchronises `stream`. Reports 0 when
 * filtering was off. */
flce_status flce_get_filter_stats(void* ws, void* stream, double* skipped_fraction);

/* The vocabulary order of the most recent backward that ran problem *p with
 * FLCE_FLAG_SORT_VOCAB on workspace `ws`: order[i] (device int32 [V]) is
 * the id visited at position i, and avg_logit (device float [V], may be
 * NULL) the average logit of every id, in id order. Both are copied from
 * the workspace on `stream` (asynchronous, no synchronisation).
 * FLCE_ERR_INVALID_ARGUMENT if p is invalid, lacks the flag, or a pointer
 * is NULL or order is not 4-byte aligned. */
flce_status flce_get_vocab_order(const flce_problem* p, const void* ws, int32_t* order, float* avg_logit,
                                 void* stream);

/* flce_forward without a caller-provided workspace, for callers that cannot
 * allocate device memory at the point they need the loss: for example a
 * plugin of an inference or training engine whose execute step must not
 * allocate, or code that runs under a fixed memory budget set at start-up
 * and has no spare buffer to hand over. The paper has no counterpart of this
 * entry point; it exists for such callers.
 *   Same arguments and results as flce_forward, minus ws and ws_bytes.
 *   The scratch it uses is a 16 MiB array in device memory that the library
 *   declares statically: every GPU that loads the library holds it until the
 *   process exits. The call allocates and frees nothing.
 *   Rows are processed in chunks small enough for the scratch. A problem
 *   whose buffers do not fit even with 256-row chunks (roughly V above two
 *   million) returns FLCE_ERR_UNSUPPORTED before launching anything.
 *   The first call on a device (and the first after its context was reset)
 *   looks up the scratch's device address (a runtime API call); make that
 *   first call before any stream capture.
 *   All calls share the one array and it keeps the last call's contents; the
 *   call initialises everything it reads. Calls that overlap on the GPU (on
 *   different streams, or from different threads) race on the scratch and
 *   must be serialised by the caller.
 *   There is no workspace to query for device-detected conditions. A bad
 *   target is handled as in flce_forward (its row is ignored) and is not
 *   reported. A bounded wait inside the kernels that ran out (an error of
 *   the device, never expected) makes the loss NaN, as in every forward. */
flce_status flce_forward_static_scratch(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                        float* lse, float* loss, void* stream);

/* Launch timing for profiling. After flce_profile_set(events, kinds, cap),
 * every kernel the compute calls enqueue is bracketed by two CUDA events
 * taken from `events` (cudaEvent_t handles created by the caller with timing
 * enabled): launch i uses events[2i] and events[2i+1], and kinds[i] receives
 * its FLCE_KERNEL_* code. At most `cap` launches are recorded; later ones
 * run untimed. flce_profile_set(NULL, NULL, 0) switches recording off.
 * flce_profile_count returns how many launches were recorded since the last
 * flce_profile_set. The recording is process-wide and guarded by a mutex;
 * it adds two event records per launch on the launch stream. */
#define FLCE_KERNEL_GEMM_LSE 0
#define FLCE_KERNEL_GEMM_DZ 1
#define FLCE_KERNEL_GEMM_DW 2 /* dW alone (only with FLCE_BWD_GROUPING=0) */
#define FLCE_KERNEL_GEMM_DH 3 /* dH alone (only with FLCE_BWD_GROUPING=0) */
#define FLCE_KERNEL_PREP 4
#define FLCE_KERNEL_COMBINE 5
#define FLCE_KERNEL_FINALIZE 6
#define FLCE_KERNEL_FILTER_STATS 7
#define FLCE_KERNEL_GEMM_BWD 8 /* one launch: dW and dH of a chunk + dZ of the next chunk */
#define FLCE_KERNEL_DBIAS 9
#define FLCE_KERNEL_SET_SCALE 10
#define FLCE_KERNEL_VOCAB_KEYS 11   /* average logits: column sums of H, their mean, W . mean */
#define FLCE_KERNEL_VOCAB_SORT 12   /* stable radix sort of the averages, inverse order */
#define FLCE_KERNEL_VOCAB_GATHER 13 /* W, bias and targets rearranged in the sorted order */
#define FLCE_KERNEL_ADAMW_PREP 14   /* constants of an AdamW step */
#define FLCE_KERNEL_ADAMW_STEP 15   /* flce_adamw_step's elementwise update */
#define FLCE_KERNEL_COUNT 16        /* flce_count_valid */
flce_status flce_profile_set(void** events, int32_t* kinds, int32_t cap);
int32_t flce_profile_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
