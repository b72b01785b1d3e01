/*
 * swin_wattn: fused Swin window / shifted-window multi-head attention (W-MSA / SW-MSA)
 * on one NVIDIA GB300 GPU (sm_103a). C ABI; every call is asynchronous on the stream
 * it is given and reports failure only through its return code.
 *
 * What is computed (sources cited by page and section):
 *  - NVIDIA "visual large-model training and inference optimisation" talk, full
 *    transcript (uticex.com, article 1598), section 1: attention among the tokens of each
 *    non-overlapping M x M window, a cyclic window shift that bridges window borders, and
 *    a learned relative position bias added to the attention logits.
 *  - same transcript, section 2: shift, window partition and window reverse are index
 *    mappings only; the mask and the bias reach the fused attention as tensors.
 *  - same transcript, section 3: the relative-position bias lookup runs once, as
 *    preprocessing, producing a dense per-head bias; batch GEMM + softmax + batch GEMM
 *    run as one fused kernel whose loads and stores absorb the layout transposes.
 *  - Baidu AIAK-Training talk (jxzklqfsx.com, article 743345), section 2, the fused
 *    WindowAttention case: one kernel staging HBM -> shared memory -> registers, tensor
 *    cores for both products, and a backward that recomputes instead of reloading.
 *
 * For an activation qkv of shape [B, H, W, 3C] (channel t*C + h*hd + d, t in {q,k,v},
 * head h < nH, hd = C/nH = 32), window size M and shift s (0 <= s < M):
 *   rolled token (y, x) reads original token ((y+s) mod H, (x+s) mod W);
 *   windows are row-major over (H/M, W/M), tokens row-major inside a window;
 *   logit(i,j) = hd^-0.5 * q_i.k_j + table[idx(i,j), h] + mask_w(i,j), with
 *   idx(i,j) = (yi-yj+M-1)*(2M-1) + (xi-xj+M-1) for local window positions,
 *   mask_w(i,j) = -100 when the two tokens carry different shift-region labels
 *   (per axis of length L on the rolled grid: [0,L-M), [L-M,L-s), [L-s,L); label =
 *   3*region_y + region_x), else 0; no mask when s = 0;
 *   P = row softmax of the logits, O = P V, written to channel h*hd + d of the same
 *   token position it was read from: out has shape [B, H, W, C].
 *
 * Conventions for every entry point:
 *  - Tensor pointers are device pointers (cudaMalloc, or torch CUDA tensors), contiguous
 *    in the layouts above, 16-byte aligned, owned by the caller. A host pointer is
 *    rejected with SWIN_WATTN_ERR_INVALID_ARG before any launch.
 *  - Activation dtype is fixed per plan: SWIN_WATTN_BF16 (bf16 in and out) or
 *    SWIN_WATTN_FP32 (fp32 in and out; values are rounded to bf16, round-to-nearest-
 *    even, on load). Arithmetic: bf16 tensor-core products with fp32 accumulation,
 *    fp32 softmax.
 *  - The bias table is fp32 [(2M-1)^2, nH], row-major; its gradient likewise.
 *  - Errors come back as status codes; nothing aborts, traps or throws across the ABI.
 *    After SWIN_WATTN_ERR_CUDA, swin_wattn_last_error() holds the CUDA error text of the
 *    calling thread.
 */
#ifndef SWIN_WATTN_H
#define SWIN_WATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

typedef struct swin_wattn_plan_s* swin_wattn_plan_t;

enum swin_wattn_status {
  SWIN_WATTN_OK = 0,
  SWIN_WATTN_ERR_INVALID_ARG = 1,  /* null/host pointer, bad dtype, s out of range, ... */
  SWIN_WATTN_ERR_UNSUPPORTED = 2,  /* M not in {4,7,12}, head width != 32, H%M or W%M != 0 */
  SWIN_WATTN_ERR_MISALIGNED = 3,   /* tensor pointer not 16-byte aligned (table: 4-byte) */
  SWIN_WATTN_ERR_BAD_PLAN = 4,     /* null, destroyed or foreign plan handle */
  SWIN_WATTN_ERR_CUDA = 5,         /* a CUDA runtime call failed; see swin_wattn_last_error */
  SWIN_WATTN_ERR_TIMEOUT = 6       /* a bounded device-side wait ran out (see
                                      swin_wattn_device_status) */
};

enum swin_wattn_dtype { SWIN_WATTN_BF16 = 0, SWIN_WATTN_FP32 = 1 };

/* Forward and backward kernels (swin_wattn_set_fwd_kernel, swin_wattn_set_bwd_kernel). */
enum swin_wattn_kernel {
  SWIN_WATTN_KERNEL_AUTO = 0,      /* the faster kernel as measured (see the setters below) */
  SWIN_WATTN_KERNEL_MMA_SYNC = 1,  /* warp-level mma.sync kernel: every M, both dtypes */
  SWIN_WATTN_KERNEL_TCGEN05 = 2    /* tensor-memory kernels: M = 7 or 12 with bf16 */
};

/*
 * Create a plan for one layer shape and run the preprocessing on `stream`:
 * the dense bias [nH, M^2, M^2] is expanded from `bias_table` (the lookup done once, as
 * in section 3 of the NVIDIA transcript) and, for s > 0, the shift mask [nW, M^2, M^2]
 * (nW = (H/M)(W/M), values 0 / -100) is built.
 *   out         receives the plan handle (set to NULL on failure).
 *   B           batch (B = 0 is allowed: every call on the plan is then a no-op,
 *               except that swin_wattn_bwd still zeroes dtable).
 *   H, W        token grid; multiples of M.
 *   C           channels per q/k/v; C = 32 * num_heads.
 *   window      M in {4, 7, 12}.  shift: s in [0, M).
 *   dtype       SWIN_WATTN_BF16 or SWIN_WATTN_FP32 activation I/O.
 *   bias_table  device fp32 [(2M-1)^2, num_heads]; read during this call's launch only.
 * The plan owns its dense bias, its mask and the backward's reduction scratch (device
 * memory allocated here, freed by swin_wattn_destroy). A plan is used by one stream at a
 * time; swin_wattn_fwd and swin_wattn_bwd allocate nothing.
 */
int swin_wattn_plan(swin_wattn_plan_t* out, int B, int H, int W, int C, int num_heads,
                    int window, int shift, int dtype, const float* bias_table,
                    struct CUstream_st* stream);

/* Re-expand the dense bias from an updated table (training). Same table layout. */
int swin_wattn_set_bias(swin_wattn_plan_t plan, const float* bias_table,
                        struct CUstream_st* stream);

/*
 * Forward: qkv [B,H,W,3C] -> out [B,H,W,C] (plan dtype). One kernel launch: the roll and
 * window partition are folded into the load addressing and the reverse and un-roll into
 * the store; logits, bias, mask and softmax stay on chip. `out` must not overlap `qkv`.
 */
int swin_wattn_fwd(swin_wattn_plan_t plan, const void* qkv, void* out,
                   struct CUstream_st* stream);

/*
 * Forward on host-resident activations, for callers whose data lives in host memory:
 * copies qkv_host [B,H,W,3C] into the caller-owned device buffer dev_qkv, runs the same
 * kernel as swin_wattn_fwd into dev_out, and copies dev_out back to out_host [B,H,W,C].
 * The batch is cut into up to four chunks that flow through a copy-in queue, `stream`
 * (the kernels) and a copy-out queue, so both copy directions and the compute overlap;
 * `stream` waits for the last copy-out, so the whole call is ordered on `stream`
 * (synchronise it before reading out_host). The two copy queues and their events are
 * created by the plan's first call. Host buffers should be page-locked (cudaHostAlloc,
 * or torch pin_memory) for the copies to be asynchronous. dev_qkv and dev_out must be
 * device pointers (16-byte aligned).
 */
int swin_wattn_fwd_host(swin_wattn_plan_t plan, const void* qkv_host, void* out_host,
                        void* dev_qkv, void* dev_out, struct CUstream_st* stream);

/*
 * Backward for an upstream gradient dout [B,H,W,C] (plan dtype):
 *   dqkv   [B,H,W,3C] plan dtype, fully overwritten (dq, dk, dv at the channels the
 *          forward read q, k, v from);
 *   dtable [(2M-1)^2, nH] fp32, overwritten (not accumulated) with the bias-table
 *          gradient summed over every batch, window and (i, j) pair.
 * The forward's probabilities are recomputed, not stored (AIAK-Training talk,
 * section 2). Deterministic: the same inputs give bit-identical outputs.
 */
int swin_wattn_bwd(swin_wattn_plan_t plan, const void* qkv, const void* dout, void* dqkv,
                   float* dtable, struct CUstream_st* stream);

/*
 * Backward without any device allocation (the pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory when they run the
 * backward, e.g. runtimes that fix their device memory plan at start-up and forbid any
 * later cudaMalloc, or frameworks whose own allocator must own every device byte; such
 * callers cannot create a plan, because a plan allocates).
 *
 * Same arguments and results as swin_wattn_plan followed by swin_wattn_bwd with the
 * MMA_SYNC backward kernel (qkv, dout, dqkv, dtable and the bias table are the caller's
 * device buffers; window must be 4 or 7), but no plan is made and nothing is allocated or
 * freed: the working memory (bias
 * fragments, mask bits, per-CTA table-gradient partials) lives in one fixed 2 MiB
 * device array inside the library, which every GPU that loads the library holds until
 * the process exits. A shape whose working memory exceeds 2 MiB is refused with
 * SWIN_WATTN_ERR_UNSUPPORTED and the reason in swin_wattn_last_error().
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture. The address
 * is kept for the life of the process, so do not call this entry point on a device after
 * a cudaDeviceReset of that device (the reset unloads the array it points into). Every
 * call on a device shares the one array and rewrites the parts it reads before reading
 * them, so two calls that overlap on the GPU (different streams without ordering between
 * them) race: order them. Three kernel launches on `stream` (fragments, backward,
 * table-gradient sum), counted by swin_wattn_launch_count.
 */
int swin_wattn_bwd_noalloc(const void* qkv, const void* dout, void* dqkv, float* dtable,
                           const float* bias_table, int B, int H, int W, int C, int num_heads,
                           int window, int shift, int dtype, struct CUstream_st* stream);

/*
 * Debug dumps of the plan's index maps and preprocessed tensors (device pointers, any
 * may be NULL to skip):
 *   gather     int32 [nW, M^2]: original token index y*W + x that window w, slot i
 *              reads (and writes), computed by the same addressing as the kernels;
 *   relidx     int32 [M^2, M^2]: relative position index idx(i, j);
 *   mask       fp32 [nW, M^2, M^2]: the plan's shift mask (all zeros when s = 0);
 *   dense_bias fp32 [nH, M^2, M^2]: the plan's expanded bias.
 */
int swin_wattn_debug_maps(swin_wattn_plan_t plan, int32_t* gather, int32_t* relidx,
                          float* mask, float* dense_bias, struct CUstream_st* stream);

/*
 * The producer step in front of the attention (NVIDIA talk, section 2, lists LayerNorm and
 * the qkv GEMM among the operations fused around the window attention): for each of
 * `tokens` tokens,
 *   xn = (x - mean) / sqrt(var + eps) * gamma + beta   (mean, population variance over C)
 *   qkv = xn W^T + b
 *   x      bf16 [tokens, C] (e.g. a [B,H,W,C] activation), device, 16-byte aligned;
 *   gamma, beta fp32 [C]; b fp32 [3C]; device;
 *   w_qkv  bf16 [3C, C] (row n = output channel n, in the order q | k | v, head-major);
 *   qkv    bf16 [tokens, 3C], device, 16-byte aligned, written (the attention's input);
 *   workspace  caller-owned device memory of at least swin_wattn_qkv_workspace_bytes(C,
 *          tokens) bytes, 256-byte aligned, overwritten (the gamma-folded weights, two
 *          per-channel vectors and the per-token statistics); one call at a time per
 *          workspace;
 *   status optional device int (may be NULL): bit 0 is OR-ed in if a bounded device wait
 *          ran out (then qkv is not valid).
 * The normalisation is applied on the other side of the product:
 *   xn W^T + b = rstd (x W'^T) - rstd mean u + v,  W' = bf16(gamma * W) (per input channel),
 *   u = row sums of W', v = beta W^T + b,
 * with the row statistics in fp32 and the product accumulated in fp32 on bf16 x and W';
 * qkv is rounded to bf16. C must be a multiple of 32 in [32, 1536]. The cyclic shift and
 * window partition are not applied here: the attention folds them into its loads. Two
 * kernel launches on `stream` (the weight fold, with the token statistics when the product
 * does not sum them itself; the product); nothing is allocated.
 * swin_wattn_qkv_workspace_bytes returns 0 for an unsupported C.
 */
size_t swin_wattn_qkv_workspace_bytes(int C, int tokens);
int swin_wattn_qkv_proj(const void* x, const float* gamma, const float* beta, const void* w_qkv,
                        const float* b_qkv, void* qkv, int tokens, int C, float eps, void* workspace,
                        size_t workspace_bytes, int* status, struct CUstream_st* stream);

/*
 * The producer step with its weights prepared once (NVIDIA Swin talk, section 3: inference
 * may transform the qkv weight and bias ahead of time). swin_wattn_qkv_prepare writes W',
 * u and v (as above) for gamma, beta, w_qkv, b_qkv into `prepared` (device, 256-byte
 * aligned, at least swin_wattn_qkv_prepared_bytes(C) bytes; one launch). Then each
 * swin_wattn_qkv_proj_prepared call computes qkv for x from them, with the same arithmetic
 * and results as swin_wattn_qkv_proj; it reads `prepared` and uses `stats_workspace`
 * (device, 16-byte aligned, at least swin_wattn_qkv_stats_bytes(tokens) bytes,
 * overwritten; one call at a time per workspace) for the per-token statistics. One or two
 * launches (the statistics pass where the product does not sum them itself; the product).
 * Errors as for swin_wattn_qkv_proj. The size queries return 0 for unsupported arguments.
 */
size_t swin_wattn_qkv_prepared_bytes(int C);
size_t swin_wattn_qkv_stats_bytes(int tokens);
int swin_wattn_qkv_prepare(const float* gamma, const float* beta, const void* w_qkv, const float* b_qkv, int C,
                           void* prepared, size_t prepared_bytes, struct CUstream_st* stream);
int swin_wattn_qkv_proj_prepared(const void* x, const void* prepared, void* qkv, int tokens, int C, float eps,
                                 void* stats_workspace, size_t stats_bytes, int* status,
                                 struct CUstream_st* stream);

/*
 * The producer step on prepared weights with OCP FP8 E4M3 output, the input of
 * swin_wattn_fwd_fp8 (NVIDIA Swin talk, section 3: the inference path takes its GEMMs to 8
 * bits with scales calibrated ahead of time; here the qkv the attention reads): the same
 * qkv as swin_wattn_qkv_proj_prepared, in fp32, then for each channel of tensor t (q, k, v)
 *   qkv8 = E4M3(qkv / scale_t), rounded to nearest even, saturated to +-448;
 *   qkv8   device, 16-byte aligned: [tokens, 3C] bytes, written (the token layout of qkv);
 *   scale_q, scale_k, scale_v  one fp32 scale per tensor, finite and positive (static
 *          scaling: e.g. the calibrated max |qkv_t| / 448);
 *   amax   optional device float[3] (may be NULL): max |qkv_t| of this call's fp32 values is
 *          max-ed into amax[t] atomically (the caller zeroes it; a later call can take its
 *          scales from it: delayed scaling).
 * Other arguments and errors as for swin_wattn_qkv_proj_prepared (INVALID_ARG also for a bad
 * scale). One or two launches; nothing is allocated.
 */
int swin_wattn_qkv_proj_prepared_fp8(const void* x, const void* prepared, void* qkv8, int tokens, int C, float eps,
                                     float scale_q, float scale_k, float scale_v, float* amax, void* stats_workspace,
                                     size_t stats_bytes, int* status, struct CUstream_st* stream);

/*
 * The consumer step after the attention: the output projection, then its bias and the
 * residual added, fused into the product's epilogue (NVIDIA Swin talk, uticex.com article
 * 1598, section 3 "inference optimisation": the bias-plus-residual pass in its half2
 * example):
 *   y[t] = residual[t] + o[t] Wp^T + bp   for each token t < tokens.
 * Arguments (device pointers unless stated):
 *   o        bf16 [tokens, C], 16-byte aligned: the attention output (swin_wattn_fwd's
 *            out, channel order h*32 + d);
 *   w_proj   bf16 [C, C] (row n = output channel n);
 *   b_proj   fp32 [C];
 *   residual bf16 [tokens, C], 16-byte aligned: the block input (the shortcut);
 *   y        bf16 [tokens, C], 16-byte aligned, written. y may be the residual buffer
 *            itself (each element is read before it is written) but must not overlap o;
 *   status   optional device int (may be NULL): bit 0 is OR-ed in if a bounded device
 *            wait ran out (then y is not valid).
 * The product is accumulated in fp32 on the bf16 operands, bp and the residual are added
 * in fp32, and y is rounded to bf16. C must be a multiple of 32 in [32, 1536]. One kernel
 * launch on `stream`; nothing is allocated. Errors: INVALID_ARG for negative tokens,
 * overlapping o and y, or a pointer that is not device memory; MISALIGNED for a pointer
 * off its alignment; UNSUPPORTED for C.
 */
int swin_wattn_proj_residual(const void* o, const void* w_proj, const float* b_proj, const void* residual,
                             void* y, int tokens, int C, int* status, struct CUstream_st* stream);

/*
 * Forward on 8-bit operands (7x7 windows, a SWIN_WATTN_BF16 plan): the attention of
 * q = scale_q * q8, k = scale_k * k8, v = scale_v * v8 for
 *   qkv8   device, 16-byte aligned: [B,H,W,3C] OCP FP8 E4M3 values, one byte each, in the
 *          token layout of qkv (q | k | v channels of a token);
 *   scale_q, scale_k, scale_v  one fp32 scale per tensor, finite and positive;
 *   out    device, 16-byte aligned: [B,H,W,C] bf16, written.
 * q8 k8^T runs on the 8-bit tensor cores (exact products, fp32 accumulation), the bias and
 * the shift mask are those of the plan, P is rounded to fp16, and v8 is widened exactly to
 * fp16 for P V: the result is the attention of the decoded values to the tolerance of
 * swin_wattn_fwd, with 3C instead of 6C bytes of qkv read per token (the pages take the
 * Swin GEMMs to 8 bits for inference, NVIDIA Swin talk section 3; here the attention's
 * operands). One kernel launch. UNSUPPORTED for another window size or dtype,
 * INVALID_ARG for a bad scale, and the pointer errors of swin_wattn_fwd.
 */
int swin_wattn_fwd_fp8(swin_wattn_plan_t plan, const void* qkv8, float scale_q, float scale_k, float scale_v,
                       void* out, struct CUstream_st* stream);

/*
 * Choose the plan's forward kernel (SWIN_WATTN_KERNEL_*): MMA_SYNC (every window size and
 * dtype) or TCGEN05 (the tensor-memory kernels: window 7 or 12, bf16). Both compute the
 * same function to the same tolerance. AUTO, the default, takes the faster as measured:
 * TCGEN05 for 12 x 12 windows when the plan has at least 16 window-heads per SM
 * (B * windows * heads >= 16 * SMs), else MMA_SYNC. Asking for TCGEN05 where it does not
 * apply returns SWIN_WATTN_ERR_UNSUPPORTED and leaves the plan unchanged. Host-side only;
 * call it between launches.
 */
int swin_wattn_set_fwd_kernel(swin_wattn_plan_t plan, int kernel);

/* The forward kernel the plan launches (MMA_SYNC or TCGEN05), or -1 for a bad handle. */
int swin_wattn_fwd_kernel(swin_wattn_plan_t plan);

/*
 * Choose the plan's backward kernel (SWIN_WATTN_KERNEL_*): MMA_SYNC (window 4 or 7, both
 * dtypes) or TCGEN05 (the tensor-memory kernel: window 7, bf16). Both compute the same
 * gradients to the same tolerance and are deterministic. AUTO, the default, takes the
 * faster as measured: TCGEN05 where it applies, except at shifted layers whose window grid
 * is at most two windows wide (there half or more of the windows wrap at the right edge
 * and are gathered four rows at a time), else MMA_SYNC. UNSUPPORTED where the choice does
 * not apply (the plan is then unchanged). Host-side only; call it between launches.
 */
int swin_wattn_set_bwd_kernel(swin_wattn_plan_t plan, int kernel);

/* The backward kernel the plan launches (MMA_SYNC or TCGEN05), or -1 for a bad handle. */
int swin_wattn_bwd_kernel(swin_wattn_plan_t plan);

/*
 * Synchronise `stream` and report the plan's device error word: SWIN_WATTN_ERR_TIMEOUT
 * if a kernel's bounded wait on the tensor core (1 s) ran out since the last call, in
 * which case that launch's output is not valid; the word is cleared. Otherwise OK.
 */
int swin_wattn_device_status(swin_wattn_plan_t plan, struct CUstream_st* stream);

/* Free the plan's device memory (synchronises the device first). NULL is a no-op. */
int swin_wattn_destroy(swin_wattn_plan_t plan);

/* Static text for a status code. */
const char* swin_wattn_status_string(int status);

/* CUDA error text behind the calling thread's last SWIN_WATTN_ERR_CUDA ("" if none). */
const char* swin_wattn_last_error(void);

/* Kernel launches issued by the calling thread since the last reset (for accounting). */
uint64_t swin_wattn_launch_count(int reset);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_WATTN_H */
