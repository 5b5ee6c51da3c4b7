/*
 * flce.h — fused linear cross-entropy (FLCE) on one NVIDIA GB300 (sm_103a).
 *
 * Given final hidden states x (N x H), an LM-head weight W (V x H) and integer
 * targets t (N), the library returns the mean cross-entropy of the logits
 * z = x·Wᵀ over the tokens whose target is not ignore_index, together with
 * dx = d loss / d x and dW = d loss / d W. It never holds the N x V logits:
 * tokens are processed in chunks of C, and only one chunk's C x V logits
 * buffer exists at a time.
 *
 * The operation is the one the FLCE pages define:
 *   - "Fused Linear Cross-Entropy: LLM 학습 logits 메모리 병목 없애기"
 *     (42jerrykim.github.io), section "FLCE의 핵심 아이디어: logits을 오래 들고
 *     있지 않는다": per chunk, (1) project the chunk to C x V logits, (2) take
 *     the CE loss and overwrite the same buffer with softmax - one_hot,
 *     (3) dx_chunk = dlogits·W at once, (4) dW += dlogits_chunkᵀ·x_chunk;
 *     drop the chunk buffers and move on.
 *   - "Unsloth 심층 아키텍처 …" (techknowgenie.com), section "스트리밍 청크
 *     기반 Fast CrossEntropy 손실 커널": per-token loss -z_y + log sum_j exp z_j,
 *     gradient softmax(z) - 1(i = y), and the running max / sum-exp kept on
 *     chip while the vocabulary is swept in blocks.
 *   - "메모리 아끼면서 Cross Entropy Loss 계산하기 — 128K Context LLM 학습 실전
 *     가이드" (sigco.tistory.com), section "즉시 적용할 수 있는 팁": bf16 logits,
 *     fp32 loss accumulation.
 * The mean runs over n_valid = #{i : t_i != ignore_index} tokens (PyTorch's
 * cross_entropy(reduction="mean") semantics, which the FLCE page's listing
 * calls per chunk). If n_valid == 0 the loss, dx and dW are all zero.
 *
 * Conventions for every entry point below:
 *   - Status codes, never exceptions or aborts. On failure, flce_last_error()
 *     gives a one-line reason.
 *   - Device pointers are CUDA device addresses on the handle's device,
 *     contiguous row-major, 16-byte aligned. The checks (INVALID_ARG when
 *     they fail): bf16 x, W, dx, dW 16-byte aligned; fp32 ones 4-byte; t
 *     8-byte. Sizes cannot be checked against the buffers: the caller
 *     passes buffers of the stated shapes. Host pointers are ordinary host
 *     memory (page-locked memory makes the copies asynchronous).
 *   - "stream" is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. All device work of a call is ordered on that stream.
 *   - A handle is not thread-safe: one host thread drives it at a time.
 *   - The caller owns x, W, t, dx, dW. The library owns only its workspace
 *     and, for the host-buffer entry point, its input staging buffers.
 *   - Outputs are overwritten, never accumulated into.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FLCE_ABI_VERSION 5

typedef struct flce_handle_s* flce_handle_t;

typedef enum flce_status {
    FLCE_OK = 0,
    FLCE_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or layout */
    FLCE_ERR_UNSUPPORTED = 2,   /* device is not compute capability 10.3, or dtype */
    FLCE_ERR_BUDGET = 3,        /* workspace above the budget, or allocation failed */
    FLCE_ERR_BAD_TARGET = 4,    /* a target outside [0, V) that is not ignore_index */
    FLCE_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
    FLCE_ERR_CUDA = 6           /* a CUDA runtime or driver call failed */
} flce_status;

/* element type of x, W and dx; dW is always fp32, the loss always fp32 */
enum { FLCE_DTYPE_BF16 = 0, FLCE_DTYPE_FP32 = 1 };

/* How the dlogits of a chunk are formed (fp32 handles run SLABS as asked and
 * every other mode in place).
 *  INPLACE:   the logits GEMM stores bf16 logits; a second pass overwrites
 *             them with (softmax - onehot)/n_valid (the FLCE page's step 2).
 *  RECOMPUTE: the logits GEMM keeps only per-row statistics; a second GEMM
 *             recomputes each logits tile and writes dlogits directly.
 *  SLABS:     the logits GEMM keeps only per-row statistics; the backward
 *             then walks the vocabulary in slabs of flce_plan.vocab_slab
 *             columns: per slab a GEMM recomputes the slab's dlogits into a
 *             C x vocab_slab buffer (at most 256 MiB, sized from the HBM
 *             budget), which the dx GEMM (dx accumulated over the slabs in
 *             fp32, in slab order) and the dW GEMM (on a second stream)
 *             consume. The workspace no longer grows with V:
 *             O(C·(vocab_slab + H)) bytes against O(C·V) for the other two,
 *             for 8·N·H·V FLOPs instead of 6·N·H·V. The Unsloth page
 *             ("Unsloth 심층 아키텍처 …", section "스트리밍 청크 기반 Fast
 *             CrossEntropy 손실 커널") keeps the logits off HBM altogether
 *             and adds dx with atomics; here the dlogits tile lives in the
 *             slab buffer, since no SM holds a token block's whole dx row,
 *             and dx is reduced in a fixed order. On an fp32 handle the
 *             same walk runs on the CUDA-core kernels, dx accumulated in
 *             place.
 *  AUTO:      INPLACE, the fastest of the three on GB300 by measurement. */
enum { FLCE_DLOGITS_AUTO = 0, FLCE_DLOGITS_INPLACE = 1, FLCE_DLOGITS_RECOMPUTE = 2,
       FLCE_DLOGITS_SLABS = 3 };

/* Tile shape of the tcgen05 GEMMs (bf16 only).
 *  SINGLE: one CTA per 128 x 256 output tile (tcgen05 cta_group::1).
 *  PAIR:   a cluster of two CTAs on two SMs per 256 x 256 tile
 *          (tcgen05 cta_group::2): each CTA loads half of the B operand.
 *  WIDE:   CTA pairs on 256 x 512 tiles: per k-step two 256 x 256 MMAs share
 *          their A operand through the tensor core's collector buffer, so a
 *          CTA's shared memory moves 25% fewer bytes per FLOP. The 512
 *          accumulator columns fill TMEM: the next tile's MMAs wait until
 *          the epilogue has read the accumulator out (its stores may still
 *          run; the logits GEMM's epilogue frees the first half early, and
 *          the next tile's first-half MMAs start on it).
 *  AUTO:   WIDE (measured fastest on GB300 for the 16384-token,
 *          128256-vocabulary step: 31.6 ms, against 34.9 ms for PAIR and
 *          36.9 ms for SINGLE).
 * Value 3 names no tile shape: flce_create and flce_make_plan refuse it with
 * INVALID_ARG. */
enum { FLCE_CTA_AUTO = 0, FLCE_CTA_SINGLE = 1, FLCE_CTA_PAIR = 2, FLCE_CTA_WIDE = 4 };

typedef struct flce_config {
    int32_t dtype;               /* FLCE_DTYPE_*                                       */
    int32_t device;              /* CUDA device ordinal                                */
    uint64_t hbm_budget_bytes;   /* workspace budget for the chunk planner; 0 = 1.25 GiB*/
    int32_t dlogits_mode;        /* FLCE_DLOGITS_*                                     */
    int32_t timeout_ms;          /* limit of every device-side wait; 0 = 2000 ms       */
    int32_t cta_pair;            /* FLCE_CTA_*                                         */
    int32_t backward_launch;     /* FLCE_BACKWARD_*                                    */
} flce_config;

/* How the dx and dW GEMMs of a chunk are launched (CTA pairs only).
 *  SEPARATE:   one launch each (the dW GEMM on a second stream beside a dx
 *              launch that fills less than two waves of SM pairs).
 *  ONE_LAUNCH: one launch on one tile shape; its work units (dx first, then
 *              dW) are handed out dynamically, so the short dW units fill the
 *              time the long dx units leave idle at the end, and the dx
 *              reduction over V needs few or no splits.
 *  AUTO:       ONE_LAUNCH where the dW GEMM runs on wide tiles (measured on
 *              GB300: 29.6 against 30.8 ms for the 16384-token,
 *              128256-vocabulary step, 35.0 against 37.2 ms at V = 151936,
 *              0.33 against 0.34 ms for 2048 tokens at V = 32000), else
 *              SEPARATE (on 256 x 256 pair tiles one launch measured slower:
 *              5.92 against 5.56 ms per 4096-token chunk at V = 128256). */
enum { FLCE_BACKWARD_AUTO = 0, FLCE_BACKWARD_SEPARATE = 1, FLCE_BACKWARD_ONE_LAUNCH = 2 };

/* The chunk plan of one call (token-chunk scheduler). */
typedef struct flce_plan {
    int64_t chunk;               /* C, tokens per chunk                                */
    int64_t num_chunks;          /* ceil(N / C)                                        */
    int64_t vocab_tiles;         /* ceil(V / 256): log-sum-exp partials per token      */
    int64_t ldv;                 /* row stride, in elements, of the chunk logits buffer */
    int64_t dx_splits;           /* split of the V reduction of the dx GEMM (fp32
                                    partials summed in split order by the reduction) */
    uint64_t workspace_bytes;    /* device bytes one call needs                        */
    uint64_t logits_bytes;       /* of which the C x ldv logits / dlogits buffer       */
    int64_t tile_m;              /* rows of a GEMM output tile: 128 (one CTA) or 256 (CTA
                                    pair, normal or wide)                               */
    int64_t tile_n;              /* columns of the logits GEMM's output tile: 256, or 512
                                    (wide). A FLCE_CTA_AUTO bf16 handle picks wide
                                    (512) or pair (256) tiles per GEMM, in-place and
                                    recompute modes, by a time model of the two:
                                    pair tiles where the reduction per tile is short */
    int64_t vocab_slab;          /* SLABS: vocabulary columns per backward slab (the
                                    buffer is chunk x vocab_slab); other modes: V       */
    int64_t dlogits_mode;        /* the FLCE_DLOGITS_* mode the call runs (AUTO and,
                                    on fp32 handles, RECOMPUTE resolved to INPLACE)     */
    int64_t tile_n_dx;           /* columns of the dx GEMM's output tile (256 or 512)  */
    int64_t tile_n_dw;           /* columns of the dW GEMM's output tile (256 or 512)  */
    int64_t dw_beside_dx;        /* 1: the dW GEMM runs beside the dx GEMM on the
                                    handle's second stream (in-place and recompute
                                    modes on CTA pairs, when the dx launch fills less
                                    than two waves of SM pairs); 0: one after the other */
    int64_t backward_one_launch; /* 1: the dx and dW GEMMs of a chunk share one launch
                                    (FLCE_BACKWARD_ONE_LAUNCH on CTA pairs, in-place
                                    and recompute modes), on the dx GEMM's tile shape,
                                    so tile_n_dw == tile_n_dx; 0: separate launches */
} flce_plan;

/* Kernel kinds, for the per-kernel timing of flce_profile_read(). */
enum {
    FLCE_K_COUNT_VALID = 0,      /* n_valid and target range check                     */
    FLCE_K_GEMM_LOGITS = 1,      /* x_c·Wᵀ on tcgen05, online max/sum-exp epilogue     */
    FLCE_K_LSE_COMBINE = 2,      /* per-token log-sum-exp from the vocab-tile partials  */
    FLCE_K_DLOGITS = 3,          /* (softmax - onehot)/n_valid in place                */
    FLCE_K_GEMM_DLOGITS = 4,     /* recompute variant: x_c·Wᵀ with dlogits epilogue    */
    FLCE_K_GEMM_DX = 5,          /* dx_c = dlogits·W on tcgen05                        */
    FLCE_K_DX_REDUCE = 6,        /* sums the dx split partials into bf16 dx            */
    FLCE_K_GEMM_DW = 7,          /* dW (+)= dlogitsᵀ·x_c on tcgen05, fp32              */
    FLCE_K_LOSS_FINALIZE = 8,    /* fixed-order sum of token losses / n_valid (bf16
                                    calls run it in their last DX_REDUCE launch unless
                                    dW work on the second stream is still to join)    */
    FLCE_K_SIMT_GEMM = 9,        /* fp32 path: CUDA-core GEMMs                         */
    FLCE_K_SIMT_TILE_STATS = 10, /* fp32 path: per-vocab-tile max/sum-exp              */
    FLCE_K_GEMM_DX_DW = 11,      /* CTA pairs: the dx and dW GEMMs of a chunk in one launch */
    FLCE_K_DEVICE_RESULT = 12,   /* loss and n_valid into caller device memory (an
                                    empty batch; otherwise the loss reduction writes them) */
    FLCE_K_COMBINE_DLOGITS = 13, /* LSE_COMBINE and DLOGITS in one launch, one block per
                                    token row (in-place mode: bf16 chunk rows of at most
                                    262144 columns; fp32, with the statistics too)    */
    FLCE_K_H2D_COPY = 14,        /* not a kernel: the host-buffer entry points' copies of
                                    x, W and t into device memory, timed on the stream
                                    that runs them (the copy stream for flce_submit_host);
                                    `bytes` counts the bytes copied                   */
    FLCE_K_NUM_KINDS = 15
};

typedef struct flce_kernel_profile {
    int64_t launches;            /* launches of this kind since the last reset         */
    double total_ms;             /* summed device time, CUDA events on the call stream
                                    (on the side stream for the SLABS mode's dW GEMMs,
                                    which overlap the dx GEMMs)                        */
    double flops;                /* algorithmic FLOPs of those launches                */
    double bytes;                /* algorithmic HBM bytes of those launches            */
} flce_kernel_profile;

/* ABI version of the loaded library (FLCE_ABI_VERSION). Host only. */
int32_t flce_abi_version(void);

/* Human-readable name of a status code. Host only; never NULL. */
const char* flce_status_string(flce_status s);

/* Plan one call without touching a device (host only).
 * The token-chunk scheduler: C = chunk if chunk > 0 (clamped to N), else the
 * largest C whose workspace fits cfg->hbm_budget_bytes, rounded to a multiple
 * of 128 and then evened out over ceil(N / C) chunks. This replaces the
 * chunk-size rule the FLCE page quotes from Liger (section "실전에서
 * 마주치는 트레이드오프", item 1), which sizes chunk logits to about N·H
 * elements: on GB300 the dW GEMM's intensity grows with C, so the budget, not
 * N·H, sets C. num_sms (0 means 152) sets the SM pairs the planner's time
 * model fills: it picks each GEMM's tile shape, the dx split and whether the
 * dx and dW GEMMs share one launch (flce_plan.backward_one_launch).
 * Errors: INVALID_ARG for a NULL or negative argument, BUDGET if even one
 * 128-token chunk (or N, if smaller) does not fit the budget. */
flce_status flce_make_plan(const flce_config* cfg, int64_t N, int64_t H, int64_t V,
                           int64_t chunk, int32_t num_sms, flce_plan* out);

/* Create a handle on cfg->device. Checks that the device is compute
 * capability 10.3 (GB300) and returns UNSUPPORTED otherwise: there is no
 * other code path. Allocates nothing on the device yet. *out is NULL on error. */
flce_status flce_create(flce_handle_t* out, const flce_config* cfg);

/* Free everything the library allocated (workspace, staging) and the handle.
 * Waits for the handle's outstanding work first. NULL is ignored. */
void flce_destroy(flce_handle_t h);

/* Workspace bytes flce_forward_backward would need for this call on handle
 * h: the planned workspace of flce_make_plan with the handle's config and
 * its device's SM count. Host only. Returns 0 when the call cannot be planned
 * (NULL handle, bad size, budget too small); flce_last_error then says why. */
uint64_t flce_workspace_bytes(flce_handle_t h, int64_t N, int64_t H, int64_t V, int64_t chunk);

/* Give the handle caller-owned device memory as its workspace (at least
 * flce_plan.workspace_bytes for the calls that follow; NULL/0 returns to
 * library-allocated workspace). The memory must stay valid until the handle
 * is destroyed or another workspace is set. Errors: INVALID_ARG. */
flce_status flce_set_workspace(flce_handle_t h, void* dev_ptr, uint64_t bytes);

/* The fused forward + backward.
 *   x   device, N x H, dtype of the handle (bf16 or fp32), row-major
 *   W   device, V x H, same dtype, row-major
 *   t   device, N int64 targets; t_i == ignore_index skips token i
 *   ignore_index  usually -100
 *   chunk   tokens per chunk, 0 = planned from the HBM budget
 *   loss    host, receives the fp32 mean loss
 *   dx      device, N x H, same dtype as x, overwritten
 *   dW      device, V x H fp32, overwritten (not accumulated into)
 * Returns after the stream has drained (the loss is read back), so the
 * outputs are ready. Steps on the stream: count n_valid; per chunk the
 * tcgen05 logits GEMM with its log-sum-exp epilogue, the log-sum-exp combine,
 * dlogits, the dx GEMM and the dW GEMM; the loss reduction.
 * Layout rules: bf16 needs H % 8 == 0 (TMA row strides are multiples of 16
 * bytes); fp32 takes any H. N may be 0 (loss 0, dW zeroed).
 * Errors: INVALID_ARG, UNSUPPORTED, BUDGET (workspace), BAD_TARGET (outputs
 * then unspecified), TIMEOUT, CUDA. */
flce_status flce_forward_backward(flce_handle_t h, const void* x, const void* W,
                                  const int64_t* t, int64_t N, int64_t H, int64_t V,
                                  int64_t ignore_index, int64_t chunk, float* loss,
                                  void* dx, float* dW, void* stream);

/* The fused forward + backward with no host synchronisation, for streams
 * under CUDA graph capture and for pipelines that must not block. Arguments
 * as flce_forward_backward, except that the results go to DEVICE memory when
 * the stream gets there: loss_dev (one fp32) and n_valid_dev (one int32);
 * either may be NULL. The call returns once its work is enqueued. A
 * device-side error (a target out of range, a wait that ran out) makes
 * *loss_dev NaN and is kept until flce_async_status reads it. Under capture
 * the call must not allocate: run it once outside capture first (or give a
 * workspace with flce_set_workspace) and keep profiling off.
 * Errors: those found on the host before any launch, as
 * flce_forward_backward; device-side errors only through flce_async_status. */
flce_status flce_forward_backward_async(flce_handle_t h, const void* x, const void* W,
                                        const int64_t* t, int64_t N, int64_t H, int64_t V,
                                        int64_t ignore_index, int64_t chunk, float* loss_dev,
                                        int32_t* n_valid_dev, void* dx, float* dW,
                                        void* stream);

/* Waits for `stream` and returns the first device-side error that
 * flce_forward_backward_async and flce_forward_backward_shard calls recorded
 * since the last flce_async_status
 * (FLCE_OK if none), then clears it. It reads the workspace the handle holds
 * now: an error recorded before the workspace was replaced is lost. */
flce_status flce_async_status(flce_handle_t h, void* stream);

/* ---- token-sharded batches (data parallelism over G GPUs) ---------------
 * The loss is a mean over the whole batch's non-ignored tokens, and dW a sum
 * over all of its tokens (the FLCE page, "Fused Linear Cross-Entropy: LLM
 * 학습 logits 메모리 병목 없애기", section "FLCE의 핵심 아이디어": dlogits,
 * dx and dW per chunk, the sums divided by the token count at the end; chunks
 * are independent but for those two sums). "Transformer Math 101"
 * (wonjae.kim), section "3D 병렬화", splits a batch over model replicas in the
 * same way. A batch whose tokens are split over G ranks, each holding a
 * replica of W, therefore needs: every rank's count of non-ignored tokens,
 * summed (one all-reduce of a scalar); each rank's fused call dividing by
 * that total; then the sum of dW and of the loss shares over the ranks (one
 * all-reduce each). dx needs nothing: its rows are the rank's own tokens.
 * The library does the two per-rank steps; the caller owns the collectives
 * (the Python wrapper linear_cross_entropy_token_gb300.token_parallel uses
 * torch.distributed). */

/* n_valid of this rank's tokens into DEVICE memory: *n_valid_dev =
 * #{i < N : t_i != ignore_index} (one int32), written when the stream gets
 * there; no host synchronisation. Targets are not range-checked here (the
 * fused call checks them). Errors: INVALID_ARG (null or misaligned pointer:
 * t 8-byte, n_valid_dev 4-byte; N < 0), CUDA. */
flce_status flce_count_valid(flce_handle_t h, const int64_t* t, int64_t N, int64_t ignore_index,
                             int32_t* n_valid_dev, void* stream);

/* flce_forward_backward_async for one shard of a token-sharded batch: every
 * step divides by *n_valid_total_dev (DEVICE, one int32: the non-ignored
 * tokens of all shards together) instead of this shard's own count, so
 *   loss_dev  (device, one fp32, may be NULL) receives this shard's share of
 *             the batch mean, sum over its tokens of the token loss / total;
 *   dx        is this shard's rows of the batch's dx, final as written;
 *   dW        is this shard's term of the batch's dW.
 * Summing loss_dev and dW over the shards gives the batch's loss and dW. A
 * total of 0 gives zeros, as for flce_forward_backward. No host
 * synchronisation; a total below this shard's own count, or negative, is
 * recorded as INVALID_ARG (and a bad target, or a wait that ran out, as for
 * the async call) and makes *loss_dev NaN; flce_async_status reports it.
 * Other arguments and errors as flce_forward_backward_async. */
flce_status flce_forward_backward_shard(flce_handle_t h, const void* x, const void* W,
                                        const int64_t* t, int64_t N, int64_t H, int64_t V,
                                        int64_t ignore_index, int64_t chunk,
                                        const int32_t* n_valid_total_dev, float* loss_dev,
                                        void* dx, float* dW, void* stream);

/* The same call with x, W and t in HOST memory: the library copies them into
 * its own device staging buffers on the stream (one cudaMemcpyAsync each),
 * then runs flce_forward_backward. dx and dW are device outputs as above.
 * Errors as flce_forward_backward, plus BUDGET if staging cannot be allocated. */
flce_status flce_forward_backward_host(flce_handle_t h, const void* x_host,
                                       const void* W_host, const int64_t* t_host,
                                       int64_t N, int64_t H, int64_t V,
                                       int64_t ignore_index, int64_t chunk, float* loss,
                                       void* dx, float* dW, void* stream);

/* The host-buffer call, pipelined: flce_submit_host enqueues it and returns
 * at once with a ticket; flce_wait(ticket) blocks until that call has
 * finished and gives its loss and status. The copies of x, W and t run on the
 * library's own copy stream into one of two staging slots, so the copies of
 * call k+1 overlap the compute of call k on `stream`; the compute still runs
 * in submission order on `stream`. At most two submissions may be
 * outstanding (submit returns INVALID_ARG otherwise). dx and dW are written
 * by the compute in submission order: a caller reusing them for several
 * submissions reads them after the wait of the call it wants. Host buffers
 * must stay unchanged until the call's wait returns; page-locked host memory
 * makes the copies asynchronous. flce_token_losses and flce_last_plan refer to
 * the most recent submission. The staging takes two buffers of the inputs'
 * size in device memory.
 * Errors: submit as flce_forward_backward_host for its arguments, plus
 * INVALID_ARG when two are outstanding; wait returns the call's status
 * (BAD_TARGET, TIMEOUT, CUDA) or INVALID_ARG for a ticket that is not
 * outstanding. */
flce_status flce_submit_host(flce_handle_t h, const void* x_host, const void* W_host,
                             const int64_t* t_host, int64_t N, int64_t H, int64_t V,
                             int64_t ignore_index, int64_t chunk, void* dx, float* dW,
                             void* stream, uint64_t* ticket);
flce_status flce_wait(flce_handle_t h, uint64_t ticket, float* loss);

/* Copy the per-token losses of the last call (N fp32, 0 for ignored tokens)
 * into device memory out. N must equal the last call's N. Errors: INVALID_ARG. */
flce_status flce_token_losses(flce_handle_t h, float* out, int64_t N, void* stream);

/* The plan the last call ran with. Errors: INVALID_ARG before any call. */
flce_status flce_last_plan(flce_handle_t h, flce_plan* out);

/* Per-kernel timing. While enabled, every launch is bracketed by CUDA
 * events recorded on the call's stream. */
flce_status flce_set_profiling(flce_handle_t h, int32_t enable);
/* Totals for one kernel kind since the last reset; synchronises on the
 * recorded events. Errors: INVALID_ARG for an unknown kind. */
flce_status flce_profile_read(flce_handle_t h, int32_t kind, flce_kernel_profile* out);
void flce_profile_reset(flce_handle_t h);
/* Name of a kernel kind (static string), "?" if unknown. */
const char* flce_kernel_name(int32_t kind);
/* Number of kernels this handle has launched (memsets and copies excluded). */
int64_t flce_launch_count(flce_handle_t h);

/* One-line reason for the handle's last failure ("" if none). */
const char* flce_last_error(flce_handle_t h);

/* ---- loss without any allocation ------------------------------------------
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot let a library allocate device memory: a framework whose pool
 * allocator must account for every byte, a runtime on a fixed memory plan
 * decided ahead of time, or code that must not pay the device-wide
 * synchronisation that cudaFree implies.
 *
 * Computes the mean loss and the per-token losses of x·Wᵀ (bf16 x and W, as
 * flce_forward_backward, same layout rules) without dx or dW, and without a
 * handle: it calls no cudaMalloc, cudaFree or allocating library routine. Its
 * scratch is one file-scope device array of 64 MiB, which every GPU that loads
 * the library holds until the process exits. That bounds V: one 128-token
 * chunk needs 128 x ceil(V/64) x 8 bytes of it (a max and a sum of exp per
 * 64 vocabulary columns), so V up to about 4.19 million. Larger V returns
 * INVALID_ARG.
 *   x, W, t      device inputs as for flce_forward_backward (current device)
 *   loss         host, receives the fp32 mean loss
 *   token_loss   device, N fp32 outputs (0 for ignored tokens)
 * The first call on a device looks up the device address of the scratch
 * array (cudaGetSymbolAddress) with that device current and keeps it for the
 * life of the process; that first call should come before any stream
 * capture begins. Calls after cudaDeviceReset (or any other teardown of the
 * device's primary context) are not supported: the kept address may then be
 * stale. Every call on a device shares the one array, which keeps the last
 * call's contents (each call clears what must start at zero), so calls that
 * overlap on the GPU (other streams, other threads) race: run them one after
 * another. Each call ends by synchronising `stream` to read the loss back.
 * Errors: INVALID_ARG, BAD_TARGET, TIMEOUT, CUDA. */
flce_status flce_loss_static(const void* x, const void* W, const int64_t* t, int64_t N,
                             int64_t H, int64_t V, int64_t ignore_index, float* loss,
                             float* token_loss, void* stream);

/* ---- checks of single parts (used by the tests) ------------------------- */

/* The tcgen05 GEMM core alone: C[M x N] (fp32, row-major, device) = A·B over
 * K, bf16 operands. a_mn_major = 0: A is M x K row-major (K contiguous);
 * 1: A is K x M row-major (M contiguous). b_mn_major = 0: B is N x K
 * row-major; 1: B is K x N row-major. M, N, K >= 1; the contiguous extent of
 * each operand must be a multiple of 8. Synchronises. Errors: INVALID_ARG,
 * UNSUPPORTED, TIMEOUT, CUDA. */
flce_status flce_check_gemm(flce_handle_t h, int32_t a_mn_major, int32_t b_mn_major,
                            const void* A, const void* B, float* C, int64_t M, int64_t N,
                            int64_t K, void* stream);

/* Runs one device-side wait on a barrier that nothing ever completes, with a
 * limit of timeout_us microseconds, and reports how it ended: TIMEOUT is the
 * expected result (the kernel gave up, recorded the error and returned
 * normally; the context stays usable). Synchronises. */
flce_status flce_check_wait_timeout(flce_handle_t h, uint32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FLCE_H */
