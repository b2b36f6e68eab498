/*
 * zero_gb300.h -- C ABI of the partitioned mixed-precision ZeRO step on one
 * GB300 (sm_103a).  N data-parallel ranks are simulated inside one GPU's
 * HBM: every rank's 16-bit gradient buffer and parameter replica are
 * separate device buffers, and the owner shards of the fp32 optimizer state
 * are laid out back to back in one flat buffer.  The collectives of the
 * method (reduce-scatter, all-gather, per-bucket broadcast, the scalar
 * all-reduce of norm and overflow flag) are HBM streams fused into the
 * update kernels.
 *
 * Sources (web pages on ZeRO, cited by title and section):
 *  - "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models"
 *    (summary), Sec. 3.1 mixed-precision Adam state (2+2+12 bytes/param),
 *    Sec. 5 stages P_os / P_os+g / P_os+g+p, Sec. 7 communication volume,
 *    residual states (gradient norm over the flattened buffer).
 *  - "zero-stages-simulation" README: flat contiguous partition, rank r owns
 *    chunk r; per-stage schedule table; byte-accurate accounting.
 *  - "CMU 11-868 L18: How ZeRO Cuts Data-Parallel Memory": ZeRO-1 call
 *    sequence (reduce-scatter into an FP32 shard, update, copy to 16-bit,
 *    all-gather); ZeRO-3 broadcast from owner before forward and backward.
 *
 * General conventions
 *  - Every call returns a zero_status_t.  Nothing aborts, throws or traps;
 *    on error the call launches nothing and zero_last_error() says why.
 *  - All tensor arguments are caller-owned DEVICE pointers (the caller
 *    allocates them, e.g. with PyTorch) unless a comment says "host".  The
 *    library owns only its workspace (status word, norm partials, chunk
 *    counters, and for some modes an fp32 gradient buffer of psi_pad floats).
 *  - Device pointers must be 16-byte aligned.  The 128-bit vector path runs
 *    when psi_pad (or a bucket's bounds) are multiples of 8, and for a bucket
 *    of double-buffered state also psi_pad (the second slot's offset);
 *    otherwise an element-wise path runs with the same arithmetic.
 *  - Calls are asynchronous on the given CUDA stream (a cudaStream_t passed
 *    as void*, NULL = legacy default stream).  One host thread per handle.
 *    The reduce-scatters and steps of one handle share its status word and
 *    norm partials, so they must run in order (one stream, or ordered by
 *    events); gathers may overlap them on another stream.  At most 64
 *    launches of one handle may be in flight at once: each takes the next
 *    of 64 work counters, round-robin.
 *  - The streaming kernels are launched with programmatic stream
 *    serialisation: the next one may be scheduled while the previous one
 *    drains, and waits in its first instruction until that one has
 *    completed.  Stream order is unchanged for the caller; a caller's own
 *    kernel or copy on the same stream runs after the library's work as
 *    usual, and the calls can be captured into a CUDA graph.
 *  - Elements [psi, psi_pad) are padding: gradients there are ignored, and
 *    master/m/v/params there are written as 0.
 *  - The loss scale, the count t of applied Adam steps and the live slot of
 *    double-buffered state are DEVICE-side handle state, so a step never
 *    waits for the host: an overflowing step halves the scale (floor 1.0)
 *    and leaves t unchanged without a host round trip.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ZERO_API __attribute__((visibility("default")))
#else
#define ZERO_API
#endif

typedef enum {
    ZERO_OK = 0,
    ZERO_EINVAL = 1,    /* bad argument: null/misaligned pointer, range, stage/mode mismatch */
    ZERO_ENOMEM = 2,    /* workspace allocation failed */
    ZERO_ECUDA = 3,     /* a CUDA runtime call or kernel launch failed */
    ZERO_ETIMEOUT = 4,  /* zero_get_status: a bounded wait inside a kernel gave up (staged step) */
    ZERO_ESTATE = 5     /* call sequence wrong (e.g. stage-3 step before every bucket was reduced) */
} zero_status_t;

typedef enum { ZERO_FP16 = 0, ZERO_BF16 = 1 } zero_dtype_t;

typedef enum {
    ZERO_MODE_AUTO = 0,            /* SPECULATIVE if possible, else TWO_PASS_WS for N > 4, else REREAD */
    ZERO_MODE_TWO_PASS_WS = 1,     /* pass 1 writes fp32 g_hat to workspace; pass 2 reads it */
    ZERO_MODE_TWO_PASS_REREAD = 2, /* pass 2 reduces the N gradient buffers again */
    ZERO_MODE_SPECULATIVE = 3,     /* one pass writing the shadow state slot; commit, roll back, or
                                      (one-shot step whose norm needs clipping) redo from the old slot */
    ZERO_MODE_SPECULATIVE_STAGED = 4 /* SPECULATIVE, inputs staged through shared memory by bulk
                                        async copies (stages 1/2 one-shot step; N <= 19, i.e. two
                                        stages of N*4 KiB + 24 KiB fit in 200 KiB of shared
                                        memory; psi_pad a multiple of 8; fp32 state 32-byte
                                        aligned; grads and master/m/v in device memory,
                                        not host memory; otherwise ZERO_EINVAL) */
} zero_mode_t;

/* zero_init_partition flags */
#define ZERO_F_DOUBLE_BUFFER 1u    /* master/m/v hold two slots of psi_pad floats (stages 1-3) */

#define ZERO_MAX_RANKS 64

typedef struct zero_handle* zero_handle_t;   /* opaque, library-owned */

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float max_norm;   /* global-norm clip threshold; <= 0 disables clipping */
    int32_t mode;     /* zero_mode_t */
} zero_hyper_t;

typedef struct {
    int32_t overflow;       /* last step skipped: a non-finite averaged gradient, or (error != 0)
                               a kernel wait that gave up */
    int32_t applied;        /* last step updated the state */
    int32_t state_slot;     /* live slot (0/1) of double-buffered master/m/v; 0 otherwise */
    int32_t error;          /* device-side error word, 0 = none; 1 = a bounded wait of the staged
                               step gave up.  Stays set until zero_set_scaler. */
    double grad_norm;       /* L2 norm of the averaged unscaled gradient of the last step; not
                               meaningful when overflow = 1 (a one-pass step stops at the
                               first non-finite value it finds) */
    double clip_coef;       /* fp32 factor applied to the gradient (1.0 when not clipping) */
    float loss_scale;       /* current loss scale, after any halving */
    float reserved;
    int64_t steps_applied;  /* t: Adam steps applied so far */
    int64_t steps_skipped;  /* steps skipped on overflow so far */
} zero_result_t;

typedef struct {
    uint64_t psi, psi_pad, shard, n_ranks, stage;
    uint64_t model_state_bytes_per_rank;  /* 16/4+12/N/2+14/N/16/N bytes x psi_pad, exact
                                             (stage 3 with a resident region: see
                                             zero_set_persistent) */
    uint64_t comm_elems_paper;            /* 2 psi_pad (stages 0-2), 3 psi_pad (stage 3) */
    uint64_t comm_elems_ring;             /* 2(N-1)/N psi_pad, 3(N-1)/N psi_pad for stage 3 */
    uint64_t hbm_read_bytes, hbm_write_bytes;   /* algorithmic HBM bytes of the last call */
    uint64_t hbm_read_total, hbm_write_total;   /* cumulative since init */
} zero_bytes_t;

/*
 * zero_init_partition -- a1: partition a flat buffer of psi parameters over
 * n_ranks simulated ranks and allocate the handle's workspace.
 *   ("zero-stages-simulation" README, flat partitioning: N near-equal
 *    contiguous chunks, rank r owns chunk r; ZeRO summary Sec. 5, P_os: N_d
 *    equal partitions.)
 * psi_pad = smallest multiple of n_ranks*align >= psi; shard = psi_pad/N;
 * offset_r = r*shard; real_r = clamp(psi - offset_r, 0, shard).
 *   psi      >= 0 (0 gives an empty step)
 *   n_ranks  1..ZERO_MAX_RANKS
 *   stage    0..3 (ZeRO-0 plain DP, P_os, P_os+g, P_os+g+p)
 *   dtype    zero_dtype_t of gradients and parameters
 *   align    >= 1 elements (8 keeps every shard 16-byte aligned)
 *   flags    ZERO_F_DOUBLE_BUFFER or 0 (stage 0 rejects it)
 *   out      host pointer receiving the handle
 * Uses the current CUDA device.  Errors: EINVAL, ENOMEM, ECUDA.
 */
ZERO_API int zero_init_partition(uint64_t psi, int n_ranks, int stage, int dtype, int align,
                        unsigned flags, zero_handle_t* out);

/*
 * zero_partition_info -- the partition (host values, exact).  offsets and
 * real are host arrays of n_ranks entries, or NULL.  Any output may be NULL.
 */
ZERO_API int zero_partition_info(zero_handle_t h, uint64_t* psi_pad, uint64_t* shard,
                        uint64_t* offsets, uint64_t* real);

/*
 * zero_set_scaler -- set the device-side loss scale, applied-step count t
 * and live state slot (0/1; must be 0 without ZERO_F_DOUBLE_BUFFER).  Used
 * before the first step and to resume from a checkpoint.  Stream-ordered.
 * The loss scale must be finite and > 0.  Errors: EINVAL, ECUDA.
 */
ZERO_API int zero_set_scaler(zero_handle_t h, float loss_scale, int64_t steps_applied,
                    int32_t state_slot, void* stream);

/*
 * zero_step -- one mixed-precision ZeRO step (a2..a8, a11).
 *   Stages 0-2: reduce the N ranks' 16-bit gradients in fixed order 0..N-1
 *   in fp32, divide by N*loss_scale (CMU notes, ZeRO-1 step 3: sum and
 *   average into an FP32 shard), test for inf/nan, form the global L2 norm
 *   (ZeRO summary, residual states: norm over the flattened gradient), clip
 *   if max_norm > 0, run AdamW on the owners' fp32 master/m/v (ZeRO summary
 *   Sec. 3.1 and Sec. 5), round to 16 bits and write every rank's replica
 *   (the all-gather; CMU notes steps 5-6).  Stage 0 all-reduces and updates
 *   N full replicas of the state (ZeRO summary Sec. 7, baseline DP).
 *   Stage 3: grads must be NULL; the N gradients were already consumed by
 *   zero_reduce_scatter_bucket calls covering [0, psi_pad) exactly once
 *   since the last step.  Stage 2 with grads NULL: the same, after
 *   zero_reduce_scatter_bucket_replicas calls.  This call finishes the norm/overflow/clip and
 *   (two-pass modes) applies Adam and writes the 16-bit shard.
 * On overflow nothing of master/m/v/params changes, the scale halves and t
 * is not advanced.
 * Speculative mode (ZERO_F_DOUBLE_BUFFER; AUTO picks it for stages 1/2):
 * one pass updates the shadow slot and the replicas assuming no clipping.
 * If the norm then calls for clipping, a second pass redoes the update
 * from the untouched old slot with the clip factor, so only clipped steps
 * pay for two passes.  Bucketed steps (stage 3, and stage 2 with NULL grads)
 * cannot re-read their gradients and use the two-pass mode when clipping.
 *   grads   host array of N device pointers, psi_pad 16-bit elements each
 *           (stages 0-2); NULL for stage 3
 *   params  host array of N device pointers to psi_pad 16-bit replicas
 *           (stages 0-2), or of 1 pointer to the psi_pad 16-bit
 *           concatenation of the owner shards (stage 3).  Replicas must
 *           equal the RNE cast of the live master on entry.
 *   master, m, v  fp32 device buffers.  Stages 1-3: psi_pad floats (the N
 *           owner shards back to back), or 2*psi_pad with
 *           ZERO_F_DOUBLE_BUFFER (slot s at offset s*psi_pad).  Stage 0:
 *           N*psi_pad floats, replica r at offset r*psi_pad.
 *   hyper   host pointer, read during the call only
 * Errors: EINVAL, ESTATE, ECUDA, ENOMEM (first two-pass call allocates the
 * fp32 workspace; make it before any stream capture).
 */
ZERO_API int zero_step(zero_handle_t h, const void* const* grads, void* const* params,
              float* master, float* m, float* v, const zero_hyper_t* hyper, void* stream);

/*
 * zero_gather_bucket -- a9: ZeRO-3 parameter gather of bucket [a, b): every
 * rank receives the owners' 16-bit values, out[r][j] = shard16[a + j].
 *   (ZeRO summary Sec. 5, P_os+g+p: the owner broadcasts a layer's
 *    parameters before its forward and again before its backward; CMU
 *    notes, ZeRO-3: ncclBroadcast from the owning GPU.)
 *   0 <= a <= b <= psi_pad.  shard16: device, psi_pad 16-bit elements.
 *   out: host array of N device pointers, b - a elements each.
 * Stage 3 only.  Errors: EINVAL, ECUDA.
 */
ZERO_API int zero_gather_bucket(zero_handle_t h, uint64_t a, uint64_t b, const void* shard16,
                       void* const* out, void* stream);

/*
 * zero_reduce_scatter_bucket -- a10: ZeRO-3 gradient reduce-scatter of
 * bucket [a, b) into the owners' shards: the a2..a5 steps restricted to the
 * bucket.  (ZeRO summary Sec. 5, P_os+g / P_os+g+p: reduce-scatter as the
 * gradients of each layer appear in backward; CMU notes, ZeRO-2/3: each
 * segment's gradients are reduced to its owner.)
 * With ZERO_F_DOUBLE_BUFFER and no clipping (mode AUTO or SPECULATIVE) the
 * bucket's AdamW update is fused here: new master/m/v go to the shadow slot
 * and the new 16-bit values straight into shard16[a, b); zero_step then
 * commits, or on overflow restores shard16 from the old master.  Otherwise
 * the averaged gradient is written to the fp32 workspace and zero_step
 * applies Adam.
 *   grads: host array of N device pointers, b - a 16-bit elements each.
 *   master, m, v, shard16: as for zero_step of stage 3 (may be NULL in
 *   two-pass modes).  Every call of one step must pass the same hyper.
 *   Buckets of one step must not overlap.  At most 4096 per step.
 * Stage 3 only.  Errors: EINVAL, ESTATE, ECUDA, ENOMEM.
 */
ZERO_API int zero_reduce_scatter_bucket(zero_handle_t h, uint64_t a, uint64_t b,
                               const void* const* grads, float* master, float* m, float* v,
                               void* shard16, const zero_hyper_t* hyper, void* stream);

/*
 * zero_reduce_scatter_gather_bucket -- zero_reduce_scatter_bucket of bucket
 * [a, b) and zero_gather_bucket of bucket [ga, gb) in one call: the
 * reduce-scatter of one layer's gradients in backward together with the
 * gather of the next layer's parameters, fetched one layer ahead.
 *   (ZeRO summary Sec. 5, P_os+g+p: in backward the parameters are gathered
 *    again in reverse order, a layer's gradients are reduce-scattered as they
 *    appear, and the next layer can be fetched while the current one is
 *    processed; "ZeRO Stage 1/2/3" guide, ZeRO-3 config: prefetch_bucket_size.)
 * The result is that of the two calls one after the other.  When both parts
 * are 8-wide (a, b - a, ga and gb - ga multiples of 8) they run as one launch
 * whose work counter hands out the reduce-scatter's chunks first and then
 * the gather's, so that the gather fills the end of the reduce-scatter;
 * otherwise the two calls are made in turn.  Either part may be empty.
 *   The two buckets must not overlap, and no out[r] may share memory with
 *   the 16-bit shard, master, m, v or a gradient row of [a, b) (ZERO_EINVAL).
 *   Arguments: those of zero_reduce_scatter_bucket, then ga, gb and out
 *   (host array of N device pointers, gb - ga elements each) as for
 *   zero_gather_bucket.  zero_bytes_moved counts both parts as this call.
 * Stage 3 only.  Errors: EINVAL, ESTATE, ECUDA, ENOMEM.
 */
ZERO_API int zero_reduce_scatter_gather_bucket(zero_handle_t h, uint64_t a, uint64_t b,
                                               const void* const* grads, float* master, float* m, float* v,
                                               void* shard16, const zero_hyper_t* hyper, uint64_t ga,
                                               uint64_t gb, void* const* out, void* stream);

/*
 * zero_reduce_scatter_bucket_replicas -- ZeRO-2 with the gradients reduced
 * during backward: the reduce-scatter of bucket [a, b) as its gradients
 * appear, after which the ranks may release or reuse their gradient
 * buffers for the next bucket (a constant-size buffer per rank).
 *   (ZeRO summary Sec. 5, P_os+g: reduce-scatter during backward, bucketized
 *    per partition, gradient memory freed; Sec. 6 CB: constant-size fused
 *    buffers; CMU notes, ZeRO-2: reduce each segment to its owner, delete.)
 * With ZERO_F_DOUBLE_BUFFER and no clipping the bucket's AdamW update and
 * its all-gather into every replica are fused here (shadow slot; replicas
 * written at once); zero_step(h, NULL grads, params, ...) then commits, or
 * on overflow restores the replicas from the old master.  Otherwise g_hat
 * goes to the fp32 workspace and that zero_step applies AdamW and writes
 * the replicas.  The buckets of one step must tile [0, psi_pad) without
 * overlap (at most 4096) and pass the same hyper.
 *   grads: host array of N device pointers, b - a 16-bit elements each
 *   params: host array of N device pointers to the psi_pad replicas
 *   master, m, v: as for zero_step (may be NULL in two-pass modes)
 * Stage 2 only.  Errors: EINVAL, ESTATE, ECUDA, ENOMEM.
 */
ZERO_API int zero_reduce_scatter_bucket_replicas(zero_handle_t h, uint64_t a, uint64_t b,
                                        const void* const* grads, float* master, float* m, float* v,
                                        void* const* params, const zero_hyper_t* hyper, void* stream);

/*
 * ZeRO++ block-quantized exchanges.  ("CMU 11-868 L18" notes, other memory
 * optimizations: ZeRO++ block-quantizes parameters from 16 bits to INT8 with
 * zero-point quantization for the forward gather, and quantizes the
 * backward reduce-scatter to INT8 or INT4.)
 * Format: blocks of ZERO_Q_BLOCK elements counted from the start of the
 * buffer (or bucket); per block lo = min and hi = max (a NaN makes both NaN),
 * scale = (hi - lo) / (2^bits - 1) in fp32, code = rint((x - lo) / scale)
 * with the subtraction and the division each rounded once, clamped to
 * [0, 2^bits - 1] (0 when scale == 0; 0 for a NaN); dequantized
 * x' = lo + code * scale (fp32 multiply, then add).  Codes: one byte per
 * element (bits = 8) or two per byte with the even element in the low nibble
 * (bits = 4); `scales` holds one {scale, lo} float pair per block.  Code
 * buffers and 16-bit buffers must be 16-byte aligned, scales 8-byte aligned.
 */
#define ZERO_Q_BLOCK 256

/* Quantize count 16-bit values (a rank's bucket gradient before the
 * reduce-scatter, qgZ).  Needs no handle: errors via zero_last_error(NULL). */
ZERO_API int zero_quantize_blocks(int dtype, int bits, const void* src16, uint64_t count, void* codes,
                         float* scales, void* stream);

/* Dequantize count values to 16 bits (RNE): what a rank computes with after
 * a quantized gather.  Needs no handle. */
ZERO_API int zero_dequantize_blocks(int dtype, int bits, const void* codes, const float* scales, uint64_t count,
                           void* out16, void* stream);

/* a9 with qwZ: the owners' 16-bit values of bucket [a, b) are quantized to
 * INT8 once and every rank r receives the codes (codes_out[r], b - a bytes)
 * and scales (scales_out[r], 2*ceil((b-a)/256) floats).  Stage 3 only.
 * Errors: EINVAL, ECUDA. */
ZERO_API int zero_gather_bucket_q8(zero_handle_t h, uint64_t a, uint64_t b, const void* shard16,
                          void* const* codes_out, float* const* scales_out, void* stream);

/* a10 with qgZ: zero_reduce_scatter_bucket whose inputs are the N ranks'
 * quantized bucket gradients (codes[r], scales[r], as zero_quantize_blocks
 * writes them for the bucket's b - a elements).  The owner sums the
 * dequantized values in rank order; everything after is as for
 * zero_reduce_scatter_bucket, and zero_step finishes the step.  Stage 3. */
ZERO_API int zero_reduce_scatter_bucket_q(zero_handle_t h, uint64_t a, uint64_t b, int bits,
                                 const void* const* codes, const float* const* scales, float* master,
                                 float* m, float* v, void* shard16, const zero_hyper_t* hyper, void* stream);

/*
 * zero_get_status -- a11: copy the device status of the last step to the
 * host struct *out (host pointer).  Synchronises the given stream.
 * Errors: EINVAL, ECUDA; ETIMEOUT (with *out filled) while the device error
 * word is set, i.e. after a staged step whose bounded wait gave up.
 */
ZERO_API int zero_get_status(zero_handle_t h, void* stream, zero_result_t* out);

/*
 * zero_debug_hold_staged -- test hook for the failure path of
 * ZERO_MODE_SPECULATIVE_STAGED.  In the next staged zero_step on this handle
 * (one-shot), CTA 0 stops issuing its bulk copies at its tile `tile` (its
 * tiles counted from 0), so its compute warps' bounded waits run out (about
 * 2 s) instead of receiving data.  No access leaves its buffers and every
 * wait ends.  That step is then skipped (overflow = 1, master/m/v and the
 * replicas unchanged, loss scale kept), the error word is set and
 * zero_get_status returns ZERO_ETIMEOUT until zero_set_scaler clears it.
 * tile < 0 clears a pending hold; a tile past CTA 0's last has no effect.
 * Errors: EINVAL (NULL handle).
 */
ZERO_API int zero_debug_hold_staged(zero_handle_t h, int64_t tile);

/*
 * zero_set_persistent -- tell a stage-3 handle that the flat region
 * [p0, psi_pad) stays replicated: every rank keeps a resident 16-bit copy of
 * it, refreshed by one gather after each update, and its buckets are not
 * gathered before forward or backward.
 *   ("ZeRO Stage 1/2/3" guide, ZeRO-3 config: param_persistence_threshold,
 *    parameters below it stay replicated; ZeRO summary Sec. 5 and Sec. 7 for
 *    the P_os+g+p memory and communication it changes.)
 * Host-only bookkeeping: it changes what zero_bytes_moved reports and
 * nothing that runs on the device (the caller makes the gathers; see the
 * package's ZeRO-3 schedule).  With psi_pers = psi_pad - p0:
 *   model_state_bytes_per_rank = 16 psi_pad / N + 2 psi_pers
 *   comm_elems_paper           = 3 psi_pad - psi_pers
 *   comm_elems_ring            = floor((N - 1)(3 psi_pad - psi_pers) / N)
 * p0 = psi_pad (the default) means no resident region.
 * Errors: EINVAL (NULL handle, stage != 3, p0 > psi_pad).
 */
ZERO_API int zero_set_persistent(zero_handle_t h, uint64_t p0);

/*
 * zero_bytes_moved -- D4/D5 accounting and algorithmic HBM bytes.
 *   (ZeRO summary Sec. 5 memory equations and Sec. 7 communication volume;
 *    "zero-stages-simulation" README: byte-accurate memory tracker and a
 *    counting interconnect.)  Host-only, exact integers.  The HBM counters
 *   count the bytes the method must move for the calls made, assuming
 *   each step applied (an overflow's rollback pass is not counted).
 */
ZERO_API int zero_bytes_moved(zero_handle_t h, zero_bytes_t* out);

/*
 * zero_step_noalloc -- the two-pass step of stages 1/2 for callers that
 * cannot allocate device memory.  The ZeRO pages have no counterpart: this
 * is a packaging of zero_step for such callers.
 * Some callers may not call cudaMalloc: code in a framework whose caching
 * allocator owns the device memory (a foreign cudaMalloc also synchronises
 * the whole device), or code under a memory budget fixed before training
 * starts.  zero_init_partition allocates a workspace, so those callers use
 * this call instead.  It takes no handle and calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *   Its scratch -- the status word, the norm partials, the chunk counters
 *   and the fp32 averaged gradient -- lives in one static device array of
 *   ZERO_NOALLOC_MAX_PSI_PAD floats plus 324,960 bytes (about 16.3 MiB),
 *   which every GPU that loads the library holds until the
 *   process exits.  psi_pad above ZERO_NOALLOC_MAX_PSI_PAD is rejected
 *   with ZERO_EINVAL.
 *   The first call on a device looks up that array's device address
 *   (cudaGetSymbolAddress) and, like any first launch of a kernel, may have
 *   the driver load the library's kernels onto the device; make that first
 *   call before any stream capture.  Later calls leave the device's free
 *   memory unchanged.
 *   Every call shares the one array and overwrites what the last call left
 *   there (it clears the status word first): calls that overlap on the GPU,
 *   from any thread or stream, race and give wrong results.  Order them.
 * Arguments are those of zero_init_partition and zero_step (stages 1/2,
 * one state slot, updated in place), plus:
 *   loss_scale, steps_applied  host values of the loss scale and of t
 *           before this step.  The caller keeps them between calls: it
 *           passes what the previous call's result reported, so it reads
 *           that result back (after synchronising the stream) first.
 *   result  pointer the GPU can write (device, managed or pinned host
 *           memory; pageable host memory is refused), 8-byte aligned,
 *           receiving the step's
 *           zero_result_t, stream-ordered: overflow, applied, norm, clip
 *           factor, the loss scale after this step (halved on overflow,
 *           floor 1.0), t after this step, and steps_skipped = 1 if this
 *           call skipped its update (0 otherwise)
 *   hyper->mode must be ZERO_MODE_AUTO or ZERO_MODE_TWO_PASS_WS.
 * Errors: EINVAL (read zero_last_error(NULL)), ECUDA.
 */
#define ZERO_NOALLOC_MAX_PSI_PAD (1ull << 22)

/*
 * zero_noalloc_scratch_bytes -- bytes of the static device array that
 * zero_step_noalloc uses, per GPU that loads the library:
 * 4 * ZERO_NOALLOC_MAX_PSI_PAD + 324,960.  A host query: no CUDA call, no
 * GPU needed, no error.
 */
ZERO_API uint64_t zero_noalloc_scratch_bytes(void);

ZERO_API int zero_step_noalloc(uint64_t psi, int n_ranks, int stage, int dtype, int align,
                      const void* const* grads, void* const* params,
                      float* master, float* m, float* v, const zero_hyper_t* hyper,
                      float loss_scale, int64_t steps_applied, zero_result_t* result,
                      void* stream);

/* Last error message of this handle (or of the last failed init when h is
 * NULL).  The string is owned by the library and valid until the next call. */
ZERO_API const char* zero_last_error(zero_handle_t h);

/* Free the handle and its workspace.  Synchronises the device first.  NULL is a no-op. */
ZERO_API void zero_destroy(zero_handle_t h);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_H */
