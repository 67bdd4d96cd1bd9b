/*
 * dpopt.h -- C ABI of the fused ZeRO gradient reduce + mixed-precision Adam
 * step for one GB300 (sm_103a).
 *
 * What one call computes, for every element i of one rank's shard:
 *
 *   g_i      = ( sum_{r=0..N-1} grad_r[i] ) / N      replica order fixed, ascending
 *   m_i     <- beta1 * m_i + (1 - beta1) * g_i
 *   v_i     <- beta2 * v_i + (1 - beta2) * g_i^2
 *   master_i <- master_i - lr * (m_i / (1 - beta1^t)) / (sqrt(v_i / (1 - beta2^t)) + eps)
 *   out_i    = bf16(master_i)                        round to nearest, ties to even
 *
 * Sources: the synchronised gradient is the sum of the replicas' local
 * gradients times 1/#Nodes, and the summation order is a choice that changes
 * floating-point results ("Data Parallelism 数据并行（二）", section "数据并行
 * 训练 (DP)"); ZeRO-3's reduce-scatter sums the gradients over all ranks and
 * each rank keeps and updates only its own 1/N shard ("Почему training 70B
 * модели требует optimizer sharding (ZeRO-3)?", sections 3 and 5); the
 * states are an fp32 master copy plus fp32 first and second moments beside a
 * 16-bit working copy, 16 bytes per parameter ("Глава 4.4 --
 * Распределённое обучение", section 2; the DP page's appendix "DNN 训练的
 * 内存需求").  The Adam equations are not printed on those pages; the
 * textbook bias-corrected form (Kingma & Ba 2015) is used, t = step, 1-based.
 *
 * Numerics: the replica sum is accumulated in fp32 with an error-free
 * transformation (TwoSum) and rounded once, so g equals the correctly rounded
 * average in all but vanishingly rare cases; m, v and the master update are
 * formed with compensated fp32 arithmetic, so stored values are within
 * 2.4e-7 relative (about 2 ulp) of an fp64 evaluation.  Every element is
 * owned by one thread and the order is fixed: results are bitwise identical
 * from run to run, and do not depend on bucket_elems or on how a shard is cut
 * into buckets.
 *
 * Conventions for every entry point:
 *  - Memory: the caller owns all memory.  Gradient, state and output pointers
 *    are DEVICE pointers of the current CUDA device; the pointer tables
 *    themselves (grads, grad_slices, slice_table) and offsets/lens are HOST
 *    arrays, read during the call only.  The library allocates no device
 *    memory (no cudaMalloc, no allocating library routine); on the host it
 *    builds each call's small launch tables in ordinary heap memory.
 *    A "DEVICE pointer" may also point into page-locked host memory that the
 *    device addresses at the same address (cudaHostAlloc, or cudaHostRegister
 *    with cudaHostRegisterMapped, on a system with unified addressing): the
 *    kernels then read the gradients from, or write param_bf16_out to, host
 *    memory in place -- on a Grace-Blackwell node over NVLink-C2C, which moves
 *    a step's host gradients in and its bf16 parameters out without separate
 *    copies.  Such operands run at the host link's bandwidth, not HBM's; the
 *    results are bitwise those of device-resident operands.  The library does
 *    not check where a pointer points: pageable host memory the device cannot
 *    reach is the caller's error, as is any other invalid pointer.
 *  - Layout: flat, contiguous, element-indexed.  bf16 values are IEEE
 *    binary32's upper 16 bits (stored as 2-byte words), fp32 are binary32.
 *  - In place: master, m, v are read and overwritten; param_bf16_out is only
 *    written.  Gradients are only read.  Gradient buffers must not overlap any
 *    state or output range, and the state/output ranges must not overlap one
 *    another (checked: DPOPT_ERR_INVALID_ARG).
 *  - Alignment: any element-aligned pointer is accepted; ranges whose pointers
 *    are all 16-byte aligned take the vectorised path, others a scalar path.
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and the call returns without waiting.  Errors in
 *    the arguments are reported synchronously; dpopt_stream_status() waits
 *    for the stream and reports anything the kernels flagged on the device.
 *  - Errors: every function returns a dpopt_status; nothing is thrown across
 *    the ABI.  On an error no work has been enqueued, except DPOPT_ERR_CUDA
 *    from a launch, after which earlier launches of the same call may have run.
 *  - Threads: all entry points may be called from several host threads; the
 *    only shared state is a per-device status word, cached device attributes,
 *    the process-wide kernel and gather policies, and the built-in array of
 *    the allocation-free norm entry (whose concurrent calls race; see there).
 */
#ifndef DPOPT_H
#define DPOPT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same types as cudaStream_t and cudaEvent_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *dpopt_stream_t;
struct CUevent_st;
typedef struct CUevent_st *dpopt_event_t;

typedef enum {
    DPOPT_OK = 0,
    DPOPT_ERR_INVALID_ARG = 1, /* a null/overlapping pointer, a size or hyper-parameter out of range */
    DPOPT_ERR_UNSUPPORTED = 2, /* valid but beyond this library's limits (n_replicas > DPOPT_MAX_REPLICAS) */
    DPOPT_ERR_CUDA = 3,        /* a CUDA call failed; dpopt_last_error() has its message */
    DPOPT_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (reported by dpopt_stream_status) */
    DPOPT_ERR_BOUNDS = 5       /* bounds-checked build only: a kernel derived an index outside
                                  its ranges and skipped the access (reported by
                                  dpopt_stream_status) */
} dpopt_status;

typedef enum {
    DPOPT_GRAD_BF16 = 0, /* 2-byte bf16 gradients */
    DPOPT_GRAD_F32 = 1,  /* 4-byte fp32 gradients */
    DPOPT_GRAD_F16 = 2   /* 2-byte IEEE binary16 gradients (loss-scaled runs) */
} dpopt_grad_dtype;

#define DPOPT_MAX_REPLICAS 64

/* Full-buffer entry.  Reduce-scatter semantics with all N contributions
 * resident in this GPU's memory ("Почему training 70B ...", section 5: sum the
 * gradients over all GPUs, keep only your own shard; then update only that
 * shard).
 *
 *  grads          HOST array of n_replicas DEVICE pointers; grads[r] is replica
 *                 r's flattened bf16 gradient buffer of `numel` elements.
 *  n_replicas     N, 1 <= N <= DPOPT_MAX_REPLICAS.
 *  numel          elements per replica buffer, a multiple of N (>= 0).
 *  shard_rank     r in [0, N): this rank updates [r*S, (r+1)*S), S = numel / N.
 *  bucket_elems   fusion-bucket size (>= 1): the shard is cut into buckets of this
 *                 many elements from its start, the last one ragged (DeepSpeed's
 *                 reduce_bucket_size over contiguous gradients in the config of
 *                 "Почему training 70B ...", section 8).  With every
 *                 contribution resident the buckets are only units of work:
 *                 the result does not depend on this value.
 *  master_f32, m_f32, v_f32
 *                 DEVICE pointers to the S-element fp32 shard states, updated in place.
 *  param_bf16_out DEVICE pointer to S bf16 elements, written: bf16(master) after the step.
 *  lr, beta1, beta2, eps
 *                 Adam hyper-parameters: finite, 0 <= beta < 1, eps >= 0.
 *  step           t >= 1, the 1-based index of this step (bias correction).
 *  stream         CUDA stream to enqueue on.
 * Returns DPOPT_OK or an error status (see the conventions above). */
int dpopt_reduce_adam(const void *const *grads, int n_replicas, int64_t numel, int shard_rank,
                      int64_t bucket_elems, float *master_f32, float *m_f32, float *v_f32,
                      void *param_bf16_out, float lr, float beta1, float beta2, float eps,
                      int64_t step, dpopt_stream_t stream);

/* dpopt_reduce_adam with the gradient type given (grad_dtype is a
 * dpopt_grad_dtype); everything else as above. */
int dpopt_reduce_adam_ex(const void *const *grads, int grad_dtype, int n_replicas, int64_t numel,
                         int shard_rank, int64_t bucket_elems, float *master_f32, float *m_f32,
                         float *v_f32, void *param_bf16_out, float lr, float beta1, float beta2,
                         float eps, int64_t step, dpopt_stream_t stream);

/* Bucket iterator over one shard.  count_out receives ceil(shard_elems /
 * bucket_elems) (0 for an empty shard); bucket idx covers [offset, offset+len)
 * of the shard, offset = idx*bucket_elems, len = bucket_elems except for a
 * ragged last bucket.  Host-only; no device work.
 * Errors: DPOPT_ERR_INVALID_ARG for shard_elems < 0, bucket_elems < 1, a null
 * output pointer, or idx outside [0, count). */
int dpopt_bucket_count(int64_t shard_elems, int64_t bucket_elems, int64_t *count_out);
int dpopt_bucket_range(int64_t shard_elems, int64_t bucket_elems, int64_t idx, int64_t *offset_out,
                       int64_t *len_out);

/* One bucket, with the gradients already cut to this rank's bucket (what a
 * reduce-scatter hands each rank).
 *  grad_slices    HOST array of n_replicas DEVICE pointers, each to `len`
 *                 gradient elements of type grad_dtype (replica r's slice).
 *  shard_offset   first shard element of the bucket (>= 0).
 *  len            elements in the bucket (>= 0; 0 is a no-op).
 *  master_f32, m_f32, v_f32, param_bf16_out
 *                 DEVICE pointers to the START of the shard's arrays; elements
 *                 [shard_offset, shard_offset+len) are updated / written.
 * Other arguments as for dpopt_reduce_adam. */
int dpopt_reduce_adam_bucket(const void *const *grad_slices, int grad_dtype, int n_replicas,
                             int64_t shard_offset, int64_t len, float *master_f32, float *m_f32,
                             float *v_f32, void *param_bf16_out, float lr, float beta1,
                             float beta2, float eps, int64_t step, dpopt_stream_t stream);

/* Many buckets per call (as few kernel launches as the pointer tables allow;
 * the buckets are put in shard order, whatever order they are listed in, and
 * those that continue one another in the shard and in every replica's
 * gradient memory are joined into one segment first, which gives the same
 * bits).
 *  slice_table    HOST array of n_buckets * n_replicas DEVICE pointers, bucket
 *                 major: slice_table[b * n_replicas + r] is replica r's slice of
 *                 bucket b (lens[b] elements of grad_dtype).
 *  offsets, lens  HOST arrays of n_buckets: bucket b updates shard elements
 *                 [offsets[b], offsets[b] + lens[b]).  Buckets must not overlap.
 * Other arguments as for dpopt_reduce_adam_bucket. */
int dpopt_reduce_adam_buckets(const void *const *slice_table, int grad_dtype, int n_replicas,
                              const int64_t *offsets, const int64_t *lens, int64_t n_buckets,
                              float *master_f32, float *m_f32, float *v_f32, void *param_bf16_out,
                              float lr, float beta1, float beta2, float eps, int64_t step,
                              dpopt_stream_t stream);

/* ------------------------------------------------------------------------- */
/* AdamW and global-norm gradient clipping                                    */
/* ------------------------------------------------------------------------- */

/* Options beyond plain Adam.  A zero-initialised struct means plain Adam.
 * The optimizer of the DeepSpeed example in "Почему training 70B модели требует
 * optimizer sharding (ZeRO-3)?" (section 8) is AdamW with weight_decay 0.01 and
 * gradient_clipping 1.0; the pages give no formulas, so these follow AdamW
 * (Loshchilov & Hutter 2019) and the usual global-norm clipping:
 *   g      <- fl32(g * c),  c = grad_unscale * min(1, max_grad_norm / (||g||_2 + 1e-6))
 *            (c in fp64, rounded once to fp32; ||g||_2 = sqrt(*grad_sqnorm))
 *   master <- (1 - lr*weight_decay) * master - lr * m_hat / (sqrt(v_hat) + eps)       */
typedef struct {
    float weight_decay;        /* decoupled weight decay, >= 0 (0: none) */
    float max_grad_norm;       /* > 0: clip to this global L2 norm (0: no clipping) */
    const double *grad_sqnorm; /* DEVICE pointer, read when max_grad_norm > 0: the squared
                                  global L2 norm of the unscaled averaged gradient, summed over
                                  every rank's shard (dpopt_grad_sqnorm per shard, then one
                                  scalar all-reduce across ranks) */
    float grad_unscale;        /* multiply the averaged gradient by this first (1/loss scale,
                                  a power of two keeps it exact); 0 means 1 */
} dpopt_step_options;

/* dpopt_reduce_adam_ex with options (opts may be NULL: plain Adam).  Always
 * takes the direct-load kernel.  Errors as for dpopt_reduce_adam_ex, plus
 * DPOPT_ERR_INVALID_ARG for a negative or non-finite option, or clipping
 * without an 8-byte aligned grad_sqnorm. */
int dpopt_reduce_adamw(const void *const *grads, int grad_dtype, int n_replicas, int64_t numel,
                       int shard_rank, int64_t bucket_elems, float *master_f32, float *m_f32,
                       float *v_f32, void *param_bf16_out, float lr, float beta1, float beta2,
                       float eps, int64_t step, const dpopt_step_options *opts,
                       dpopt_stream_t stream);

/* dpopt_reduce_adam_buckets with options. */
int dpopt_reduce_adamw_buckets(const void *const *slice_table, int grad_dtype, int n_replicas,
                               const int64_t *offsets, const int64_t *lens, int64_t n_buckets,
                               float *master_f32, float *m_f32, float *v_f32,
                               void *param_bf16_out, float lr, float beta1, float beta2,
                               float eps, int64_t step, const dpopt_step_options *opts,
                               dpopt_stream_t stream);

/* Every bucket in ONE launch: the launch table in caller-owned device memory.
 * dpopt_reduce_adam_buckets passes its pointer tables in the kernel's
 * parameter space, which holds 2048 slice pointers per launch (32 buckets at
 * 64 replicas), so one 70B model's ZeRO-3 shard at N = 64 in 4M-element
 * buckets ("Почему training 70B модели требует optimizer sharding (ZeRO-3)?",
 * sections 4 and 8: a 1/64 shard, reduce_bucket_size) could take nine launches
 * per step.  This form runs every bucket in one launch.  Like
 * dpopt_reduce_adam_buckets it first joins buckets that continue one another
 * (taken in shard order, one bucket starting where the previous one ends, in
 * the shard and in every replica's gradient memory, as in a flat contiguous
 * gradient buffer); if
 * what remains fits one launch's parameter space it launches from there and
 * leaves `table` untouched, otherwise it writes the checked launch table into
 * `table` and the direct-load kernel reads it from device memory.  Its
 * results are bitwise those of dpopt_reduce_adam_buckets (opts NULL) and
 * dpopt_reduce_adamw_buckets (opts given).
 *
 * dpopt_bucket_table_bytes: bytes of `table` for n_buckets buckets of
 *   n_replicas slices: 32 * (n_buckets + 1) + 8 * n_buckets * n_replicas.
 *   Errors: DPOPT_ERR_INVALID_ARG for a null bytes_out, n_replicas outside
 *   [1, DPOPT_MAX_REPLICAS] or n_buckets outside [0, 2^30].
 *
 * dpopt_reduce_adam_buckets_table:
 *  slice_table, offsets, lens, n_buckets, states, hyper-parameters
 *                 as for dpopt_reduce_adam_buckets (host arrays, read during
 *                 the call only).
 *  opts           NULL for plain Adam, else as for dpopt_reduce_adamw.
 *  table          DEVICE pointer, 16-byte aligned, at least
 *                 dpopt_bucket_table_bytes() bytes, owned by the caller and
 *                 overlapping no state, output or gradient range.  When it is
 *                 used, the call enqueues on `stream` one host-to-device copy
 *                 of the packed table into it, then the kernel that reads it;
 *                 its previous contents do not matter.  It is stream ordered
 *                 like the states: work on another stream must not touch it
 *                 until this call's kernel has finished.
 *  table_bytes    size of `table` in bytes.
 * Errors: as for dpopt_reduce_adamw_buckets, plus DPOPT_ERR_INVALID_ARG for a
 * null or misaligned table, too small a table_bytes, or a table overlapping a
 * state, output or gradient range; DPOPT_ERR_CUDA if the copy or the launch
 * fails. */
int dpopt_bucket_table_bytes(int n_replicas, int64_t n_buckets, int64_t *bytes_out);
int dpopt_reduce_adam_buckets_table(const void *const *slice_table, int grad_dtype,
                                    int n_replicas, const int64_t *offsets, const int64_t *lens,
                                    int64_t n_buckets, float *master_f32, float *m_f32,
                                    float *v_f32, void *param_bf16_out, float lr, float beta1,
                                    float beta2, float eps, int64_t step,
                                    const dpopt_step_options *opts, void *table,
                                    int64_t table_bytes, dpopt_stream_t stream);

/* Squared L2 norm of this shard's averaged gradient (the clipping pre-pass):
 *   *sqnorm_out = sum_i (g_i * grad_unscale)^2      (fp64, DEVICE pointer)
 * with g_i the same fixed-order average the step computes.  Partial sums over
 * fixed 4096-element chunks go to `scratch` (a DEVICE buffer the caller owns,
 * at least dpopt_grad_sqnorm_scratch_bytes() bytes, 8-byte aligned) and are
 * added in chunk order, so the result is bitwise reproducible and does not
 * depend on the GPU's SM count.  Arguments as for dpopt_reduce_adam_ex;
 * grad_unscale 0 means 1.  Errors: DPOPT_ERR_INVALID_ARG for the usual
 * argument errors, a null/misaligned sqnorm_out or scratch, too small a
 * scratch, or gradients overlapping either. */
int dpopt_grad_sqnorm(const void *const *grads, int grad_dtype, int n_replicas, int64_t numel,
                      int shard_rank, float grad_unscale, double *sqnorm_out, void *scratch,
                      int64_t scratch_bytes, dpopt_stream_t stream);

/* The same over a batch of bucket slices (arguments as for
 * dpopt_reduce_adam_buckets).  The buckets are taken in shard order, in
 * whatever order they are listed, and those that continue one another (in the
 * shard and in every replica's gradient memory, as in a flat contiguous
 * gradient buffer) are joined first: the result does not depend on the
 * listing order, and such buckets covering the whole shard give the bits of
 * dpopt_grad_sqnorm over the full buffers.  The scratch size of
 * dpopt_grad_sqnorm_scratch_bytes(elems, n_buckets) covers every case. */
int dpopt_grad_sqnorm_buckets(const void *const *slice_table, int grad_dtype, int n_replicas,
                              const int64_t *offsets, const int64_t *lens, int64_t n_buckets,
                              float grad_unscale, double *sqnorm_out, void *scratch,
                              int64_t scratch_bytes, dpopt_stream_t stream);

/* dpopt_grad_sqnorm without a scratch buffer.  Not part of the method on the
 * source pages (they have no counterpart): it serves callers that cannot call
 * cudaMalloc for the step's scratch -- code whose device memory is all owned by
 * another allocator (a framework's caching allocator that has reserved the
 * GPU), or that must not trigger the device-wide synchronisation cudaMalloc /
 * cudaFree can cause in the middle of a training step.  The chunk partials go
 * to an array built into the library: 524288 fp64 values (4 MB) on every
 * device that loads the library, held until the process exits, which limits a
 * shard to 2^31 elements (DPOPT_ERR_UNSUPPORTED beyond that, with a message
 * from dpopt_last_error()).  It allocates nothing and calls no allocating
 * routine.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for the
 * process; make that first call before any stream capture (a call with
 * numel = 0 does only that set-up and writes 0 to *sqnorm_out).  The kept
 * address belongs to the device's primary context: it is not valid in other
 * contexts made current through the driver API, nor after cudaDeviceReset.
 * With lazy module loading (CUDA_MODULE_LOADING=LAZY, the default) the 4 MB
 * are committed when the library's kernels are first used on the device, which
 * may be this first call; if the device is full by then, it fails with
 * DPOPT_ERR_CUDA (out of memory).  Every call on a device shares the one array, and each
 * call writes every partial it reads, so no state carries over between calls;
 * but calls that can run at the same time on the GPU (other streams, other host
 * threads) race on it -- serialise them.  Arguments, result and other errors
 * as for dpopt_grad_sqnorm. */
int dpopt_grad_sqnorm_noalloc(const void *const *grads, int grad_dtype, int n_replicas,
                              int64_t numel, int shard_rank, float grad_unscale,
                              double *sqnorm_out, dpopt_stream_t stream);

/* dpopt_grad_sqnorm that also stores the shard's averaged gradient -- the
 * reduced gradient partition a reduce-scatter leaves on each rank in ZeRO's
 * stage 2 ("ZeRO: Memory Optimizations Toward Training Trillion Parameter
 * Models", Pos+g): avg_out[i] = g_i for i = 0 .. S-1 (S = numel / n_replicas),
 * the fixed-order average of element i of this rank's shard in fp32, before
 * grad_unscale -- the same g the fused step forms.  avg_out is a DEVICE buffer
 * of S floats that the caller owns, 4-byte aligned (16- or 32-byte alignment
 * lets the kernel store vectors), overlapping neither the gradients nor
 * sqnorm_out nor scratch.  A following step can read the average instead of
 * the N replicas: dpopt_reduce_adamw(&avg_out, DPOPT_GRAD_F32, 1, S, 0, ...)
 * (or dpopt_amp_step with the same arguments) gives bit for bit the states
 * that the fused call on the N replicas gives, moving 4 + 26 bytes per
 * parameter in that pass instead of 2N + 26.  Errors: as for
 * dpopt_grad_sqnorm, and DPOPT_ERR_INVALID_ARG for a null, misaligned or
 * overlapping avg_out. */
int dpopt_grad_average_sqnorm(const void *const *grads, int grad_dtype, int n_replicas,
                              int64_t numel, int shard_rank, float grad_unscale, float *avg_out,
                              double *sqnorm_out, void *scratch, int64_t scratch_bytes,
                              dpopt_stream_t stream);

/* The norm pass bucket by bucket as the gradients become ready (row f4's
 * overlap for the clipped and loss-scaled steps: the pass over each bucket runs
 * while the backward pass is still producing the others; only the short step
 * on the stored average waits for the last bucket).  For each bucket with
 * lens[b] > 0, in the listed order: if ready[b] is non-null, `stream` waits
 * for that event, then the bucket's pass is launched; after the last bucket
 * the ordered finish writes *sqnorm_out.  The buckets are not joined: each
 * bucket's partials sit at its rank in shard order, so the result is bitwise
 * that of dpopt_grad_sqnorm_buckets over the same buckets held in separate
 * memory, whatever the listing order.  avg_out: NULL (norm only), or a DEVICE
 * array indexed like the states (as for dpopt_grad_average_sqnorm_buckets,
 * here for any buckets) that receives each element's average.
 *  ready          HOST array of n_buckets events (dpopt_event_t = cudaEvent_t).
 * Other arguments and errors as for dpopt_grad_average_sqnorm_buckets, plus
 * DPOPT_ERR_INVALID_ARG for a null `ready` with n_buckets > 0. */
int dpopt_grad_sqnorm_buckets_when_ready(const void *const *slice_table, int grad_dtype,
                                         int n_replicas, const int64_t *offsets,
                                         const int64_t *lens, int64_t n_buckets,
                                         const dpopt_event_t *ready, float grad_unscale,
                                         float *avg_out, double *sqnorm_out, void *scratch,
                                         int64_t scratch_bytes, dpopt_stream_t stream);

/* dpopt_grad_average_sqnorm over bucket slices: dpopt_grad_sqnorm_buckets that
 * also stores each element's average at its shard offset, avg_out[offsets[b]
 * + j] for element j of bucket b.  The buckets must join into one segment
 * (contiguous gradients, ZeRO's `contiguous_gradients` layout, as in the
 * ZeRO-3 answer's config, section 8), else DPOPT_ERR_UNSUPPORTED.  avg_out is
 * a DEVICE array indexed like the states, 4-byte aligned, whose span the
 * buckets cover overlapping neither the gradients nor sqnorm_out nor scratch.
 * The step then reads the average as one fp32 replica --
 * dpopt_reduce_adamw(&avg_out, DPOPT_GRAD_F32, 1, S, 0, ...) for buckets
 * covering the shard -- with the bits of the fused bucket step, moving
 * 2N + 4 bytes per parameter here and 4 + 26 in the step instead of 2N + 26:
 * at N = 64 about 162 bytes per parameter for the clipped step in place of
 * 282.  Errors: as for dpopt_grad_sqnorm_buckets, plus DPOPT_ERR_INVALID_ARG
 * for a null, misaligned or overlapping avg_out. */
int dpopt_grad_average_sqnorm_buckets(const void *const *slice_table, int grad_dtype,
                                      int n_replicas, const int64_t *offsets,
                                      const int64_t *lens, int64_t n_buckets, float grad_unscale,
                                      float *avg_out, double *sqnorm_out, void *scratch,
                                      int64_t scratch_bytes, dpopt_stream_t stream);

/* Scratch bytes dpopt_grad_sqnorm{,_buckets} need for `elems` gradient elements
 * per replica cut into n_buckets buckets (use n_buckets = 1 for the full-buffer
 * form): 8 * (ceil(elems / 4096) + n_buckets).  Host-only. */
int dpopt_grad_sqnorm_scratch_bytes(int64_t elems, int64_t n_buckets, int64_t *bytes_out);

/* ------------------------------------------------------------------------- */
/* fp16 gradients with dynamic loss scaling                                   */
/* ------------------------------------------------------------------------- */

/* The fp16 block of the ZeRO-3 answer's DeepSpeed config (section 8: loss_scale 0
 * = dynamic, initial_scale_power 16, loss_scale_window 1000, hysteresis 2,
 * min_loss_scale 1); the pages give only the keys.  Reading used here:
 *  - the gradients arrive multiplied by the loss scale; the step divides the
 *    averaged gradient by it (exact for a power-of-two scale);
 *  - a step overflows when any averaged gradient element of any rank is not
 *    finite, i.e. the global squared norm of the unscaled gradient is not finite;
 *  - an overflowing step is skipped: master, m, v, the bf16 copy and the step
 *    count stay as they were; the run of clean steps restarts, and every
 *    `hysteresis`-th overflow since the scale last changed halves the scale
 *    (never below min_scale);
 *  - after `window` clean steps in a row the scale doubles.
 * The state lives in DEVICE memory the caller owns and is read and written only
 * by the library's kernels, so a run needs no host synchronisation per step. */
typedef struct {
    float scale;             /* current loss scale */
    int32_t good_steps;      /* clean steps since the last overflow or scale change */
    int32_t hysteresis_left; /* overflows left before the scale is halved */
    int32_t last_overflow;   /* 1 when the last step was skipped */
    int64_t step;            /* optimizer steps applied (bias-correction t of the next = step+1) */
    int64_t skipped;         /* steps skipped for overflow */
} dpopt_loss_scale_state;    /* 32 bytes, 8-byte aligned */

typedef struct {
    float init_scale;        /* e.g. 65536 = 2^initial_scale_power */
    int32_t window;          /* loss_scale_window, >= 1 */
    int32_t hysteresis;      /* >= 1 */
    float min_scale;         /* min_loss_scale, > 0 */
} dpopt_loss_scale_config;

/* Write the initial state (scale = init_scale, counters 0) into *state (DEVICE). */
int dpopt_loss_scale_init(dpopt_loss_scale_state *state, const dpopt_loss_scale_config *cfg,
                          dpopt_stream_t stream);

/* dpopt_grad_sqnorm with the gradient unscaled by 1 / state->scale read on the
 * device.  Sum the ranks' results (one scalar all-reduce) into the global
 * squared norm that dpopt_amp_step reads; a non-finite value means overflow. */
int dpopt_amp_sqnorm(const void *const *grads, int grad_dtype, int n_replicas, int64_t numel,
                     int shard_rank, const dpopt_loss_scale_state *state, double *sqnorm_out,
                     void *scratch, int64_t scratch_bytes, dpopt_stream_t stream);

/* dpopt_amp_sqnorm that also stores the averaged gradient (before the unscale)
 * in avg_out, as dpopt_grad_average_sqnorm does; dpopt_amp_step on
 * (&avg_out, DPOPT_GRAD_F32, 1, S, 0, ...) then gives the fused step's states. */
int dpopt_amp_average_sqnorm(const void *const *grads, int grad_dtype, int n_replicas,
                             int64_t numel, int shard_rank, const dpopt_loss_scale_state *state,
                             float *avg_out, double *sqnorm_out, void *scratch,
                             int64_t scratch_bytes, dpopt_stream_t stream);

/* dpopt_amp_average_sqnorm over bucket slices that join into one segment (as
 * dpopt_grad_average_sqnorm_buckets, with the unscale 1 / state->scale read on
 * the device): the loss-scaled step of a bucketed, contiguous gradient buffer
 * is this pass, the scalar all-reduce, then dpopt_amp_step on (&avg_out,
 * DPOPT_GRAD_F32, 1, S, 0, ...). */
int dpopt_amp_average_sqnorm_buckets(const void *const *slice_table, int grad_dtype,
                                     int n_replicas, const int64_t *offsets, const int64_t *lens,
                                     int64_t n_buckets, const dpopt_loss_scale_state *state,
                                     float *avg_out, double *sqnorm_out, void *scratch,
                                     int64_t scratch_bytes, dpopt_stream_t stream);

/* dpopt_grad_sqnorm_buckets_when_ready for the loss-scaled step: the unscale
 * 1 / state->scale read on the device.  With the ZeRO-3 answer's config
 * (section 8: fp16 with a dynamic loss scale, overlap_comm) each bucket's pass
 * runs as soon as the bucket's gradients exist; the scalar all-reduce and
 * dpopt_amp_step on avg_out follow the last bucket. */
int dpopt_amp_sqnorm_buckets_when_ready(const void *const *slice_table, int grad_dtype,
                                        int n_replicas, const int64_t *offsets,
                                        const int64_t *lens, int64_t n_buckets,
                                        const dpopt_event_t *ready,
                                        const dpopt_loss_scale_state *state, float *avg_out,
                                        double *sqnorm_out, void *scratch, int64_t scratch_bytes,
                                        dpopt_stream_t stream);

/* One loss-scaled step of this rank's shard (full-buffer layout, arguments as for
 * dpopt_reduce_adam_ex): if *global_sqnorm is finite, AdamW (weight_decay) on the
 * averaged gradient times c = (1/scale) * min(1, max_grad_norm / (||g|| + 1e-6))
 * (max_grad_norm 0: no clipping), with the bias corrections of step state->step
 * + 1; then the state is advanced (or the step is counted as skipped).  The
 * step index comes from the state, not from the caller.
 * global_sqnorm may be NULL when max_grad_norm is 0: then there is no overflow
 * test, the step is always taken, and only state->step advances (the scale and
 * its counters are left as they are; with scale 1 the gradient is used as it
 * is).  That is the step of a run without loss scaling whose step count lives
 * on the device -- the form to capture in a CUDA graph (see below).
 * lr_dev: NULL, or a DEVICE pointer (4-byte aligned) to the learning rate as
 * one float, read by the step when it runs (the `lr` argument is then not
 * used): a learning-rate schedule writes it between replays of a captured
 * graph.  The step forms lr / (1 - beta1^t) and 1 - lr * weight_decay from it
 * in fp64 exactly as the host forms them from `lr`, so the same rate gives the
 * same bits either way; a non-finite rate gives non-finite states.
 * Errors: as for dpopt_reduce_adam_ex, plus DPOPT_ERR_INVALID_ARG for a
 * misaligned global_sqnorm, a NULL one with max_grad_norm > 0, or a state
 * overlapping a state or output array. */
int dpopt_amp_step(const void *const *grads, int grad_dtype, int n_replicas, int64_t numel,
                   int shard_rank, int64_t bucket_elems, float *master_f32, float *m_f32,
                   float *v_f32, void *param_bf16_out, float lr, float beta1, float beta2,
                   float eps, float weight_decay, float max_grad_norm,
                   const double *global_sqnorm, dpopt_loss_scale_state *state,
                   const dpopt_loss_scale_config *cfg, const float *lr_dev,
                   dpopt_stream_t stream);

/* ------------------------------------------------------------------------- */
/* CUDA graphs                                                                */
/* ------------------------------------------------------------------------- */

/* Every entry that takes a stream only enqueues kernels (and, for the table
 * entry, one copy) on it, allocates nothing and never synchronises, so it may
 * be called while the stream is being captured into a CUDA graph; the graph
 * then holds the call's launches with the arguments of the call.  What a
 * replay does follows from that:
 *  - the entries that take `step` (and lr) from the caller repeat that step on
 *    every replay: capture them once per step, or update the kernel nodes'
 *    parameters between replays;
 *  - dpopt_amp_sqnorm / dpopt_amp_step read the loss scale and the step count
 *    from the device state and advance it themselves, and dpopt_amp_step can
 *    read the learning rate from device memory (lr_dev), so one captured graph
 *    of an iteration replays iteration after iteration, learning-rate schedule
 *    included (with global_sqnorm NULL for a run without loss scaling);
 *  - dpopt_reduce_adam_buckets_table refuses with DPOPT_ERR_UNSUPPORTED when
 *    its launch table must be written (the buckets do not fit the parameter
 *    space) while `stream` is capturing: the table is copied from host memory
 *    that the next call reuses, which a replay would read stale;
 *  - dpopt_stream_status synchronises and must not be called on a capturing
 *    stream; dpopt_reduce_adam_buckets_when_ready waits on the caller's events,
 *    which must then belong to the same capture;
 *  - dpopt_grad_sqnorm_noalloc must have been called once (numel 0 will do)
 *    before the capture, so that its device array's address is resolved. */

/* ------------------------------------------------------------------------- */
/* ZeRO-3 parameter all-gather                                                */
/* ------------------------------------------------------------------------- */

/* Write this rank's bf16 shard into every replica's parameter buffer
 * ("Почему training 70B ...", section 5: before each layer's forward and backward
 * the full parameters are all-gathered from the ranks' shards).  With every
 * replica resident the gather is a local broadcast:
 *   param_replicas[r][shard_rank*shard_elems + i] = shard_bf16[i],  r < n_replicas.
 *  shard_bf16      DEVICE pointer to shard_elems bf16 values (e.g. param_bf16_out of
 *                  a step); a replica whose destination is this very range is skipped.
 *  param_replicas  HOST array of n_replicas DEVICE pointers, each to a flat bf16
 *                  buffer of at least n_replicas*shard_elems elements.
 * Calling it for every shard_rank gives every replica the full updated vector.
 * Errors: DPOPT_ERR_INVALID_ARG for null or misaligned pointers, a rank outside
 * [0, n_replicas), destinations overlapping the shard or one another;
 * DPOPT_ERR_UNSUPPORTED for n_replicas > DPOPT_MAX_REPLICAS. */
int dpopt_allgather_bf16(const void *shard_bf16, int64_t shard_elems, int shard_rank,
                         void *const *param_replicas, int n_replicas, dpopt_stream_t stream);

/* The step of dpopt_reduce_adam_ex and the all-gather of its bf16 shard in one
 * pass over memory (the same section: the optimizer updates the rank's shard,
 * then every rank's parameters are gathered for the next forward pass).  The
 * rank's own replica buffer holds the working copy: with S = numel/n_replicas
 * and base = shard_rank*S,
 *   param_replicas[r][base + i] = bf16(master_f32[i] after the step),  r < n_replicas,
 * bit for bit what dpopt_reduce_adam_ex(..., param_replicas[shard_rank] + base, ...)
 * followed by dpopt_allgather_bf16 of that range writes, and master/m/v as that
 * step leaves them.  The call runs one fused kernel -- the bf16 copy is never
 * read back: g*N + 24 + 2N bytes per parameter instead of g*N + 28 + 2N, and
 * each CTA's 4 KB tile of new bf16 values goes to every replica buffer as bulk
 * copies from shared memory; it measured faster than the two launches at
 * every replica count and size on GB300 (dpopt_set_gather_policy can still
 * select the two launches).
 *  grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, master_f32,
 *  m_f32, v_f32, lr, beta1, beta2, eps, step, stream
 *                  as for dpopt_reduce_adam_ex.
 *  param_replicas  HOST array of n_replicas DEVICE pointers, each to a flat bf16
 *                  buffer of at least numel elements; only [base, base + S) of
 *                  each is written.  The ranges written must not overlap one
 *                  another, the states or the gradients.  16-byte aligned
 *                  ranges take 16-byte stores, others go one element at a time.
 * Errors: as for dpopt_reduce_adam_ex, and DPOPT_ERR_INVALID_ARG for a null
 * table or replica pointer, a misaligned replica pointer, or overlapping
 * ranges. */
int dpopt_reduce_adam_allgather(const void *const *grads, int grad_dtype, int n_replicas,
                                int64_t numel, int shard_rank, int64_t bucket_elems,
                                float *master_f32, float *m_f32, float *v_f32,
                                void *const *param_replicas, float lr, float beta1, float beta2,
                                float eps, int64_t step, dpopt_stream_t stream);

/* Bucket-as-ready: the batched-bucket step with one launch per bucket, each made
 * to wait on the stream for that bucket's readiness event first.  The producer
 * of the gradients (a backward pass on another stream, last layer first) records
 * ready[b] when bucket b's slices are complete, so the step of early buckets runs
 * while later ones are still being produced -- the one-GPU counterpart of
 * starting each bucket's reduction as soon as its gradients exist instead of
 * after the whole backward pass ("Глава 4.4", section 7: overlap of communication
 * with computation; the ZeRO-3 answer's overlap_comm; the DP page's gradient
 * hooks that launch a non-blocking all-reduce per parameter).
 *  ready  HOST array of n_buckets events (cudaEvent_t); a NULL entry means the
 *         bucket is ready already.  Buckets run in array order, so list them in the
 *         order their gradients become ready (a backward pass: last bucket first).
 * Other arguments and errors as for dpopt_reduce_adam_buckets, plus
 * DPOPT_ERR_CUDA if waiting on an event fails.  Results equal the batched
 * entry's bit for bit. */
int dpopt_reduce_adam_buckets_when_ready(const void *const *slice_table, int grad_dtype,
                                         int n_replicas, const int64_t *offsets,
                                         const int64_t *lens, int64_t n_buckets,
                                         const dpopt_event_t *ready, float *master_f32,
                                         float *m_f32, float *v_f32, void *param_bf16_out,
                                         float lr, float beta1, float beta2, float eps,
                                         int64_t step, dpopt_stream_t stream);

/* Wait for `stream`, then return and clear the current device's status word:
 * DPOPT_OK, or DPOPT_ERR_TIMEOUT if a bounded device-side wait gave up since the
 * last call, or DPOPT_ERR_CUDA if the wait itself failed; in the bounds-checked
 * build also DPOPT_ERR_BOUNDS if a kernel's index check failed since the last
 * call. */
int dpopt_stream_status(dpopt_stream_t stream);

/* The bounds-checked build (libdpopt_bounds.so: the same sources compiled with
 * -DDPOPT_DEBUG_BOUNDS; dpopt_version() ends in "+bounds") is the library's
 * stand-in for a memory checker.  Before each access whose index a kernel
 * derives from its launch tables (segment, element offset, state span) it tests
 * the index against the segment's length and the call's span of shard elements;
 * a failed test skips the access and sets a device word that
 * dpopt_stream_status() reports as DPOPT_ERR_BOUNDS.  Results are otherwise
 * bitwise those of the release build, which compiles the tests away.
 * dpopt_selftest_bounds enqueues a kernel whose check fails on purpose (it
 * touches no memory), so that a test can see the report arrive: DPOPT_OK in the
 * bounds-checked build, DPOPT_ERR_UNSUPPORTED in the release build. */
int dpopt_selftest_bounds(dpopt_stream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *dpopt_status_string(int status);

/* Message of the last DPOPT_ERR_CUDA / DPOPT_ERR_INVALID_ARG raised on the
 * calling host thread ("" if none).  Valid until the thread's next call. */
const char *dpopt_last_error(void);

/* Model-state bytes one data-parallel device holds for psi parameters.
 *  variant 0: mixed-precision Adam, 16 bytes/parameter: 2 (16-bit params) + 2
 *             (16-bit grads) + 12 (fp32 master, m, v) ("Глава 4.4", section 2).
 *  variant 1: the ZeRO-3 answer's conservative 70B figure as printed, 2 + 2 + 4
 *             bytes/parameter (140 + 140 + 280 GB = 560 GB, its section 2).
 *  zero_stage 0 keeps all; 1 shards the optimizer states over n_dp devices;
 *  2 also the gradients; 3 also the parameters ("Глава 4.4", section 6:
 *  16*Psi/N_dp at the most aggressive stage).
 * Errors: DPOPT_ERR_INVALID_ARG for psi < 0, n_dp < 1, an unknown variant or
 * stage, or a null bytes_out.  Host-only. */
int dpopt_state_bytes(int64_t psi, int variant, int n_dp, int zero_stage, double *bytes_out);

/* Which kernel carries the step (process-wide; default DPOPT_KERNEL_AUTO).
 *  DPOPT_KERNEL_AUTO    the faster of the two for the replica count, by measurement
 *  DPOPT_KERNEL_DIRECT  direct vector loads from global memory into registers
 *  DPOPT_KERNEL_BULK    bulk copies (TMA) into a shared-memory ring, where it applies
 *                       (master/m/v 32-byte aligned, every other pointer 16-byte
 *                       aligned, two stages of 2048 elements fit 100 KB of shared
 *                       memory: bf16 N <= 6, fp32 N <= 3); other calls still take
 *                       the direct-load kernel
 * Both kernels give bitwise identical results.  Errors: DPOPT_ERR_INVALID_ARG for an
 * unknown value. */
typedef enum { DPOPT_KERNEL_AUTO = 0, DPOPT_KERNEL_DIRECT = 1, DPOPT_KERNEL_BULK = 2 } dpopt_kernel_policy;
int dpopt_set_kernel_policy(int policy);
int dpopt_get_kernel_policy(void);

/* Which form dpopt_reduce_adam_allgather takes (process-wide; default
 * DPOPT_GATHER_AUTO).
 *  DPOPT_GATHER_AUTO      the faster by measurement: the fused kernel (see the entry)
 *  DPOPT_GATHER_FUSED     always the one fused kernel
 *  DPOPT_GATHER_SEPARATE  always the step into the own replica, then the
 *                         broadcast into the others
 * All give bitwise identical results.  Errors: DPOPT_ERR_INVALID_ARG for an
 * unknown value. */
typedef enum {
    DPOPT_GATHER_AUTO = 0,
    DPOPT_GATHER_FUSED = 1,
    DPOPT_GATHER_SEPARATE = 2
} dpopt_gather_policy;
int dpopt_set_gather_policy(int policy);
int dpopt_get_gather_policy(void);

/* Diagnostic: enqueue a kernel whose one bounded wait can never be satisfied, so
 * that it gives up after limit_cycles GPU clock cycles (1 .. 2e9) and sets the
 * device status word; dpopt_stream_status() then returns DPOPT_ERR_TIMEOUT.  Lets
 * a caller check that time-outs are reported and that the context stays usable. */
int dpopt_selftest_wait_timeout(int64_t limit_cycles, dpopt_stream_t stream);

/* Kernel launches this library has made from the calling host thread since
 * the thread started (a running count; the caller takes differences). */
int64_t dpopt_launch_count(void);

/* Library version, "major.minor.patch". */
const char *dpopt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DPOPT_H */
