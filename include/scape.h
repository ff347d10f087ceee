/*
 * scape.h -- C ABI of the SCAPE sharded sparse optimizer step on one GB300 (sm_103a).
 *
 * SCAPE ("SCAPE: Accurate and Efficient LLM Training with Extremely Sparse
 * Communication", arXiv 2607.01678) is a momentum-masked, error-feedback,
 * extreme-sparsity AdamS optimizer for sharded data parallelism.  This library
 * runs its per-step update for W data-parallel workers held as W gradient
 * slices on one GPU, so the cross-worker sparse reduce is an on-device sum and
 * no collective runs.  The same step split over several GPUs: shard-range
 * handles (scape_create_range; no data-path collective) and the exchange
 * form (scape_xc_*; the caller issues the collectives between its phases).
 *
 * Citations below name the paper ("SCAPE", Chinese translation page, sections
 * I and II-A..II-C) and the technical summary ("Sintesi Tecnica: SCAPE",
 * gist.science, Sec. 2 "Metodologia").
 *
 * Conventions for every entry point
 *   - Return value: SCAPE_OK (0) or a negative scape_status.  Nothing throws
 *     across the ABI.  scape_last_error() returns a message for the last
 *     failure on a handle (or, with a NULL handle, for the last failed
 *     scape_create on the calling thread).
 *   - Pointers are device pointers unless the name starts with host_.
 *   - The caller owns every device buffer (parameters, first moment, residuals,
 *     gradients, workspace).  The library keeps non-owning pointers and small
 *     host metadata only; it allocates no device buffers (it creates CUDA
 *     streams, events and, for the replayed warm refresh, a CUDA graph).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All GPU work is enqueued asynchronously on it; a non-zero status reports
 *     argument, state or launch errors only.  Faults of enqueued work surface
 *     at the caller's next synchronisation.
 *   - A handle is not thread-safe: one thread at a time per handle.
 *
 * Layout
 *   P = sum of the layer sizes; parameters are one flat float32 vector w[P]
 *   (layers concatenated in the order given).  Optimizer shard s of W covers
 *   [floor(s*P/W), floor((s+1)*P/W)) ("SCAPE" Sec. II-A: the distributed
 *   optimizer partitions states and parameters evenly over the workers), and
 *   keeps k_s = ceil(n_s * (1 - sparsity)) coordinates (sparsity rounded to
 *   parts per million); k = sum k_s is fixed for the life of the handle.
 *   The global mask is a bitmap, bit (i % 32) of 32-bit word i / 32 set when
 *   parameter i is selected; bits past P in the last word are zero.
 */
#ifndef SCAPE_H
#define SCAPE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct scape scape_t;

enum scape_status {
    SCAPE_OK = 0,
    SCAPE_EINVAL = -1, /* bad argument: null/misaligned pointer, size, range */
    SCAPE_ECUDA = -2,  /* a CUDA runtime call or kernel launch failed */
    SCAPE_ESTATE = -4  /* call out of order (e.g. step before bind) */
};

enum scape_dtype {
    SCAPE_F32 = 0, /* gradients are float32 */
    SCAPE_BF16 = 1 /* gradients are bfloat16 */
};

/* Upper bound on W (simulated workers = optimizer shards). */
#define SCAPE_MAX_WORKERS 256

/*
 * Create a handle.  Host only: validates the arguments and computes the shard
 * layout and k; no GPU work.
 *   host_layer_numel  n_layers sizes (each >= 0, sum P in [1, 2^31 - 1])
 *   W                 workers = optimizer shards, 1..SCAPE_MAX_WORKERS
 *   sparsity          fraction of coordinates NOT sent per shard, in [0, 1)
 *                     (90% and 99% in "SCAPE" abstract)
 *   beta1, beta2      AdamS coefficients in [0, 1) ("SCAPE" Sec. II-C, Eq. 2)
 *   lr                learning rate eta; eps > 0; weight_decay lambda >= 0
 *   grad_dtype        SCAPE_F32 or SCAPE_BF16
 * On success *out owns host memory only; release it with scape_destroy().
 */
int scape_create(scape_t **out, int n_layers, const int64_t *host_layer_numel, int W,
                 double sparsity, float beta1, float beta2, float lr, float eps,
                 float weight_decay, int grad_dtype);

/*
 * Create a handle for the optimizer shards [shard_begin, shard_end) of the
 * problem scape_create() would lay out for these layers and W: one rank's
 * share of the sharded optimizer ("SCAPE" Sec. II-A: the distributed optimizer
 * partitions parameters and states evenly over the workers; "Sintesi Tecnica:
 * SCAPE" Sec. 2: each worker computes the mask only for its own partition).
 * The handle covers the contiguous parameters [lo, hi), lo = floor(shard_begin
 * * P_global / W), hi = floor(shard_end * P_global / W), with the global shard
 * boundaries and per-shard k_s; every buffer bound to it and every gradient
 * passed to it is the [lo, hi) slice (local index 0 = global index lo).  Each
 * step still takes W gradient slices (all workers) and averages over W.
 * Because shards are independent, running every range of a partition of
 * [0, W) gives, slice by slice, exactly the whole problem's results.  Bitmap,
 * index list and packed buffers are in local coordinates (bit i of the
 * handle's bitmap is global parameter lo + i).  scape_get_range() gives the
 * range; scape_get_geometry() reports P = hi - lo and the shard_end -
 * shard_begin local shards.
 * Errors: as scape_create(), plus SCAPE_EINVAL unless 0 <= shard_begin <
 * shard_end <= W and the range holds at least one parameter.
 */
int scape_create_range(scape_t **out, int n_layers, const int64_t *host_layer_numel, int W,
                       int shard_begin, int shard_end, double sparsity, float beta1,
                       float beta2, float lr, float eps, float weight_decay, int grad_dtype);

/* Global size, offset of the first covered parameter and the covered shard
 * range [shard_begin, shard_end) of a handle (0 and [0, W) for scape_create()
 * handles).  Any output pointer may be NULL. */
int scape_get_range(const scape_t *h, int64_t *P_global, int64_t *offset, int *shard_begin,
                    int *shard_end);

/* Release a handle (NULL is a no-op).  Does not free caller-owned memory. */
void scape_destroy(scape_t *h);

/* Message for the last failure (never NULL; "" when none). */
const char *scape_last_error(const scape_t *h);

/*
 * Geometry of a handle: P (parameters covered), W (workers), k and, when the
 * host_ arrays are non-NULL, the S + 1 local shard boundaries and the S
 * per-shard k_s, S = W for scape_create() handles and shard_end - shard_begin
 * for scape_create_range() ones (partitioned mask: each worker selects only
 * within its own optimizer shard, "Sintesi Tecnica: SCAPE" Sec. 2).  Any
 * output pointer may be NULL.
 */
int scape_get_geometry(const scape_t *h, int64_t *P, int *W, int64_t *k,
                       int64_t *host_shard_start, int64_t *host_shard_k);

/* Bytes of device workspace scape_bind() needs (mask bitmap, packed index
 * list, W packed buffers of k floats, the synchronised buffer, tile tables and
 * mask-refresh scratch). */
int scape_workspace_bytes(const scape_t *h, size_t *bytes);

/*
 * Bind caller-owned device memory.  Must precede every GPU call; may be
 * called again to re-bind (the optimizer step count and the mask are reset to
 * "no step taken").
 *   params       float32 w[P], updated in place
 *   m            float32 first moment m[P], updated in place (caller zeroes it
 *                before the first step)
 *   host_e_ptrs  host array of W device-accessible pointers, each float32
 *                e^w[P]: the per-worker error-feedback residual ("SCAPE"
 *                Sec. II-B; FP32, same size as the gradient), updated in place
 *                (caller zeroes).  They may point to pinned host memory: the
 *                kernels then read and write the residuals over the host link
 *                in place, keeping W*P*4 bytes out of HBM (the pages offload
 *                these buffers to the CPU side, "SCAPE" Sec. I)
 *   workspace    >= scape_workspace_bytes(), 256-byte aligned
 * params, m and every e^w must be 16-byte aligned and must not overlap.
 */
int scape_bind(scape_t *h, float *params, float *m, float *const *host_e_ptrs,
               void *workspace, size_t ws_bytes);

/*
 * One optimizer step t -> t + 1 on `stream`.
 *   host_grad_ptrs  host array of W device pointers, each the worker's
 *                   gradient g^w[P] of the bound dtype; read only.  Any
 *                   alignment is accepted; 16-byte alignment of every
 *                   gradient and residual selects the vectorised path.
 * Step 1 is dense (mask of all ones): a^w = g^w + e^w, g_bar = mean_w a^w,
 * AdamS on all P, e^w <- 0.  Every later step uses the mask of the most recent
 * scape_refresh_mask() (built from m after the previous step: the one-step
 * lagged mask of "Sintesi Tecnica: SCAPE" Sec. 2):
 *   1. error feedback and compaction ("SCAPE" Sec. II-B): a^w = g^w + e^w; the
 *      selected a^w are packed in ascending index order into worker w's
 *      k-long buffer, e^w <- a^w - (sent part);
 *   2. the W packed buffers are summed in worker order 0..W-1 and divided by
 *      W: the single synchronised sparse buffer g_bar;
 *   3. AdamS at the k selected coordinates from that one buffer ("SCAPE"
 *      Sec. II-C Eq. 2, bias corrections 1 - beta^t; "Sintesi Tecnica:
 *      SCAPE" Sec. 2, second moment rebuilt from the single buffer):
 *      m' = b1 m + (1-b1) g;  v = b2 m^2 + (1-b2) g^2;
 *      w <- w - lr (m'/bc1 / (sqrt(v/bc2) + eps) + wd w);  m <- m'.
 *      Unselected w and m are left unchanged.
 * Errors: SCAPE_ESTATE before scape_bind() or, for t >= 1, before the first
 * scape_refresh_mask(); SCAPE_EINVAL for a NULL gradient pointer.
 */
int scape_step(scape_t *h, const void *const *host_grad_ptrs, void *stream);

/*
 * Build the mask for the next step from the current first moment: for each
 * shard s independently, select the k_s coordinates with the largest |m|
 * (key = IEEE bits of m with the sign cleared, compared as unsigned; equal
 * keys go to the lower index), write them into the global bitmap (the shard
 * masks land in disjoint ranges: the mask all-gather of "Sintesi Tecnica:
 * SCAPE" Sec. 2), then the ascending packed index list and the per-tile rank
 * table the next step's compaction uses.  The mask comes from first-moment
 * statistics, not gradients ("SCAPE" Sec. I).
 * The result is exact whatever the data.  Its cost is not: the first call
 * after scape_bind() reads m two or three times; every later call reads it
 * once, writing the bitmap from the previous threshold and correcting it,
 * as long as each shard's threshold stays near the previous one (a shard
 * whose threshold moved further is counted and re-marked in full).  When
 * every shard keeps all of its coordinates (sparsity 0, or shards of one
 * parameter) the mask is all ones and only the first call does any work.
 * Errors: SCAPE_ESTATE before the first step.
 */
int scape_refresh_mask(scape_t *h, void *stream);

/*
 * Variant readings (flags, combinable; default SCAPE_VARIANT_PAPER).  They
 * change what later steps compute:
 *   SCAPE_VARIANT_DENSE_OFFMASK  unselected coordinates also take the AdamS
 *       update with a zero synchronised gradient (m decays by b1, v = b2 m^2),
 *       the other reading of "SCAPE" Sec. II-C under a sparse buffer;
 *   SCAPE_VARIANT_MOMENT_SYNC    the synchronised buffer holds first moments
 *       ("Sintesi Tecnica: SCAPE" Sec. 2): each worker packs
 *       b = b1 m_{t-1} + (1 - b1) a, m_t is the mean of the b, and the gradient
 *       of the second moment is recovered as (m_t - b1 m_{t-1}) / (1 - b1).
 * Errors: SCAPE_EINVAL for an unknown flag.
 */
enum scape_variant {
    SCAPE_VARIANT_PAPER = 0,
    SCAPE_VARIANT_DENSE_OFFMASK = 1,
    SCAPE_VARIANT_MOMENT_SYNC = 2
};
int scape_set_variant(scape_t *h, int flags);

/*
 * How much of the step the compaction pass does (results are bit-identical
 * at every level).  The compaction sees every worker of a tile, so it can
 * form the synchronised buffer while the residuals stream through:
 *   SCAPE_FUSE_NONE    the ordered sum of the W packed buffers and the
 *       unpack + AdamS run as two separate launches after it, the layout of
 *       "Sintesi Tecnica: SCAPE" Sec. 2;
 *   SCAPE_FUSE_SUM     the compaction also writes g_bar (worker-ordered
 *       sum / W); the unpack + AdamS runs as its own launch;
 *   SCAPE_FUSE_UPDATE  the compaction also applies AdamS at the selected
 *       coordinates (no further launch; its w and m accesses interleave with
 *       the residual stream).
 * Default, set by scape_create / scape_create_range from the handle's own
 * k and P: SCAPE_FUSE_UPDATE when at least 5% of the coordinates are
 * selected (20 k >= P; with W <= 2 workers 0.5%: 200 k >= P) and not all of
 * them, SCAPE_FUSE_SUM otherwise.
 * The packed buffers and g_bar are written at every level.
 * scape_get_fusion writes the current level to *level.
 * Errors: SCAPE_EINVAL for an unknown level or a NULL pointer.
 */
enum scape_fusion { SCAPE_FUSE_NONE = 0, SCAPE_FUSE_SUM = 1, SCAPE_FUSE_UPDATE = 2 };
int scape_set_fusion(scape_t *h, int level);
int scape_get_fusion(const scape_t *h, int *level);

/*
 * Device staging for residuals bound in host memory (the pages keep the
 * error-feedback buffers on the CPU side, "SCAPE" Sec. I).  With a staging
 * buffer bound, every sparse scape_step() moves the residuals through it in
 * worker groups of rows/3: one group copies in on an internal stream while
 * the previous one is compacted on `stream` and the one before copies its
 * updated residuals back on a second internal stream, so both directions of
 * the host link are in use and the compaction reads HBM.  Without one (NULL
 * or 0 bytes, the default) the kernels access host residuals in place.
 * Ignored while the residuals are device memory; the dense first step,
 * scape_step_host() and the union baseline always access them in place.
 * scape_residual_staging_bytes() gives the size for `rows` residual rows
 * (rows >= 3; each row is P floats rounded up to 64).
 *   device_buffer  caller-owned device memory, 16-byte aligned
 * Errors: SCAPE_EINVAL if the buffer is misaligned or holds fewer than 3 rows.
 */
int scape_residual_staging_bytes(const scape_t *h, int rows, size_t *bytes);
int scape_set_residual_staging(scape_t *h, void *device_buffer, size_t bytes);

/*
 * Dense baselines the pages compare SCAPE against ("SCAPE" abstract, Sec. I),
 * on the handle's bound w and m: the gradient is the plain ordered mean of
 * the W workers' gradients (no error feedback, no mask; residuals untouched)
 * and every coordinate is updated:
 *   scape_dense_adams_step  AdamS of "SCAPE" Sec. II-C, Eq. 2;
 *   scape_adamw_step        AdamW, v_t = b2 v_{t-1} + (1 - b2) g^2 in the
 *                           caller's float32 v[P] (zero it before step 1).
 * Both use and advance the handle's step count t for the bias corrections.
 * Errors as scape_step().
 */
int scape_dense_adams_step(scape_t *h, const void *const *host_grad_ptrs, void *stream);
int scape_adamw_step(scape_t *h, const void *const *host_grad_ptrs, float *v, void *stream);

/*
 * Union-mask gradient top-k baseline: the second synchronisation scheme of
 * "SCAPE" Sec. II-B, which the partitioned mask is designed against.  Each
 * worker selects the k_w = ceil(P (1 - sparsity)) largest |g^w + e^w| over the
 * whole vector (ties to the lower index); the W masks are OR-ed into their
 * union (the mask all-gather); every worker sends its error-fed gradient at
 * every union position (the all-reduce over the global mask), so its residual
 * becomes a - a there and g + e elsewhere; AdamS ("SCAPE" Sec. II-C) runs on
 * the ordered mean at the union positions, others unchanged.  The union grows
 * with W (fill-in); its size is returned in *host_k_union.
 *   workspace  caller device memory of scape_union_workspace_bytes(capacity)
 *              bytes, 256-byte aligned; it keeps per-worker selection state
 *              between calls (a new pointer starts it afresh)
 *   capacity   the largest union the packed buffers hold, 1..P (P never
 *              overflows).  A larger union returns SCAPE_EINVAL after the
 *              selection, with the residuals holding g + e: do not retry.
 * Synchronises `stream` once (to read the union size).  Uses and advances the
 * handle's step count; the SCAPE mask state is not touched.
 */
int scape_union_workspace_bytes(const scape_t *h, int64_t capacity, size_t *bytes);
int scape_union_step(scape_t *h, const void *const *host_grad_ptrs, void *workspace,
                     size_t ws_bytes, int64_t capacity, int64_t *host_k_union, void *stream);

/*
 * Whether the steady warm refresh is replayed as a CUDA graph (default on).
 * Once the warm-up widening of the bucket windows is over, every warm
 * scape_refresh_mask() enqueues the same launches with the same arguments;
 * the first such call captures them (and the rebuild of the index list) into
 * a graph on an internal stream and later calls launch that graph on
 * `stream`, which saves the launch gaps of its ~20 small kernels.  Calls made
 * while profiling brackets any refresh kernel, or while `stream` is being
 * captured by the caller, enqueue the launches themselves.  scape_bind()
 * drops the graph.
 */
int scape_set_graphs(scape_t *h, int on);

/* Learning rate for subsequent steps (schedules).  lr must be finite. */
int scape_set_lr(scape_t *h, float lr);

/*
 * Current state: t = steps taken, k, and device pointers (inside the bound
 * workspace) to the mask bitmap (ceil(P/32) words) and the packed index list
 * (k uint32, ascending) that the NEXT step will use.  Pointers stay valid
 * until re-bind.  Any output may be NULL.
 */
int scape_get_state(const scape_t *h, int64_t *t, int64_t *k, const uint32_t **bits,
                    const uint32_t **idx);

/*
 * Device pointers to the last step's packed buffers (W rows of k floats,
 * row w at pack + w * (*pack_stride)) and to the synchronised buffer g_bar
 * (k floats).  Valid after a step t >= 2 (step 1 is dense and packs nothing).
 */
int scape_get_buffers(const scape_t *h, const float **pack, int64_t *pack_stride,
                      const float **gbar);

/*
 * Resume from a checkpoint: set the step count t (>= 1) and the mask the next
 * step uses from a caller bitmap (ceil(P/32) words, device), then rebuild the
 * index list and rank table.  Synchronises `stream`; returns SCAPE_EINVAL if
 * the bitmap does not hold exactly k_s set bits in each shard or has bits set
 * past P.  Parameters, m and residuals are the caller's buffers: restore them
 * before the next step.
 */
int scape_set_state(scape_t *h, int64_t t, const uint32_t *bits, void *stream);

/*
 * End-to-end step from host memory: copy each worker's gradient from host
 * memory (pinned for asynchronous copies) into the caller's device gradient
 * buffers, run scape_step() and scape_refresh_mask(), then copy w[P] back to
 * host_params_out.  From step 2 on, the uploads run on an internal copy stream
 * in up to 16 worker groups and each group's compaction starts on `stream` as
 * soon as its gradients have landed.  When host_params_out is page-locked and
 * only the selected coordinates change (the default reading), w is downloaded
 * on a second internal stream while the gradients upload (the previous
 * parameters) and a kernel then writes the k updated values into
 * host_params_out through its device address; otherwise w is downloaded after
 * the update, overlapping the mask refresh.  Either way host_params_out ends
 * holding all P parameters after the step.  All of the call's work is ordered
 * before later work on `stream`: synchronise `stream` before reading
 * host_params_out or reusing the host gradient buffers.  The first call
 * creates the internal streams and their events.
 */
int scape_step_host(scape_t *h, const void *const *host_grads_src,
                    void *const *host_dev_grad_ptrs, float *host_params_out, void *stream);

/*
 * Per-kernel timing.  With profiling on, every kernel launch is bracketed by
 * CUDA events on its stream.  scape_profile_collect() waits for the recorded
 * events, adds their durations to per-kernel totals and clears the record;
 * scape_profile_read() copies the totals (milliseconds and launch counts,
 * SCAPE_NUM_KERNELS entries each) and scape_kernel_name() names entry i.
 */
#define SCAPE_NUM_KERNELS 25
int scape_profile_enable(scape_t *h, int on);
/* Which kernels profiling brackets: bit i for kernel i (default: all).  Two
 * event records per launch cost the GPU a few microseconds; a timing run can
 * keep them to the kernels it reports. */
int scape_profile_select(scape_t *h, uint32_t kernel_mask);
int scape_profile_collect(scape_t *h);
int scape_profile_read(const scape_t *h, double *host_ms, int64_t *host_launches);
int scape_profile_reset(scape_t *h);
const char *scape_kernel_name(int i);

/* Total kernel launches made through this handle since creation. */
int64_t scape_launch_count(const scape_t *h);

/*
 * A timing probe of the GPU, not a step of the method: the memory accesses of
 * the sparse update -- the index list and the synchronised buffer read in
 * order, w[i] and m[i] read and written back at the k coordinates of the
 * current mask -- without its arithmetic.  w and m are left bit for bit as
 * they were.  Its time is the floor the scattered update can reach on this
 * GPU (the accesses are scattered 4-byte reads and writes, bound by the rate
 * of random DRAM accesses rather than by bytes).  Profiled as "probe_rmw".
 * Errors: SCAPE_ESTATE before a mask exists.
 */
int scape_probe_random_access(scape_t *h, void *stream);

/*
 * Per-shard top-k mask that allocates nothing.  The SCAPE pages have no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc where they need a mask -- code running inside a custom device
 * allocator or memory-pool callback (allocating would re-enter it), plug-ins
 * handed only input and output buffers, loops that cannot take cudaMalloc's
 * implicit device synchronisation -- and so cannot supply the workspace of
 * scape_bind().
 *
 * Computes the same mask as scape_refresh_mask() does for a handle with this
 * P, W and sparsity: bits[ceil(P/32)] (bit i % 32 of word i / 32) and the
 * ascending index list idx[k], k = sum_s k_s.  m (float32, P, 16-byte
 * aligned), bits and idx are the caller's device buffers.  Scratch lives in
 * one fixed __device__ array inside the library (under 1 MiB, held by every
 * GPU that loads the library until the process exits); no call allocates
 * device or host memory.  All calls share that array and it keeps the last
 * call's contents: calls that overlap on the GPU race and must be ordered by
 * the caller.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for the life
 * of the process; make that first call before any stream capture.  The kept
 * address belongs to the device's current context: after cudaDeviceReset()
 * on that device, do not call this entry point again in the same process.
 * Limits: 1 <= P <= SCAPE_STATIC_MAX_P, 1 <= W <= SCAPE_STATIC_MAX_WORKERS;
 * larger sizes, NULL pointers, a misaligned m or sparsity outside [0, 1)
 * return SCAPE_EINVAL without touching the GPU; CUDA failures return
 * SCAPE_ECUDA.  Work is enqueued on `stream`.
 */
#define SCAPE_STATIC_MAX_P (1LL << 26)
#define SCAPE_STATIC_MAX_WORKERS 64
int scape_topk_mask_static(const float *m, int64_t P, int W, double sparsity, uint32_t *bits,
                           uint32_t *idx, void *stream);

/*
 * ---------------------------------------------------------------------------
 * Several data-parallel ranks with a real exchange.
 *
 * Rank `rank` of G owns the workers and the optimizer shards [a, b),
 * a = floor(W rank / G), b = floor(W (rank + 1) / G), of the problem
 * scape_create() would lay out for these layers and W (one optimizer shard
 * per worker: "SCAPE" Sec. II-A, sharded data parallelism with a distributed
 * optimizer).  The rank holds a full replica of the parameters w[P], the first
 * moment of its own parameter range [lo, hi) (the shards it owns), and for
 * each of its b - a workers the full-length gradient and residual.  Every
 * step is cut around three collectives that the caller runs (NCCL, gloo, ...)
 * on the buffers scape_xc_buffers() returns, with the element counts of
 * scape_xc_counts():
 *   1. scape_xc_pack(): error feedback and compaction of the local workers
 *      with the lagged global mask ("SCAPE" Sec. II-B), laid out in the send
 *      buffer as one contiguous block per destination rank q (rows: local
 *      workers in order; columns: q's selected coordinates, padded to a
 *      multiple of 4).
 *   2. caller: all-to-all with those per-rank counts, send -> recv.  recv then
 *      holds the W workers' rows of the owned columns in worker order: the
 *      sparse reduce-scatter of "SCAPE" Sec. I, its sum taken by the owner in
 *      worker order so that every G gives the one-device result bit for bit.
 *   3. scape_xc_update(): the ordered mean of the W rows and AdamS at the
 *      owned selected coordinates ("SCAPE" Sec. II-C, Eq. 2; "Sintesi
 *      Tecnica: SCAPE" Sec. 2, one synchronised buffer), the updated values
 *      copied to param_send.
 *   4. caller: all-gather param_send -> param_recv (rank q's values at row q,
 *      params_per_rank[q] of them, row stride param_stride): the sparse
 *      parameter all-gather ("SCAPE" Sec. I).
 *   5. scape_xc_refresh(): the next mask of the owned shards from their first
 *      moment ("Sintesi Tecnica: SCAPE" Sec. 2, partitioned mask), aligned to
 *      the global 32-bit word grid in mask_send (words floor(lo/32) ..).
 *   6. caller: all-gather mask_send -> mask_recv (mask_words_per_rank[q]
 *      words at row q, stride mask_stride).  Steps 4 and 6 may overlap: the
 *      mask is only used by the next step (the one-step lag of "Sintesi
 *      Tecnica: SCAPE" Sec. 2).
 *   7. scape_xc_finish(): the other ranks' updated parameters written into w,
 *      the gathered words merged into the global mask and its index list
 *      rebuilt for the next step.
 * Step 1 is dense (every coordinate is sent and every parameter gathered).
 * All work is enqueued on `stream`; the caller orders its collectives after
 * the previous call's work (e.g. on the same stream, or after synchronising).
 * Calls out of this order return SCAPE_ESTATE.  The handle never allocates
 * device memory: the caller binds one workspace of the size scape_xc_layout()
 * reports, which holds the exchange buffers (the dense first step needs about
 * 2 (b - a) P + W (hi - lo) floats of them).
 * ---------------------------------------------------------------------------
 */
typedef struct scape_xc scape_xc_t;

/* Host only.  Errors: as scape_create(), and SCAPE_EINVAL unless
 * 1 <= G <= W and 0 <= rank < G. */
int scape_xc_create(scape_xc_t **out, int n_layers, const int64_t *host_layer_numel, int W,
                    int G, int rank, double sparsity, float beta1, float beta2, float lr,
                    float eps, float weight_decay, int grad_dtype);
void scape_xc_destroy(scape_xc_t *h);
const char *scape_xc_last_error(const scape_xc_t *h);

/* P, global k, local workers b - a, the owned range [own_begin, own_end) and
 * its k, and the workspace bytes.  Any output may be NULL. */
int scape_xc_layout(const scape_xc_t *h, int64_t *P, int64_t *k, int *local_workers,
                    int64_t *own_begin, int64_t *own_end, int64_t *own_k, size_t *ws_bytes);

/*
 * Bind caller memory: params w[P] (the replica, 16-byte aligned), m_own
 * (own_end - own_begin floats, zeroed, 16-byte aligned), host array of b - a
 * residual pointers (each P floats, zeroed, 16-byte aligned), the workspace
 * (256-byte aligned).  Resets the step count.
 */
int scape_xc_bind(scape_xc_t *h, float *params, float *m_own, float *const *host_e_ptrs,
                  void *workspace, size_t ws_bytes);

/* Element counts of the coming (or current) step's collectives, per rank q:
 * floats sent to q and received from q in the all-to-all; the parameter and
 * mask-word all-gathers' per-rank counts and row strides.  Any output may be
 * NULL (arrays have G entries). */
int scape_xc_counts(const scape_xc_t *h, int64_t *host_send_counts, int64_t *host_recv_counts,
                    int64_t *params_per_rank, int64_t *param_stride,
                    int64_t *mask_words_per_rank, int64_t *mask_stride);

/* Device pointers of the exchange buffers inside the bound workspace, and of
 * the global mask bitmap (ceil(P/32) words) the next step uses.  SCAPE_ESTATE
 * before scape_xc_bind().  Any output may be NULL. */
int scape_xc_buffers(const scape_xc_t *h, float **send, float **recv, float **param_send,
                     float **param_recv, uint32_t **mask_send, uint32_t **mask_recv,
                     const uint32_t **global_bits);

/* The four phases of a step (see above).  host_grad_ptrs: b - a device
 * pointers, the local workers' gradients g^w[P] of the handle's dtype. */
int scape_xc_pack(scape_xc_t *h, const void *const *host_grad_ptrs, void *stream);
int scape_xc_update(scape_xc_t *h, void *stream);
int scape_xc_refresh(scape_xc_t *h, void *stream);
int scape_xc_finish(scape_xc_t *h, void *stream);

/* Steps completed and the owned shards' current mask bitmap and index list
 * (local coordinates: bit i is parameter own_begin + i). */
int scape_xc_get_state(const scape_xc_t *h, int64_t *t, const uint32_t **own_bits,
                       const uint32_t **own_idx);

/* Resume after t >= 1 completed steps from a checkpoint: `global_bits` (device,
 * ceil(P/32) words) is the global mask the next step uses -- the bitmap behind
 * the global_bits buffer of scape_xc_buffers() when the checkpoint was taken,
 * the same on every rank; w, m_own and the residuals are the caller's
 * (restored by the caller before the next step).  The owned shards' part is
 * checked (SCAPE_EINVAL if a shard does not hold exactly k_s set bits); the
 * next refresh of the owned shards is a cold one.  Call between steps.
 * Errors: SCAPE_EINVAL (t < 1, NULL bitmap, wrong counts), SCAPE_ESTATE (not
 * bound, or a step in progress), SCAPE_ECUDA. */
int scape_xc_set_state(scape_xc_t *h, int64_t t, const uint32_t *global_bits, void *stream);

/* Kernel launches made through this handle. */
int64_t scape_xc_launch_count(const scape_xc_t *h);

#ifdef __cplusplus
}
#endif

#endif /* SCAPE_H */
