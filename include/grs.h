/*
 * grs.h — ownership-aware sharded gradient reduction and AdamW for GB300.
 *
 * C ABI of libgrs.so.  Plain pointers and sizes only: host pointers are
 * marked "host", device pointers "device".  Every entry point returns a
 * grs_status; on failure a thread-local message is available from
 * grs_last_error().  Nothing here synchronises with the host except
 * grs_check_device_errors(), and nothing allocates device memory except
 * grs_plan_create() (its small tables and error flags).
 *
 * The operation follows these web pages (cited by title and section):
 *   [ISSUE]  "refactor(distributed): establish shared native TP replica
 *            ownership" (NeMo Automodel issue) — "Why this needs separate
 *            work" (the four owner semantics), "Preserved prototype and
 *            evidence" (FP32 reduction hook, accumulation, clipping),
 *            "Proposed scope and acceptance criteria" (one reduction owner
 *            per parameter; reject unsupported compositions).
 *   [COSMOS] "Cosmos 3 training framework > distributed parallelism" —
 *            section 1 (dp_shard / dp_replicate; -1 = whole world;
 *            dp_replicate x dp_shard = world), section 2 (2x4 dp_mesh:
 *            all-reduce across replicas, all-gather across shards).
 *   [MIXLE]  "Distributed Transformer Training" (Mixle integration note) —
 *            "Backend split" (fail before fitting), "Optimizer and
 *            checkpoint semantics" (routes planned from logical parameters
 *            before wrapping; Adam state).
 *
 * Simulated ranks.  The R = world ranks of a tp x dp_replicate x dp_shard
 * job are buffers in one GPU's memory.  Rank index of mesh coordinate
 * (replica r, shard s, tensor-parallel index t):
 *     rank = (r * dp_shard + s) * tp + t
 * ([COSMOS] section 2: replica 0 holds g0..g3, so replicas are the slow
 * axis; the tp index is innermost).
 *
 * Layouts (all element counts, not bytes):
 *   per-rank gradient buffer  bf16 [n_rank_pad]: the buckets' per-rank
 *       slices back to back; bucket b occupies [rank_offset, +padded).
 *       A LOCAL_SHARD tensor contributes numel/tp elements per rank: rank
 *       with tp index t holds the t-th contiguous chunk of the row-major
 *       logical tensor.
 *   state (accumulator, fp32 master, first and second moment, bf16
 *       parameters) [n_state_pad]: per bucket, `copies` rows of `padded`
 *       elements at state_offset (copies = tp for LOCAL_SHARD: row t holds
 *       the reduction over the ranks of tp index t; 1 otherwise).  Each
 *       row splits into dp_shard contiguous shards of shard_len elements:
 *       shard s is what rank (r, s, t) owns after the reduce-scatter.
 *   Padding (bucket element index >= used) is ignored on input, may hold
 *       anything (NaN included), and is written as exact zeros in every
 *       output.
 *
 * Concurrency.  A plan does not change after grs_plan_create except for its
 * device error flags and the copy stream and events that grs_step_from_host
 * creates on first use.  Calls on one plan may come from several host
 * threads and streams as long as the buffers they write do not overlap on
 * the GPU; the error flags are shared, so grs_check_device_errors reports
 * (and clears) a flag raised by any call on the plan.  grs_step_from_host
 * calls on one plan must not overlap each other (they share the plan's copy
 * stream and events).  Separate plans share nothing but the allocation-free
 * norm's static scratch.
 */
#ifndef GRS_H
#define GRS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GRS_MAX_WORLD 128

/* Owner tag of a parameter ([ISSUE] "Why this needs separate work").
 *  GRS_REPLICA_AVG      complete gradients from redundant computation:
 *                       averaged across TP (and DP)             scale 1/R
 *  GRS_PARTIAL_SUM      partial contributions (head/sequence sharding):
 *                       summed across TP, averaged across DP    scale 1/dp
 *  GRS_LOCAL_SHARD      TP/EP/model-owned shard: never synchronised across
 *                       TP, averaged over its own DP group      scale 1/dp
 *  GRS_ALREADY_REDUCED  reduced by another owner: never reduced again;
 *                       rank 0's copy is taken as is            scale 1   */
typedef enum grs_owner {
  GRS_REPLICA_AVG = 0,
  GRS_PARTIAL_SUM = 1,
  GRS_LOCAL_SHARD = 2,
  GRS_ALREADY_REDUCED = 3
} grs_owner;

typedef enum grs_status {
  GRS_OK = 0,
  GRS_ERR_INVALID_ARG = 1,              /* null/out-of-range argument       */
  GRS_ERR_UNSUPPORTED_COMPOSITION = 2,  /* degrees do not compose to world  */
  GRS_ERR_SHAPE = 3,                    /* numel < 0, LOCAL_SHARD % tp != 0 */
  GRS_ERR_ALIGNMENT = 4,                /* device pointer not 16-B aligned  */
  GRS_ERR_CUDA = 5,                     /* CUDA runtime error (message set) */
  GRS_ERR_TIMEOUT = 6,                  /* a bounded device wait gave up    */
  GRS_ERR_NONFINITE = 7,                /* global gradient norm is NaN/Inf  */
  GRS_ERR_NO_DEVICE = 8,                /* plan was created host-only       */
  GRS_ERR_BOUNDS = 9                    /* checked build: an index left its buffer (library bug) */
} grs_status;

/* grs_plan_create flags */
#define GRS_PLAN_HOST_ONLY 1u  /* build host tables only (queries work, launches fail) */
#define GRS_PLAN_FP32_GRADS 2u /* rank gradients are fp32 instead of bf16 ([ISSUE] "Proposed
                                  scope": BF16/FP32); same layout, 4-byte elements */

/* per-tensor flags (grs_plan_create_ex) */
#define GRS_TENSOR_FROZEN 1u /* no gradient and no optimizer state: left out of the plan */

typedef struct grs_plan grs_plan; /* opaque; owned by the caller via create/destroy */

typedef struct grs_plan_info {
  int32_t n_tensors;
  int32_t n_buckets;
  int32_t world;          /* R */
  int32_t tp;
  int32_t dp_replicate;
  int32_t dp_shard;       /* resolved (never -1) */
  int32_t dp;             /* dp_replicate * dp_shard */
  int32_t device;         /* CUDA device of the tables, -1 when host-only */
  int64_t n_unique;       /* N: logical parameter elements */
  int64_t n_rank_pad;     /* elements of each rank's gradient buffer */
  int64_t n_state_pad;    /* elements of accumulator / master / m / v / params */
  int64_t workspace_bytes;/* device workspace needed by reduce / norm calls; zero it once */
  int64_t n_reduce_tiles; /* norm partial slots (one per reduction tile) */
  int32_t grad_bytes;     /* bytes per gradient element: 2 (bf16) or 4 (fp32) */
  int32_t reserved;
} grs_plan_info;

typedef struct grs_bucket_desc {
  int32_t tag;            /* grs_owner of every tensor in the bucket */
  int32_t copies;         /* state rows: tp for LOCAL_SHARD, else 1 */
  int32_t group_size;     /* ranks reduced per output element (R, dp or 1) */
  int32_t n_tensors;
  int64_t used;           /* per-rank elements holding tensor data */
  int64_t padded;         /* per-rank elements incl. padding (multiple of 8*dp_shard) */
  int64_t shard_len;      /* padded / dp_shard */
  int64_t rank_offset;    /* offset of the bucket in each rank buffer */
  int64_t state_offset;   /* offset of row 0 in the state arrays */
  int32_t n_segments;     /* copies * n_tensors (see grs_segment_info) */
  int32_t reserved;
} grs_bucket_desc;

/* One segment of a bucket: the part of one tensor that lives in one state
 * row of the bucket (a LOCAL_SHARD tensor has one segment per tp rank, any
 * other tensor one).  Segments tile each row's [0, used) back to back. */
typedef struct grs_segment_desc {
  int32_t tensor;         /* index in the plan's tensor list */
  int32_t tp_index;       /* state row: the tp rank for LOCAL_SHARD buckets, else 0 */
  int64_t bucket_offset;  /* element offset inside the bucket row (the same in every rank buffer) */
  int64_t tensor_offset;  /* element offset inside the tensor's row-major flattening */
  int64_t numel;          /* elements in the segment */
  int64_t state_offset;   /* absolute offset in the state arrays and the full-parameter buffer */
} grs_segment_desc;

typedef struct grs_tensor_desc {
  int32_t bucket;         /* -1 for a frozen tensor */
  int32_t owner;
  int64_t numel;          /* logical elements */
  int64_t per_rank;       /* numel/tp for LOCAL_SHARD, else numel (0 when frozen) */
  int64_t bucket_offset;  /* element offset inside the bucket (per rank and per state row) */
  uint32_t flags;         /* GRS_TENSOR_* as given to grs_plan_create_ex */
  uint32_t reserved;
} grs_tensor_desc;

/* AdamW hyper-parameters (decoupled weight decay, Loshchilov & Hutter;
 * the form torch.optim.AdamW documents) and clipping. */
typedef struct grs_adamw {
  float lr;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  float max_norm;         /* <= 0: clipping off */
  int32_t step;           /* 1-based index of this update (bias correction) */
  int32_t n_micro;        /* M: the accumulator holds the sum of M microbatches */
} grs_adamw;

/* ---------------------------------------------------------------- plan */

/* Build the reduction plan from the logical parameter list, in model order
 * ([MIXLE] "Optimizer and checkpoint semantics": routes planned from
 * stable logical parameters before wrapping).
 *   numels, owners : host arrays [n_tensors]; owners are grs_owner values.
 *   world          : number of simulated ranks, 1..GRS_MAX_WORLD.
 *   tp, dp_replicate, dp_shard : degrees; dp_shard = -1 resolves to
 *                    world / (tp * dp_replicate) ([COSMOS] section 1).
 *   bucket_bytes   : cap on a bucket's per-rank bf16 bytes; a tensor larger
 *                    than the cap gets a bucket of its own.
 *   flags          : GRS_PLAN_HOST_ONLY (no device tables; without it they go
 *                    to the current CUDA device) and/or GRS_PLAN_FP32_GRADS
 *                    (rank gradient buffers hold fp32; every "bf16 bits"
 *                    gradient pointer below then points at floats).
 * Buckets hold one owner tag each, in tag order REPLICA_AVG, PARTIAL_SUM,
 * LOCAL_SHARD, ALREADY_REDUCED, model order inside a tag, filled greedily,
 * tensors packed back to back, padded to a multiple of 8 * dp_shard.
 * Errors (nothing is launched or allocated; [MIXLE] "Backend split": fail
 * before fitting; [ISSUE] "Proposed scope": reject unsupported
 * compositions): n_tensors <= 0, bad tag, bucket_bytes <= 0, a degree <= 0
 * (dp_shard may be -1) -> INVALID_ARG; tp*dp_replicate*dp_shard != world
 * -> UNSUPPORTED_COMPOSITION; numel < 0 or LOCAL_SHARD numel % tp != 0 ->
 * SHAPE; device table upload failure -> CUDA.  *out is set only on OK. */
grs_status grs_plan_create(const int64_t* numels, const int32_t* owners, int32_t n_tensors,
                           int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                           int64_t bucket_bytes, uint32_t flags, grs_plan** out);

/* grs_plan_create with per-tensor flags ([ISSUE] "Proposed scope": frozen
 * parameters and EP/model-owned exclusions).  tensor_flags: host array
 * [n_tensors] of GRS_TENSOR_* bits, or NULL.  A GRS_TENSOR_FROZEN tensor
 * keeps its index but gets no bucket, no rank-buffer space and no state:
 * it is never reduced, clipped, updated or gathered.  Unknown bits ->
 * INVALID_ARG. */
grs_status grs_plan_create_ex(const int64_t* numels, const int32_t* owners, const uint32_t* tensor_flags,
                              int32_t n_tensors, int32_t world, int32_t tp, int32_t dp_replicate,
                              int32_t dp_shard, int64_t bucket_bytes, uint32_t flags, grs_plan** out);

/* The shard view of rank (r, shard, tp_index): a plan, destroyed with
 * grs_plan_destroy, whose state layout is what that rank owns after the
 * reduce-scatter ([COSMOS] section 2: rank (r, s) of the dp_mesh holds shard
 * s of every parameter, replicas r hold the same shard): per bucket b, in
 * bucket order, shard_len elements — elements [shard * shard_len,
 * (shard + 1) * shard_len) of row tp_index for LOCAL_SHARD buckets, of row 0
 * for the others (every tp rank keeps its own copy of those).  A job that
 * runs one rank per GPU brings the rank's reduced gradient shard into this
 * layout with its own collectives (reduce-scatter over the shard group,
 * all-reduce across replicas, per [COSMOS] section 2); the view then gives
 * the rank-local steps:
 *   grs_grad_norm_sq (partials_ready = 0): the squared norm over the
 *     elements this rank holds uniquely within its tp group (LOCAL_SHARD
 *     rows always, the other rows only at tp_index 0), so that the sum over
 *     all (shard, tp_index) views of one replica is the global S — the one
 *     scalar all-reduce of the norm;
 *   grs_accumulate: microbatch accumulation of reduced shards;
 *   grs_clip_adamw_step: clip + AdamW + bf16 cast of the shard, bit for bit
 *     the plan's own update restricted to these elements (given the same S),
 *     whose bf16 shards an all-gather over the shard group reassembles.
 * grs_plan_query reports the view's n_state_pad (the sum of the slices),
 * n_unique (the elements it counts in the norm), workspace_bytes and
 * n_rank_pad = 0; grs_bucket_info describes each slice (copies 1, padded =
 * used-or-padding extent = shard_len, used = its valid elements,
 * state_offset in the view).  Entry points that need rank gradient buffers
 * or the tensor layout (reductions, gather, masked calls, layout conversion,
 * grs_step_from_host, grs_segment_info, grs_update_small) return
 * UNSUPPORTED_COMPOSITION for a view.  The view's device tables go to the
 * parent's device (none for a host-only parent).
 * Errors: INVALID_ARG (NULL, shard or tp_index out of range, a view as the
 * parent), CUDA. */
grs_status grs_plan_shard_view(const grs_plan* plan, int32_t shard, int32_t tp_index, grs_plan** out);

/* Free the plan and its device tables.  NULL is a no-op.  The caller must
 * ensure no launch using the plan is still in flight. */
void grs_plan_destroy(grs_plan* plan);

/* Plan queries (host only; no CUDA call). */
grs_status grs_plan_query(const grs_plan* plan, grs_plan_info* out);
grs_status grs_bucket_info(const grs_plan* plan, int32_t bucket, grs_bucket_desc* out);
grs_status grs_tensor_info(const grs_plan* plan, int32_t tensor, grs_tensor_desc* out);
/* Segment i of bucket b, 0 <= i < n_segments, in state-memory order: row
 * t = i / n_tensors, then the bucket's tensors by increasing offset
 * ([COSMOS] section 2: a LOCAL_SHARD tensor's tp slices are its dim-0
 * chunks, rank t's chunk in row t).  Index out of range -> INVALID_ARG. */
grs_status grs_segment_info(const grs_plan* plan, int32_t bucket, int32_t segment, grs_segment_desc* out);

/* ---------------------------------------------------------- hot path */

/* Reduce one bucket of one microbatch: for every output element e of every
 * row of bucket b,
 *     acc[e] (= | +=) scale(tag) * sum_{k in group} float(g_k[e])
 * in fp32 with ranks k in ascending order ([ISSUE] "Preserved prototype":
 * FP32 reduction of BF16 gradients; "Why this needs separate work": the
 * group and scale come from the owner tag).  This is the reduce-scatter of
 * the bucket over dp_shard plus the all-reduce over dp_replicate plus the
 * TP reduction ([COSMOS] section 2), all shards computed.
 *   rank_grads : host array [world] of device pointers; rank_grads[k]
 *                points at rank k's copy of THIS bucket ([padded] elements,
 *                bf16 bits, or fp32 for GRS_PLAN_FP32_GRADS plans).  Only the ranks of the tag's group are
 *                read (ALREADY_REDUCED reads rank 0 only).
 *   acc        : device fp32 [copies * padded]: this bucket's state rows.
 *   accumulate : 0 overwrite (first microbatch), 1 add (later ones).
 *   emit_norm_partials : 1 on the last microbatch: also write the bucket's
 *                per-tile sums of acc^2 into the workspace, so that
 *                grs_grad_norm_sq needs no second pass over acc.
 *   workspace  : device, >= workspace_bytes, zero-filled once before its
 *                first use (the library leaves its counter at zero after
 *                every call); required when emitting.
 * Errors: INVALID_ARG, ALIGNMENT (every pointer 16-B aligned), NO_DEVICE,
 * CUDA (launch failure). */
grs_status grs_reduce_bucket(const grs_plan* plan, int32_t bucket, const void* const* rank_grads,
                             float* acc, int32_t accumulate, int32_t emit_norm_partials,
                             void* workspace, void* stream);

/* grs_reduce_bucket for overlap with the backward pass ([ISSUE] "Preserved
 * prototype": asynchronous FP32 reduction hook; "Proposed scope": overlap
 * during backward): buckets become ready one by one (in reverse model
 * order during backward) and each is reduced as soon as its gradients
 * exist, on a side stream, while the backward pass goes on.
 *   wait_event : a cudaEvent_t recorded after the bucket's gradients were
 *                written (on the producing stream), or NULL; `stream`
 *                waits for it before the reduction.
 *   max_ctas   : cap on the reduction's persistent grid (0 = one CTA per
 *                SM), leaving the other SMs to concurrent kernels.
 * Results (accumulator and norm partials) do not depend on the grid: they
 * are bit-identical to grs_reduce_bucket / grs_reduce_all. */
grs_status grs_reduce_bucket_ex(const grs_plan* plan, int32_t bucket, const void* const* rank_grads,
                                float* acc, int32_t accumulate, int32_t emit_norm_partials,
                                void* workspace, int32_t max_ctas, void* wait_event, void* stream);

/* The same for every bucket in one launch.
 *   rank_grads : host array [world] of device pointers to each rank's
 *                whole gradient buffer ([n_rank_pad], bf16 bits or fp32).
 *   acc        : device fp32 [n_state_pad]. */
grs_status grs_reduce_all(const grs_plan* plan, const void* const* rank_grads, float* acc,
                          int32_t accumulate, int32_t emit_norm_partials, void* workspace,
                          void* stream);

/* grs_reduce_all for a step where some tensors have no gradient (PyTorch's
 * grad None; [ISSUE] "Proposed scope": unused parameters), for use with
 * grs_grad_norm_sq_masked and grs_clip_adamw_step_masked.  d_tensor_used:
 * device uint8 [n_tensors], as for those calls.  Reduction tiles that lie
 * wholly inside one tensor with used = 0 are neither read nor written, so
 * those tensors' gradients need not exist; every other tile is reduced as
 * grs_reduce_all reduces it (tiles spanning several tensors in full).  The
 * accumulator of a tensor with used = 0 is therefore unspecified: the
 * masked norm and update never use it.
 *   emit_norm_partials : 1 on the last microbatch to write, into
 *                        `workspace`, the per-tile partials of the MASKED
 *                        norm (elements of tensors with used = 0 count as
 *                        zero; skipped tiles give +0), bit-identical to
 *                        those of grs_grad_norm_sq_masked.  Then
 *                        grs_grad_norm_sq(..., partials_ready = 1, ...)
 *                        gives grs_grad_norm_sq_masked's S bit for bit
 *                        without a pass over acc.
 *   workspace          : as for grs_reduce_bucket; may be NULL when
 *                        emit_norm_partials = 0.
 * Errors as grs_reduce_all, INVALID_ARG for a NULL mask, SHAPE beyond
 * 32768 reduction tiles per SM. */
grs_status grs_reduce_all_masked(const grs_plan* plan, const void* const* rank_grads, float* acc,
                                 int32_t accumulate, int32_t emit_norm_partials,
                                 const uint8_t* d_tensor_used, void* workspace, void* stream);

/* acc_b += mb_b over bucket b's rows (fp32), padding kept at zero: adds a
 * separately reduced microbatch gradient into the accumulator ([ISSUE]
 * "Proposed scope": gradient accumulation).  Both device [copies*padded]. */
grs_status grs_accumulate(const grs_plan* plan, int32_t bucket, float* acc, const float* mb,
                          void* stream);

/* Global squared gradient norm S = sum_e (acc[e]/n_micro)^2 over every
 * unique element (each state element once; LOCAL_SHARD rows each count;
 * padding is zero), kept on the device in *d_norm_sq ([ISSUE] "Proposed
 * scope": global norms for clipping).  Deterministic: fixed tiles, fixed
 * summation trees, fp32 inside a tile and fp64 across tiles.
 *   acc            : device fp32 [n_state_pad] (read unless partials_ready).
 *   partials_ready : 1 when every bucket's last reduce emitted its
 *                    partials into `workspace` (no pass over acc).
 *   d_norm_sq      : device double [1].
 *   workspace      : as for grs_reduce_bucket (zero-filled before first use).
 * Calls sharing one workspace must not overlap on the GPU.
 * A non-finite S raises the device flag reported as NONFINITE by
 * grs_check_device_errors; the step still proceeds (NaN propagates). */
grs_status grs_grad_norm_sq(const grs_plan* plan, const float* acc, int32_t n_micro,
                            void* workspace, int32_t partials_ready, double* d_norm_sq,
                            void* stream);

/* Clip + AdamW + bf16 cast, fused, over all n_state_pad elements:
 *   c = min(1, max_norm / (sqrt(S) + 1e-6))   (1 when max_norm <= 0)
 *   g = c * acc / n_micro
 *   p = p*(1 - lr*wd); m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*g^2
 *   p = p - lr/(1-b1^step) * m / (sqrt(v)/sqrt(1-b2^step) + eps)
 *   params_bf16 = round-to-nearest-even(p)
 * ([ISSUE] "Proposed scope": clipping on/off, optimizer updates; AdamW per
 * Loshchilov & Hutter as torch.optim.AdamW documents it).  S is read on
 * the device: no host synchronisation.  The bf16 output is written in the
 * bucket-ordered full-parameter layout, i.e. the all-gathered parameters
 * ([COSMOS] section 2).
 *   hp        : host struct.  d_norm_sq: device double (may be NULL when
 *               max_norm <= 0).  acc: device fp32 (read only).  master, m,
 *               v: device fp32, updated in place.  params_bf16: device
 *               bf16 bits.  All [n_state_pad].
 * Errors: INVALID_ARG (step < 1, n_micro < 1, NULL), ALIGNMENT, NO_DEVICE,
 * CUDA. */
grs_status grs_clip_adamw_step(const grs_plan* plan, const grs_adamw* hp, const double* d_norm_sq,
                               const float* acc, float* master, float* m, float* v,
                               uint16_t* params_bf16, void* stream);

/* grs_clip_adamw_step with the gather fused in: the same update, and every
 * bf16 parameter written straight into its own tensor's storage, as
 * grs_gather_params would copy it there from the bucket-ordered buffer
 * ([COSMOS] section 2: the parameters all-gathered across shards for the
 * forward; LOCAL_SHARD tensors reassembled from their tp rows in dim-0
 * order).  One pass instead of two: the bucket-ordered copy need not exist.
 *   params_bf16   : device bf16 bits [n_state_pad] also written in the
 *                   bucket-ordered layout, or NULL (per-tensor output only).
 *   d_tensor_ptrs : DEVICE array [n_tensors] of device pointers (8-byte
 *                   aligned), entry i pointing at tensor i's numel bf16
 *                   elements (2-byte aligned; 16-byte-aligned destinations
 *                   are written with 16-byte stores); NULL entries and frozen
 *                   tensors are skipped.  The entries live in device memory,
 *                   so the library cannot check them: the caller guarantees
 *                   their extent and alignment.  The kernel reads the table,
 *                   so it must stay valid until the launch has run.
 * The other arguments, the results in master, m, v (and params_bf16) and
 * the errors are those of grs_clip_adamw_step; ALIGNMENT also when the
 * table is not 8-byte aligned.  The tensors must not overlap each other or
 * the state. */
grs_status grs_clip_adamw_step_to_tensors(const grs_plan* plan, const grs_adamw* hp, const double* d_norm_sq,
                                          const float* acc, float* master, float* m, float* v,
                                          uint16_t* params_bf16, uint16_t* const* d_tensor_ptrs,
                                          void* stream);

/* Tensors without a gradient this step (PyTorch's grad None; [ISSUE]
 * "Proposed scope": unused parameters).  d_tensor_used: device uint8
 * [n_tensors], 1 = the tensor's rank-buffer region holds this step's
 * gradient, 0 = no gradient.
 *
 * grs_grad_norm_sq_masked: like grs_grad_norm_sq with partials_ready = 0,
 * but elements of tensors with used = 0 count as zero (clip_grad_norm_
 * skips parameters without a gradient): a separate pass over acc.  After a
 * grs_reduce_all_masked that emitted its norm partials, the same S comes
 * from grs_grad_norm_sq(..., partials_ready = 1, ...) without that pass.
 *
 * grs_clip_adamw_step_masked: like grs_clip_adamw_step for tensors with
 * used = 1, each with its own step count: d_tensor_steps (device int32
 * [n_tensors], zero before the first update, updated in place) is advanced
 * for used tensors and its new value sets their bias correction.  hp->step
 * is only a hint (0 = none): tensors whose new step equals it take factors
 * computed on the host, exactly those of grs_clip_adamw_step at that step;
 * the others' factors are computed on the device in fp64 (the same values
 * up to the last bit of the fp32 factor, more slowly).  Tensors with
 * used = 0 keep master, m, v, the bf16 copy and
 * their step count unchanged (torch.optim.AdamW skips parameters without a
 * gradient: no moment decay, no weight decay).  Entries of frozen tensors
 * are ignored.  workspace as for the norm (the per-tensor factors live
 * after the norm's part).  Padding stays exactly zero. */
grs_status grs_grad_norm_sq_masked(const grs_plan* plan, const float* acc, int32_t n_micro,
                                   const uint8_t* d_tensor_used, void* workspace, double* d_norm_sq,
                                   void* stream);
grs_status grs_clip_adamw_step_masked(const grs_plan* plan, const grs_adamw* hp, const double* d_norm_sq,
                                      const float* acc, float* master, float* m, float* v,
                                      uint16_t* params_bf16, const uint8_t* d_tensor_used,
                                      int32_t* d_tensor_steps, void* workspace, void* stream);

/* ------------------------------------------ single-launch small plans */

#define GRS_SMALL_MAX_TILES 128   /* reduction tiles (grs_plan_info.n_reduce_tiles), and bucket rows */
#define GRS_SMALL_MAX_BUFFERS 256 /* n_micro x world gradient buffers */

/* The whole update of a small plan in one kernel launch: the reductions of
 * hp->n_micro microbatches (as grs_reduce_all with accumulate = j > 0),
 * the global squared norm (as grs_grad_norm_sq) and clip + AdamW + bf16
 * cast (as grs_clip_adamw_step), with the same arithmetic in the same
 * order, so every output equals the three calls' bit for bit ([ISSUE]
 * "Preserved prototype and evidence", "Proposed scope": FP32 reduction,
 * accumulation, clipping, optimizer update).  For plans whose four
 * launches cost more than their memory traffic: one thread-block cluster
 * of 16 CTAs, the norm partials exchanged through distributed shared
 * memory.
 *   rank_grads : host array [n_micro * world] of device pointers,
 *                microbatch-major (buffer j * world + k is rank k's
 *                gradients of microbatch j), each [n_rank_pad] bf16 bits (fp32
 *                for GRS_PLAN_FP32_GRADS plans), 16-byte aligned, non-NULL.
 *   acc, master, m, v : device fp32 [n_state_pad]; acc is written (the
 *                accumulated gradient sum), master, m, v updated in place.
 *   params_bf16: device bf16 bits [n_state_pad], written.
 *   d_norm_sq  : device double, written (S of grs_grad_norm_sq); required.
 * No workspace.  Errors: INVALID_ARG (NULL, step or n_micro < 1), SHAPE
 * (more than GRS_SMALL_MAX_TILES reduction tiles or bucket rows, or more
 * than GRS_SMALL_MAX_BUFFERS gradient buffers: use the multi-kernel path),
 * ALIGNMENT, NO_DEVICE, CUDA.
 * A non-finite norm raises the flag grs_check_device_errors reports. */
grs_status grs_update_small(const grs_plan* plan, const grs_adamw* hp, const void* const* rank_grads,
                            float* acc, float* master, float* m, float* v, uint16_t* params_bf16,
                            double* d_norm_sq, void* stream);

/* Gather: copy every tensor from the bucket-ordered bf16 parameter buffer
 * to its own full logical tensor ([COSMOS] section 2: all-gather of
 * parameters across shards; LOCAL_SHARD tensors reassembled from their tp
 * rows in dim-0 order).
 *   params_bf16 : device [n_state_pad].
 *   tensor_ptrs : host array [n_tensors] of device pointers, each to
 *                 numel bf16 elements; NULL entries (and frozen tensors)
 *                 are skipped.  Any 2-byte alignment is accepted. */
grs_status grs_gather_params(const grs_plan* plan, const uint16_t* params_bf16,
                             uint16_t* const* tensor_ptrs, void* stream);

/* One whole update from host-resident gradients ([ISSUE] "Preserved
 * prototype": asynchronous FP32 reduction hook; "Proposed scope": overlap
 * during backward).  Per microbatch and bucket: the bucket's rank rows are
 * copied host->device on the plan's own copy stream (one cudaMemcpyAsync per
 * rank read by the owner group; ALREADY_REDUCED copies rank 0 only) while the
 * previous bucket is reduced on `stream`; then the norm finish, clip + AdamW
 * + bf16 cast, and (optionally) the bf16 parameters and the squared norm are
 * copied back to the host.  Same results as the device-buffer calls.
 *   hp            : host struct; hp->n_micro microbatches.
 *   host_grads    : host array [n_micro * world] of HOST pointers (pinned
 *                   memory for full speed), microbatch-major (j*world + k),
 *                   each [n_rank_pad] bf16 bits (fp32 for FP32_GRADS plans).
 *   dev_stage     : host array [2 * world] of device pointers (only the
 *                   first `world` are used when n_micro == 1), each
 *                   [n_rank_pad] gradient elements, 16-byte aligned: two staging halves
 *                   alternating across microbatches.
 *   acc, master, m, v, params_bf16, workspace, d_norm_sq : as for the
 *                   device calls.
 *   host_params   : host [n_state_pad] bf16 bits, or NULL (no read-back).
 *   host_norm_sq  : host double [1], or NULL.
 * The host buffers must stay valid until `stream` has run the call's work;
 * the read-backs are complete after the caller synchronises `stream`.  The
 * first call creates the plan's copy stream and events (freed by
 * grs_plan_destroy) and its copies wait for all work queued on `stream`
 * before; later calls' copies wait only for the previous call's reductions,
 * so consecutive steps overlap (step N+1's host-to-device copies run during
 * step N's update and read-back).  The staging buffers therefore belong to
 * these calls: do not touch them on other streams in between.  Errors:
 * INVALID_ARG, ALIGNMENT, NO_DEVICE, CUDA. */
grs_status grs_step_from_host(const grs_plan* plan, const grs_adamw* hp,
                              const void* const* host_grads, void* const* dev_stage,
                              float* acc, float* master, float* m, float* v, uint16_t* params_bf16,
                              void* workspace, double* d_norm_sq, uint16_t* host_params,
                              double* host_norm_sq, void* stream);

/* ------------------------------------------------- allocation-free variant */

/* Size of the library's own scratch array for grs_grad_norm_sq_noalloc. */
#define GRS_NOALLOC_SCRATCH_BYTES (4u << 20)

/* The pages have no counterpart to this entry point: it is a convenience
 * for callers that cannot allocate device memory — e.g. a process whose
 * framework caching allocator already holds (nearly) all of the GPU's
 * memory, latency-critical code that cannot take the device synchronisation
 * an allocation may cause, or a host that only receives device pointers
 * from another runtime.
 *
 * Computes the same global squared norm as grs_grad_norm_sq with
 * partials_ready = 0 (a pass over the accumulator, then the fixed-order
 * fp64 finish; bit-identical results) but needs no workspace: the scratch
 * is a file-scope device array of GRS_NOALLOC_SCRATCH_BYTES (4 MiB) that
 * every GPU loading the library holds until the process exits.
 *   acc       : device fp32 [n_state_pad] (read).
 *   d_norm_sq : device double [1] (written).
 * The caller passes the input and the output; nothing is allocated (no
 * cudaMalloc/cudaFree, no allocating library call).  The first call on a
 * device looks up the array's device address with that device current;
 * make that first call before any stream capture.  The address is kept for
 * the life of the process: after cudaDeviceReset (which unloads the
 * library's device code with the context) it is stale, so do not call this
 * entry point again in a process that has reset the device.  All calls share the
 * array and it keeps the last call's contents (its counter is cleared on
 * the stream before each launch); calls that overlap on the GPU — from two
 * streams or two threads — race and must be serialised by the caller.
 * Errors: INVALID_ARG (NULL, n_micro < 1), ALIGNMENT, NO_DEVICE, SHAPE when
 * the plan needs more scratch than the array holds (more than about a
 * million reduction tiles; the message gives both sizes), CUDA. */
grs_status grs_grad_norm_sq_noalloc(const grs_plan* plan, const float* acc, int32_t n_micro,
                                    double* d_norm_sq, void* stream);

/* Validation of ALREADY_REDUCED buckets ([ISSUE] "Why this needs separate
 * work": an existing reduction must not be applied again, so the data it
 * produced must already agree everywhere): compares every rank's copy of
 * every ALREADY_REDUCED bucket with rank 0's, bit for bit, over the valid
 * elements.  rank_grads as for grs_reduce_all (whole per-rank buffers).  A
 * mismatch raises a device flag that the next grs_check_device_errors
 * reports as GRS_ERR_INVALID_ARG. */
grs_status grs_check_already_reduced(const grs_plan* plan, const void* const* rank_grads, void* stream);

/* Failure-detection self-test: one kernel waits on an mbarrier that nothing
 * completes, through the same bounded wait the reduction uses, gives up
 * after limit_ns (1 us .. 2 s) and raises the plan's timeout flag; a
 * following grs_check_device_errors returns GRS_ERR_TIMEOUT and the CUDA
 * context stays usable ([MIXLE] "Backend split": failures surface as
 * errors, not hangs). */
grs_status grs_selftest_bounded_wait(const grs_plan* plan, int64_t limit_ns, void* stream);

/* Layout conversion of an fp32 state array (master, m, v or the
 * accumulator) between the plan's bucket layout [n_state_pad] and the
 * canonical logical order [n_unique]: every live (not frozen) tensor in
 * model order, each over its full logical extent (a LOCAL_SHARD tensor's tp
 * rows concatenated in dim-0 order).  The logical order does not depend on
 * tp, dp_replicate, dp_shard, owner tags or bucket size, so a checkpoint
 * written under one plan restores exactly under another: state_to_logical
 * with the writer's plan, state_from_logical with the reader's ([ISSUE]
 * "Preserved prototype": checkpoints restored exactly across ownership
 * changes, matching the next Adam update; [MIXLE] "Optimizer and checkpoint
 * semantics").  state_from_logical writes every padding element as 0.
 * Both pointers are device memory, 4-byte aligned. */
grs_status grs_state_to_logical(const grs_plan* plan, const float* state, float* logical, void* stream);
grs_status grs_state_from_logical(const grs_plan* plan, const float* logical, float* state, void* stream);

/* Synchronise `stream`, read and clear the plan's device flags.  Returns
 * BOUNDS if a checked build (below) found an index outside its buffer,
 * TIMEOUT if a bounded device wait gave up, NONFINITE if a global norm was
 * NaN/Inf since the last check, INVALID_ARG if grs_check_already_reduced
 * found copies that differ, else OK (or CUDA). */
grs_status grs_check_device_errors(const grs_plan* plan, void* stream);

/* Build features of the loaded library.  GRS_FEATURE_CHECKED: compiled with
 * GRS_CHECKED=1 — every kernel checks each index it derives against the
 * extent of the buffer it addresses (the sizes this header documents for
 * that call) before the access; a failed check skips the access and raises
 * a device flag that grs_check_device_errors reports as BOUNDS (the message
 * names the kernel).  Slower; for tests and debugging. */
#define GRS_FEATURE_CHECKED 1u
uint32_t grs_build_features(void);

/* Message of the last failing call on this thread ("" if none). */
const char* grs_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* GRS_H */
