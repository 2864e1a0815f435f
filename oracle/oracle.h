/*
 * CPU oracle for ownership-aware sharded gradient reduction + clip + AdamW.
 *
 * TEST INFRASTRUCTURE ONLY.  This header and oracle.c form a plain, slow,
 * scalar fp64 restatement of what the GPU path computes.  It shares no code,
 * header, table or constant with the CUDA library; only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * Sources (web pages, cited by title and section):
 *   [ISSUE]  "refactor(distributed): establish shared native TP replica
 *            ownership" (NeMo Automodel issue): sections "Why this needs
 *            separate work", "Preserved prototype and evidence",
 *            "Proposed scope and acceptance criteria".
 *   [COSMOS] "Cosmos 3 training framework > distributed parallelism":
 *            section 1 (the four ParallelDims axes) and section 2 (the
 *            world=8 dp_mesh figure).
 *   [MIXLE]  "Distributed Transformer Training" (Mixle frontier integration
 *            note): sections "Backend split", "Optimizer and checkpoint
 *            semantics".
 *   AdamW is not written out on any page; the oracle uses decoupled weight
 *   decay (Loshchilov & Hutter, "Decoupled Weight Decay Regularization",
 *   2019, Algorithm 2) in the form torch.optim.AdamW documents, and the
 *   clipping rule of torch.nn.utils.clip_grad_norm_.
 *
 * Parity pins: every function here is pinned by a CPU test against values
 * fixed by the pages or by mathematics (hand-checked brute force, closed
 * forms, torch.optim.AdamW, clip_grad_norm_, real gloo collectives).
 */
#ifndef GRS_ORACLE_H
#define GRS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Owner tags ([ISSUE], "Why this needs separate work", four bullets). */
enum { OR_REPLICA_AVG = 0, OR_PARTIAL_SUM = 1, OR_LOCAL_SHARD = 2, OR_ALREADY_REDUCED = 3 };

/* Status values, numbered as the library documents its status codes. */
enum {
  OR_OK = 0,
  OR_ERR_INVALID_ARG = 1,
  OR_ERR_UNSUPPORTED_COMPOSITION = 2,
  OR_ERR_SHAPE = 3
};

/* Resolve the parallel degrees.  world = tp * dp_replicate * dp_shard;
 * dp_shard = -1 means "the rest of the world" ([COSMOS] section 1: -1 takes
 * the full world).  Writes dims[0] = dp_shard, dims[1] = dp, dims[2] = R. */
int oracle_resolve_dims(int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                        int32_t* dims);

/* Bucket plan.  Inputs: n tensors (numel, owner) in model order.
 * Outputs (caller-allocated):
 *   dims[4]        = dp_shard, dp, R, n_buckets
 *   t_bucket[n]    = bucket of tensor i
 *   t_offset[n]    = element offset of tensor i inside its bucket (per rank)
 *   b_tag[nb], b_padded[nb], b_used[nb], b_rank_off[nb], b_state_off[nb]
 * `max_buckets` bounds the bucket arrays. */
int oracle_plan(const int64_t* numel, const int32_t* owner, int32_t n,
                int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                int64_t bucket_bytes, int32_t max_buckets,
                int32_t* dims, int32_t* t_bucket, int64_t* t_offset,
                int32_t* b_tag, int64_t* b_padded, int64_t* b_used,
                int64_t* b_rank_off, int64_t* b_state_off);

/* Tensor flag: frozen (no gradient, no state). */
enum { OR_TENSOR_FROZEN = 1 };

/* oracle_plan with per-tensor flags (NULL = none); frozen tensors get
 * t_bucket = -1 and no space anywhere. */
int oracle_plan_ex(const int64_t* numel, const int32_t* owner, const uint32_t* flags, int32_t n,
                   int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                   int64_t bucket_bytes, int32_t max_buckets,
                   int32_t* dims, int32_t* t_bucket, int64_t* t_offset,
                   int32_t* b_tag, int64_t* b_padded, int64_t* b_used,
                   int64_t* b_rank_off, int64_t* b_state_off);

/* Rank index of mesh coordinate (replica r, shard s, tensor-parallel t). */
int32_t oracle_rank(int32_t r, int32_t s, int32_t t, int32_t dp_shard, int32_t tp);

/* Reduce one bucket over all microbatches.
 * grads: [M][R][P] bf16 bit patterns (microbatch-major, then rank).
 * acc:   [copies][P] fp64 output, copies = tp for LOCAL_SHARD else 1,
 *        acc = sum over microbatches of the reduced per-microbatch gradient.
 * Elements at index >= used (padding) are ignored on input and 0 on output. */
int oracle_reduce_bucket(int32_t tag, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                         int64_t P, int64_t used, int32_t M, const uint16_t* grads,
                         double* acc);

/* The same with fp32 gradients: grads is [M][R][P] float. */
int oracle_reduce_bucket_f32(int32_t tag, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                             int64_t P, int64_t used, int32_t M, const float* grads, double* acc);

/* Sum of (acc[e]/M)^2 over n values, fp64, in index order. */
double oracle_norm_sq(const double* acc, int64_t n, int32_t M);

/* Clip coefficient from the global squared norm; max_norm <= 0: off (1). */
double oracle_clip_coef(double norm_sq, double max_norm);

/* One AdamW step over n elements of one unit (bucket copy).  g = c*acc/M.
 * Elements at index >= used are padding: every output there is exactly 0.
 * hp = {lr, beta1, beta2, eps, weight_decay}; step is 1-based. */
void oracle_adamw(int64_t n, int64_t used, const double* acc, int32_t M, double c,
                  const double* hp, int32_t step,
                  const float* master0, const float* m0, const float* v0,
                  float* master1, float* m1, float* v1, uint16_t* param_bf16);

/* Round fp32 to bf16, round-to-nearest-even; NaN stays NaN. */
uint16_t oracle_bf16_rne(float x);

/* Gather tensor i of the plan from the bucket-ordered full parameter
 * buffer (length = total state elements) into dst[numel]. */
void oracle_gather_tensor(int64_t numel, int32_t owner, int32_t tp, int64_t bucket_state_off,
                          int64_t bucket_padded, int64_t tensor_offset,
                          const uint16_t* params_full, uint16_t* dst);

/* fp32 state of one tensor: bucket layout -> logical (gather) and back
 * (scatter; padding untouched). */
void oracle_gather_tensor_f32(int64_t numel, int32_t owner, int32_t tp, int64_t bucket_state_off,
                              int64_t bucket_padded, int64_t tensor_offset, const float* state,
                              float* dst);
void oracle_scatter_tensor_f32(int64_t numel, int32_t owner, int32_t tp, int64_t bucket_state_off,
                               int64_t bucket_padded, int64_t tensor_offset, const float* src,
                               float* state);

#ifdef __cplusplus
}
#endif
#endif
