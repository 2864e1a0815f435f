/*
 * CPU oracle: plain scalar fp64 definition of ownership-aware gradient
 * reduction, reduce-scatter, microbatch accumulation, global-norm clipping,
 * AdamW and the bf16 cast.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h for the sources and the pins).
 * Nothing here is blocked, fused or reordered beyond what the definition
 * states; every loop runs in plain index order.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Parallel degrees.
 * [COSMOS] section 1: dp_replicate x dp_shard = world (the DP world: tensor
 * parallelism is not one of that descriptor's axes, so with TP the
 * invariant reads tp x dp_replicate x dp_shard = number of ranks);
 * dp_shard = -1 takes whatever the other degrees leave.
 * ------------------------------------------------------------------------ */
int oracle_resolve_dims(int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                        int32_t* dims) {
  if (world <= 0 || tp <= 0 || dp_replicate <= 0) return OR_ERR_INVALID_ARG;
  if (dp_shard == -1) {
    if (world % (tp * dp_replicate) != 0) return OR_ERR_UNSUPPORTED_COMPOSITION;
    dp_shard = world / (tp * dp_replicate);
  }
  if (dp_shard <= 0) return OR_ERR_INVALID_ARG;
  if ((int64_t)tp * dp_replicate * dp_shard != world) return OR_ERR_UNSUPPORTED_COMPOSITION;
  dims[0] = dp_shard;
  dims[1] = dp_replicate * dp_shard;
  dims[2] = world;
  return OR_OK;
}

/* Mesh coordinate -> rank.  [COSMOS] section 2: in the 2x4 dp_mesh the
 * ranks of replica 0 are g0..g3 (shards 0..3), replica 1 is g4..g7, so the
 * replica index is the slow axis and the shard index the fast one.  The
 * tensor-parallel index is placed innermost (the pages do not place it). */
int32_t oracle_rank(int32_t r, int32_t s, int32_t t, int32_t dp_shard, int32_t tp) {
  return (r * dp_shard + s) * tp + t;
}

/* ------------------------------------------------------------------------
 * Bucket plan.
 * [MIXLE] "Optimizer and checkpoint semantics": optimizer routes are planned
 * from the stable logical parameter list before any wrapping, so the plan
 * is a pure function of (numel, owner) in model order.
 * [ISSUE] "Proposed scope": exactly one reduction owner per parameter, and
 * unsupported compositions are rejected ([MIXLE] "Backend split": fail
 * before fitting).  Reading of the unspecified bucket layout:
 *   - tensors are grouped by owner tag in the order REPLICA_AVG,
 *     PARTIAL_SUM, LOCAL_SHARD, ALREADY_REDUCED, keeping model order inside
 *     a tag, so every bucket has one owner;
 *   - buckets fill greedily on per-rank bf16 bytes: a tensor opens a new
 *     bucket when it would push a non-empty bucket past bucket_bytes; a
 *     tensor is never split;
 *   - a LOCAL_SHARD tensor holds numel/tp elements per rank (its rank's
 *     contiguous dim-0 chunk); numel % tp != 0 is a shape error;
 *   - a bucket is padded to a multiple of 8 * dp_shard elements and split
 *     into dp_shard equal contiguous shards ([COSMOS] section 1: each
 *     shard holds 1/dp_shard of parameters, gradients and optimizer state);
 *   - per-rank buffers concatenate the buckets; the state (accumulator,
 *     master, moments, bf16 parameters) concatenates, per bucket, one copy
 *     per output: tp copies for LOCAL_SHARD (one per tp index), else one.
 * ------------------------------------------------------------------------ */
int oracle_plan(const int64_t* numel, const int32_t* owner, int32_t n,
                int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                int64_t bucket_bytes, int32_t max_buckets,
                int32_t* dims, int32_t* t_bucket, int64_t* t_offset,
                int32_t* b_tag, int64_t* b_padded, int64_t* b_used,
                int64_t* b_rank_off, int64_t* b_state_off) {
  return oracle_plan_ex(numel, owner, 0, n, world, tp, dp_replicate, dp_shard, bucket_bytes,
                        max_buckets, dims, t_bucket, t_offset, b_tag, b_padded, b_used, b_rank_off,
                        b_state_off);
}

/* The plan with per-tensor flags ([ISSUE] "Proposed scope": frozen
 * parameters).  A frozen tensor (flag bit 1) has no gradient and no
 * optimizer state: it is left out of every bucket (t_bucket = -1). */
int oracle_plan_ex(const int64_t* numel, const int32_t* owner, const uint32_t* flags, int32_t n,
                   int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                   int64_t bucket_bytes, int32_t max_buckets,
                   int32_t* dims, int32_t* t_bucket, int64_t* t_offset,
                   int32_t* b_tag, int64_t* b_padded, int64_t* b_used,
                   int64_t* b_rank_off, int64_t* b_state_off) {
  int32_t d[3];
  int st, i, tag, nb = 0;
  if (n <= 0 || numel == 0 || owner == 0) return OR_ERR_INVALID_ARG;
  if (bucket_bytes <= 0) return OR_ERR_INVALID_ARG;
  st = oracle_resolve_dims(world, tp, dp_replicate, dp_shard, d);
  if (st != OR_OK) return st;
  for (i = 0; i < n; ++i) {
    if (owner[i] < 0 || owner[i] > 3) return OR_ERR_INVALID_ARG;
    if (numel[i] < 0) return OR_ERR_SHAPE;
    if (owner[i] == OR_LOCAL_SHARD && numel[i] % tp != 0) return OR_ERR_SHAPE;
    if (flags && (flags[i] & ~(uint32_t)OR_TENSOR_FROZEN)) return OR_ERR_INVALID_ARG;
  }
  for (i = 0; i < n; ++i) {
    t_bucket[i] = -1;
    t_offset[i] = 0;
  }
  for (tag = 0; tag < 4; ++tag) {
    int open = 0;
    int64_t used = 0;
    for (i = 0; i < n; ++i) {
      int64_t per_rank;
      if (owner[i] != tag) continue;
      if (flags && (flags[i] & OR_TENSOR_FROZEN)) continue;
      per_rank = (tag == OR_LOCAL_SHARD) ? numel[i] / tp : numel[i];
      if (open && used > 0 && 2 * (used + per_rank) > bucket_bytes) {
        b_used[nb - 1] = used;
        open = 0;
      }
      if (!open) {
        if (nb >= max_buckets) return OR_ERR_INVALID_ARG;
        b_tag[nb] = tag;
        ++nb;
        open = 1;
        used = 0;
      }
      t_bucket[i] = nb - 1;
      t_offset[i] = used;
      used += per_rank;
    }
    if (open) b_used[nb - 1] = used;
  }
  {
    int b;
    int64_t quantum = 8 * (int64_t)d[0];
    int64_t rank_off = 0, state_off = 0;
    for (b = 0; b < nb; ++b) {
      int64_t copies = (b_tag[b] == OR_LOCAL_SHARD) ? tp : 1;
      b_padded[b] = (b_used[b] + quantum - 1) / quantum * quantum;
      b_rank_off[b] = rank_off;
      b_state_off[b] = state_off;
      rank_off += b_padded[b];
      state_off += copies * b_padded[b];
    }
  }
  dims[0] = d[0];
  dims[1] = d[1];
  dims[2] = d[2];
  dims[3] = nb;
  return OR_OK;
}

/* bf16 bit pattern -> value (bf16 is the top half of an IEEE binary32). */
static double bf16_value(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------------
 * Reduction of one bucket, all microbatches.
 * [ISSUE] "Why this needs separate work":
 *   REPLICA_AVG      redundant full computation -> complete gradients,
 *                    averaged across TP;
 *   PARTIAL_SUM      head/sequence-sharded partial contributions, summed
 *                    across TP;
 *   LOCAL_SHARD      TP/EP/model-owned shards, never synchronised as
 *                    replicas; "Preserved prototype": DP-only ownership;
 *   ALREADY_REDUCED  already reduced by another owner: never reduced again
 *                    (the value of the canonical rank 0 is taken as is).
 * Across data parallelism every tag but ALREADY_REDUCED is averaged:
 * all-reduce across dp_replicate replicas and reduce-scatter over dp_shard
 * ([COSMOS] section 2).  The reduce-scatter leaves shard s of the bucket's
 * output (elements [s*P/Ds, (s+1)*P/Ds)) on shard s; since every shard is
 * a slice of the one output, the oracle writes the whole output.
 * Microbatches ([ISSUE] "Proposed scope": gradient accumulation) are summed;
 * the mean over microbatches is taken where the gradient is used.
 * ------------------------------------------------------------------------ */
/* Value of input element `i` of a gradient array, as fp64. */
typedef double (*grad_value_fn)(const void* grads, int64_t i);

static double value_bf16(const void* grads, int64_t i) {
  return bf16_value(((const uint16_t*)grads)[i]);
}

static double value_f32(const void* grads, int64_t i) {
  return (double)((const float*)grads)[i];
}

static int reduce_core(int32_t tag, int32_t tp, int32_t dp_replicate, int32_t dp_shard, int64_t P,
                       int64_t used, int32_t M, const void* grads, grad_value_fn value, double* acc) {
  int32_t R = tp * dp_replicate * dp_shard;
  int32_t dp = dp_replicate * dp_shard;
  int32_t copies = (tag == OR_LOCAL_SHARD) ? tp : 1;
  int32_t c, j, r, s, t;
  int64_t e;
  if (tag < 0 || tag > 3 || M <= 0 || P < 0 || used < 0 || used > P) return OR_ERR_INVALID_ARG;
  for (c = 0; c < copies; ++c) {
    for (e = 0; e < P; ++e) {
      double total = 0.0;
      if (e >= used) {
        acc[(int64_t)c * P + e] = 0.0;
        continue;
      }
      for (j = 0; j < M; ++j) {
        int64_t mb = (int64_t)j * R * P; /* first element of microbatch j */
        double dp_sum = 0.0;
        double reduced;
        if (tag == OR_ALREADY_REDUCED) {
          reduced = value(grads, mb + (int64_t)oracle_rank(0, 0, 0, dp_shard, tp) * P + e);
        } else {
          for (r = 0; r < dp_replicate; ++r) {
            for (s = 0; s < dp_shard; ++s) {
              double tp_value;
              if (tag == OR_LOCAL_SHARD) {
                /* no tensor-parallel reduction: this rank's own shard */
                tp_value = value(grads, mb + (int64_t)oracle_rank(r, s, c, dp_shard, tp) * P + e);
              } else {
                double tp_sum = 0.0;
                for (t = 0; t < tp; ++t)
                  tp_sum += value(grads, mb + (int64_t)oracle_rank(r, s, t, dp_shard, tp) * P + e);
                tp_value = (tag == OR_REPLICA_AVG) ? tp_sum / tp : tp_sum;
              }
              dp_sum += tp_value;
            }
          }
          reduced = dp_sum / dp;
        }
        total += reduced;
      }
      acc[(int64_t)c * P + e] = total;
    }
  }
  return OR_OK;
}

int oracle_reduce_bucket(int32_t tag, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                         int64_t P, int64_t used, int32_t M, const uint16_t* grads,
                         double* acc) {
  return reduce_core(tag, tp, dp_replicate, dp_shard, P, used, M, grads, value_bf16, acc);
}

/* The same with fp32 gradients ([ISSUE] "Proposed scope": BF16/FP32). */
int oracle_reduce_bucket_f32(int32_t tag, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                             int64_t P, int64_t used, int32_t M, const float* grads, double* acc) {
  return reduce_core(tag, tp, dp_replicate, dp_shard, P, used, M, grads, value_f32, acc);
}

/* Global squared norm of G = acc/M ([ISSUE] "Proposed scope": compare global
 * norms; clipping uses the norm of the whole gradient, every unique element
 * once). */
double oracle_norm_sq(const double* acc, int64_t n, int32_t M) {
  double s = 0.0;
  int64_t e;
  for (e = 0; e < n; ++e) {
    double g = acc[e] / M;
    s += g * g;
  }
  return s;
}

/* Clip coefficient, the clip_grad_norm_ rule: c = min(1, max/(||G|| + 1e-6)).
 * A NaN norm gives a NaN coefficient (clamping does not hide it). */
double oracle_clip_coef(double norm_sq, double max_norm) {
  double c;
  if (!(max_norm > 0.0)) return 1.0;
  c = max_norm / (sqrt(norm_sq) + 1e-6);
  if (isnan(c)) return c;
  return c < 1.0 ? c : 1.0;
}

/* Round-to-nearest-even fp32 -> bf16: add half an ulp of the kept part,
 * plus one when the kept part is odd, then truncate. */
uint16_t oracle_bf16_rne(float x) {
  uint32_t w;
  memcpy(&w, &x, sizeof w);
  if ((w & 0x7f800000u) == 0x7f800000u && (w & 0x007fffffu) != 0)
    return (uint16_t)((w >> 16) | 0x0040u); /* quiet NaN */
  w += 0x7fffu + ((w >> 16) & 1u);
  return (uint16_t)(w >> 16);
}

/* ------------------------------------------------------------------------
 * AdamW on one unit (Loshchilov & Hutter, decoupled weight decay; the form
 * of torch.optim.AdamW), with the clipped, microbatch-averaged gradient:
 *   g  = c * acc / M
 *   p  = p * (1 - lr * wd)
 *   m  = b1 * m + (1 - b1) * g
 *   v  = b2 * v + (1 - b2) * g^2
 *   p  = p - lr / (1 - b1^t) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)
 * fp64 throughout from the fp32 state; outputs rounded to fp32 and the new
 * parameter additionally to bf16 ([ISSUE] "Proposed scope": compare
 * optimizer updates; [MIXLE] "Optimizer and checkpoint semantics").
 * Padding elements (index >= used) are written as exact zeros.
 * ------------------------------------------------------------------------ */
void oracle_adamw(int64_t n, int64_t used, const double* acc, int32_t M, double c,
                  const double* hp, int32_t step,
                  const float* master0, const float* m0, const float* v0,
                  float* master1, float* m1, float* v1, uint16_t* param_bf16) {
  double lr = hp[0], b1 = hp[1], b2 = hp[2], eps = hp[3], wd = hp[4];
  double bc1 = 1.0 - pow(b1, step);
  double bc2 = 1.0 - pow(b2, step);
  int64_t e;
  for (e = 0; e < n; ++e) {
    double g, p, m, v;
    if (e >= used) {
      master1[e] = 0.0f;
      m1[e] = 0.0f;
      v1[e] = 0.0f;
      param_bf16[e] = 0;
      continue;
    }
    g = c * (acc[e] / M);
    p = (double)master0[e];
    m = (double)m0[e];
    v = (double)v0[e];
    p = p * (1.0 - lr * wd);
    m = b1 * m + (1.0 - b1) * g;
    v = b2 * v + (1.0 - b2) * g * g;
    p = p - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps);
    master1[e] = (float)p;
    m1[e] = (float)m;
    v1[e] = (float)v;
    param_bf16[e] = oracle_bf16_rne((float)p);
  }
}

/* Gather one tensor back to its full logical layout ([COSMOS] section 2:
 * parameters are all-gathered across shards for the forward).  A
 * LOCAL_SHARD tensor is the concatenation of its tp chunks, chunk t living
 * in bucket copy t. */
void oracle_gather_tensor(int64_t numel, int32_t owner, int32_t tp, int64_t bucket_state_off,
                          int64_t bucket_padded, int64_t tensor_offset,
                          const uint16_t* params_full, uint16_t* dst) {
  int64_t i;
  if (owner == OR_LOCAL_SHARD) {
    int64_t chunk = numel / tp;
    int32_t t;
    for (t = 0; t < tp; ++t)
      for (i = 0; i < chunk; ++i)
        dst[t * chunk + i] =
            params_full[bucket_state_off + (int64_t)t * bucket_padded + tensor_offset + i];
  } else {
    for (i = 0; i < numel; ++i) dst[i] = params_full[bucket_state_off + tensor_offset + i];
  }
}

/* fp32 state of one tensor, bucket layout <-> its full logical extent (the
 * same placement as oracle_gather_tensor), for checkpoints ([ISSUE]
 * "Preserved prototype": exact restore across ownership changes). */
void oracle_gather_tensor_f32(int64_t numel, int32_t owner, int32_t tp, int64_t bucket_state_off,
                              int64_t bucket_padded, int64_t tensor_offset, const float* state,
                              float* dst) {
  int64_t i;
  if (owner == OR_LOCAL_SHARD) {
    int64_t chunk = numel / tp;
    int32_t t;
    for (t = 0; t < tp; ++t)
      for (i = 0; i < chunk; ++i)
        dst[t * chunk + i] = state[bucket_state_off + (int64_t)t * bucket_padded + tensor_offset + i];
  } else {
    for (i = 0; i < numel; ++i) dst[i] = state[bucket_state_off + tensor_offset + i];
  }
}

void oracle_scatter_tensor_f32(int64_t numel, int32_t owner, int32_t tp, int64_t bucket_state_off,
                               int64_t bucket_padded, int64_t tensor_offset, const float* src,
                               float* state) {
  int64_t i;
  if (owner == OR_LOCAL_SHARD) {
    int64_t chunk = numel / tp;
    int32_t t;
    for (t = 0; t < tp; ++t)
      for (i = 0; i < chunk; ++i)
        state[bucket_state_off + (int64_t)t * bucket_padded + tensor_offset + i] = src[t * chunk + i];
  } else {
    for (i = 0; i < numel; ++i) state[bucket_state_off + tensor_offset + i] = src[i];
  }
}
