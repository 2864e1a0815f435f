// C-ABI entry points of libgrs: argument checks ("fail before fitting"),
// device table upload, stream-ordered launches, device flag readback.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>
#include <string>

#include "internal.h"

namespace {

thread_local std::string g_last_error;

grs_status fail(grs_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

grs_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GRS_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                cudaGetErrorString(e) + ")");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Runs the body with the plan's device current, restoring the caller's.
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    ok_ = cudaGetDevice(&prev_) == cudaSuccess;
    if (ok_ && prev_ != dev) {
      ok_ = cudaSetDevice(dev) == cudaSuccess;
      switched_ = ok_;
    }
  }
  ~DeviceGuard() {
    if (switched_) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = 0;
  bool ok_ = false;
  bool switched_ = false;
};

grs_status check_plan_device(const grs_plan* p) {
  if (p == nullptr) return fail(GRS_ERR_INVALID_ARG, "plan is NULL");
  if (p->device < 0) return fail(GRS_ERR_NO_DEVICE, "plan was created with GRS_PLAN_HOST_ONLY");
  return GRS_OK;
}

// Entry points that need rank gradient buffers or the plan's tensor layout,
// which a shard view does not have.
grs_status check_not_view(const grs_plan* p, const char* who) {
  if (p != nullptr && p->view_shard >= 0)
    return fail(GRS_ERR_UNSUPPORTED_COMPOSITION,
                std::string(who) + ": not defined on a shard view (it holds one rank's state, no rank "
                                   "gradients and no tensor layout)");
  return GRS_OK;
}

template <typename T>
cudaError_t upload(T** dst, const std::vector<T>& src) {
  const size_t bytes = (src.empty() ? 1 : src.size()) * sizeof(T);
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), bytes);
  if (e != cudaSuccess) return e;
  if (!src.empty()) e = cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
  return e;
}

void free_device(grs_plan* p) {
  cudaFree(p->d_seg_start);
  cudaFree(p->d_seg_tensor);
  cudaFree(p->d_bucket_seg0);
  cudaFree(p->d_tensor_live);
  p->d_tensor_live = nullptr;
  cudaFree(p->d_red_tile_tensor);
  cudaFree(p->d_upd_tile_tensor);
  cudaFree(p->d_red_tile_unit);
  cudaFree(p->d_upd_tile_unit);
  p->d_red_tile_tensor = p->d_upd_tile_tensor = nullptr;
  p->d_red_tile_unit = p->d_upd_tile_unit = nullptr;
  cudaFree(p->d_state_jobs);
  cudaFree(p->d_upd_tile_job);
  cudaFree(p->d_upd_tile_info);
  p->d_state_jobs = nullptr;
  p->d_upd_tile_job = nullptr;
  p->d_upd_tile_info = nullptr;
  p->d_seg_start = nullptr;
  p->d_seg_tensor = nullptr;
  p->d_bucket_seg0 = nullptr;
  cudaFree(p->d_units);
  cudaFree(p->d_red_prefix);
  cudaFree(p->d_jobs);
  cudaFree(p->d_chunk_job);
  cudaFree(p->d_flags);
  p->d_units = nullptr;
  p->d_red_prefix = nullptr;
  p->d_jobs = nullptr;
  p->d_chunk_job = nullptr;
  p->d_flags = nullptr;
}

}  // namespace

namespace grs {
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace grs

extern "C" {

grs_status grs_plan_create(const int64_t* numels, const int32_t* owners, int32_t n_tensors,
                           int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                           int64_t bucket_bytes, uint32_t flags, grs_plan** out) {
  return grs_plan_create_ex(numels, owners, nullptr, n_tensors, world, tp, dp_replicate, dp_shard,
                            bucket_bytes, flags, out);
}

grs_status grs_plan_create_ex(const int64_t* numels, const int32_t* owners, const uint32_t* tensor_flags,
                              int32_t n_tensors, int32_t world, int32_t tp, int32_t dp_replicate,
                              int32_t dp_shard, int64_t bucket_bytes, uint32_t flags, grs_plan** out) {
  if (out == nullptr) return fail(GRS_ERR_INVALID_ARG, "out is NULL");
  grs_plan* p = new (std::nothrow) grs_plan();
  if (p == nullptr) return fail(GRS_ERR_INVALID_ARG, "host allocation failed");
  std::string why;
  if ((flags & ~(GRS_PLAN_HOST_ONLY | GRS_PLAN_FP32_GRADS)) != 0) {
    delete p;
    return fail(GRS_ERR_INVALID_ARG, "grs_plan_create: unknown flag bits");
  }
  const int32_t esize = (flags & GRS_PLAN_FP32_GRADS) ? 4 : 2;
  const grs_status st = grs::build_plan(numels, owners, tensor_flags, n_tensors, world, tp, dp_replicate,
                                        dp_shard, bucket_bytes, esize, p, &why);
  if (st != GRS_OK) {
    delete p;
    return fail(st, why);
  }
  if ((flags & GRS_PLAN_HOST_ONLY) == 0) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = upload(&p->d_units, p->units);
    if (e == cudaSuccess) e = upload(&p->d_red_prefix, p->red_prefix);
    if (e == cudaSuccess) e = upload(&p->d_jobs, p->jobs);
    if (e == cudaSuccess) e = upload(&p->d_chunk_job, p->chunk_job);
    if (e == cudaSuccess) e = upload(&p->d_seg_start, p->seg_start);
    if (e == cudaSuccess) e = upload(&p->d_seg_tensor, p->seg_tensor);
    if (e == cudaSuccess) e = upload(&p->d_bucket_seg0, p->bucket_seg0);
    if (e == cudaSuccess) e = upload(&p->d_tensor_live, p->tensor_live);
    if (e == cudaSuccess) e = upload(&p->d_red_tile_tensor, p->red_tile_tensor);
    if (e == cudaSuccess) e = upload(&p->d_upd_tile_tensor, p->upd_tile_tensor);
    if (e == cudaSuccess) e = upload(&p->d_red_tile_unit, p->red_tile_unit);
    if (e == cudaSuccess) e = upload(&p->d_upd_tile_unit, p->upd_tile_unit);
    if (e == cudaSuccess) e = upload(&p->d_state_jobs, p->state_jobs);
    if (e == cudaSuccess) e = upload(&p->d_upd_tile_job, p->upd_tile_job);
    if (e == cudaSuccess) e = upload(&p->d_upd_tile_info, p->upd_tile_info);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->d_flags), grs::FLAG_COUNT * sizeof(int));
    if (e == cudaSuccess) e = cudaMemsetAsync(p->d_flags, 0, grs::FLAG_COUNT * sizeof(int), nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);  // cleared before any launch on any stream
    if (e != cudaSuccess) {
      free_device(p);
      delete p;
      return cuda_fail(e, "grs_plan_create: device tables");
    }
    p->device = dev;
  }
  *out = p;
  return GRS_OK;
}

grs_status grs_plan_shard_view(const grs_plan* parent, int32_t shard, int32_t tp_index, grs_plan** out) {
  if (parent == nullptr || out == nullptr) return fail(GRS_ERR_INVALID_ARG, "grs_plan_shard_view: NULL argument");
  if (parent->view_shard >= 0)
    return fail(GRS_ERR_INVALID_ARG, "grs_plan_shard_view: the parent is itself a shard view");
  if (shard < 0 || shard >= parent->dp_shard || tp_index < 0 || tp_index >= parent->tp)
    return fail(GRS_ERR_INVALID_ARG, "grs_plan_shard_view: shard must be in [0, dp_shard) and tp_index in [0, tp)");
  grs_plan* v = new (std::nothrow) grs_plan();
  if (v == nullptr) return fail(GRS_ERR_INVALID_ARG, "grs_plan_shard_view: host allocation failed");
  grs::build_shard_view(*parent, shard, tp_index, v);
  if (parent->device >= 0) {
    DeviceGuard g(parent->device);
    cudaError_t e = g.ok() ? cudaSuccess : cudaErrorInvalidDevice;
    v->sm_count = parent->sm_count;
    if (e == cudaSuccess) e = upload(&v->d_units, v->units);
    if (e == cudaSuccess) e = upload(&v->d_red_prefix, v->red_prefix);
    if (e == cudaSuccess) e = upload(&v->d_red_tile_unit, v->red_tile_unit);
    if (e == cudaSuccess) e = upload(&v->d_upd_tile_unit, v->upd_tile_unit);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&v->d_flags), grs::FLAG_COUNT * sizeof(int));
    if (e == cudaSuccess) e = cudaMemsetAsync(v->d_flags, 0, grs::FLAG_COUNT * sizeof(int), nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) {
      free_device(v);
      delete v;
      return cuda_fail(e, "grs_plan_shard_view: device tables");
    }
    v->device = parent->device;
  }
  *out = v;
  return GRS_OK;
}

void grs_plan_destroy(grs_plan* p) {
  if (p == nullptr) return;
  if (p->device >= 0) {
    DeviceGuard g(p->device);
    grs::destroy_host_step_resources(p);
    free_device(p);
  }
  delete p;
}

grs_status grs_plan_query(const grs_plan* p, grs_plan_info* o) {
  if (p == nullptr || o == nullptr) return fail(GRS_ERR_INVALID_ARG, "NULL argument");
  std::memset(o, 0, sizeof(*o));
  o->n_tensors = static_cast<int32_t>(p->numel.size());
  o->n_buckets = static_cast<int32_t>(p->buckets.size());
  o->world = p->world;
  o->tp = p->tp;
  o->dp_replicate = p->dp_replicate;
  o->dp_shard = p->dp_shard;
  o->dp = p->dp;
  o->device = p->device;
  o->n_unique = p->n_unique;
  o->n_rank_pad = p->n_rank_pad;
  o->n_state_pad = p->n_state_pad;
  o->workspace_bytes = p->workspace_bytes;
  o->n_reduce_tiles = p->n_red_tiles;
  o->grad_bytes = p->grad_esize;
  return GRS_OK;
}

grs_status grs_bucket_info(const grs_plan* p, int32_t b, grs_bucket_desc* o) {
  if (p == nullptr || o == nullptr) return fail(GRS_ERR_INVALID_ARG, "NULL argument");
  if (b < 0 || b >= static_cast<int32_t>(p->buckets.size()))
    return fail(GRS_ERR_INVALID_ARG, "bucket index out of range");
  const grs::Bucket& bk = p->buckets[b];
  std::memset(o, 0, sizeof(*o));
  o->tag = bk.tag;
  o->copies = bk.copies;
  o->group_size = bk.group_size;
  o->n_tensors = bk.n_tensors;
  o->used = bk.used;
  o->padded = bk.padded;
  o->shard_len = bk.shard_len;
  o->rank_offset = bk.rank_off;
  o->state_offset = bk.state_off;
  o->n_segments = bk.copies * (p->bucket_seg0[b + 1] - p->bucket_seg0[b]);
  return GRS_OK;
}

grs_status grs_segment_info(const grs_plan* p, int32_t b, int32_t i, grs_segment_desc* o) {
  if (p == nullptr || o == nullptr) return fail(GRS_ERR_INVALID_ARG, "NULL argument");
  const grs_status vs = check_not_view(p, "grs_segment_info");
  if (vs != GRS_OK) return vs;
  if (b < 0 || b >= static_cast<int32_t>(p->buckets.size()))
    return fail(GRS_ERR_INVALID_ARG, "bucket index out of range");
  const grs::Bucket& bk = p->buckets[b];
  const int32_t nt = p->bucket_seg0[b + 1] - p->bucket_seg0[b];
  if (i < 0 || nt == 0 || i >= bk.copies * nt) return fail(GRS_ERR_INVALID_ARG, "segment index out of range");
  const int32_t t = i / nt;
  const int32_t tensor = p->seg_tensor[p->bucket_seg0[b] + i % nt];
  const int64_t per_rank = (p->owner[tensor] == GRS_LOCAL_SHARD) ? p->numel[tensor] / p->tp : p->numel[tensor];
  std::memset(o, 0, sizeof(*o));
  o->tensor = tensor;
  o->tp_index = t;
  o->bucket_offset = p->t_offset[tensor];
  o->tensor_offset = static_cast<int64_t>(t) * per_rank;
  o->numel = per_rank;
  o->state_offset = bk.state_off + static_cast<int64_t>(t) * bk.padded + p->t_offset[tensor];
  return GRS_OK;
}

grs_status grs_tensor_info(const grs_plan* p, int32_t i, grs_tensor_desc* o) {
  if (p == nullptr || o == nullptr) return fail(GRS_ERR_INVALID_ARG, "NULL argument");
  if (i < 0 || i >= static_cast<int32_t>(p->numel.size()))
    return fail(GRS_ERR_INVALID_ARG, "tensor index out of range");
  std::memset(o, 0, sizeof(*o));
  o->bucket = p->t_bucket[i];
  o->owner = p->owner[i];
  o->numel = p->numel[i];
  o->per_rank = p->t_bucket[i] < 0 ? 0 : (p->owner[i] == GRS_LOCAL_SHARD) ? p->numel[i] / p->tp : p->numel[i];
  o->bucket_offset = p->t_offset[i];
  o->flags = p->tensor_flags[i];
  return GRS_OK;
}

static grs_status reduce_common(const grs_plan* p, const void* const* rank_grads, float* acc,
                                int32_t accumulate, int32_t emit, void* workspace, void* stream,
                                int32_t unit_begin, int32_t unit_end, int64_t state_base,
                                int64_t rank_base, int64_t state_len, int64_t rank_len, int32_t tag,
                                const char* who, int32_t max_ctas = 0,
                                void* wait_event = nullptr, const uint8_t* used_mask = nullptr) {
  if (rank_grads == nullptr || acc == nullptr)
    return fail(GRS_ERR_INVALID_ARG, std::string(who) + ": rank_grads/acc is NULL");
  if (emit && workspace == nullptr)
    return fail(GRS_ERR_INVALID_ARG, std::string(who) + ": emit_norm_partials needs a workspace");
  if (!aligned16(acc) || (workspace != nullptr && !aligned16(workspace)))
    return fail(GRS_ERR_ALIGNMENT, std::string(who) + ": acc/workspace not 16-byte aligned");
  // Ranks actually read: every rank, or rank 0 only for an ALREADY_REDUCED bucket.
  const int32_t nread = (tag == GRS_ALREADY_REDUCED) ? 1 : p->world;
  for (int32_t k = 0; k < nread; ++k) {
    if (rank_grads[k] == nullptr)
      return fail(GRS_ERR_INVALID_ARG, std::string(who) + ": rank " + std::to_string(k) + " buffer is NULL");
    if (!aligned16(rank_grads[k]))
      return fail(GRS_ERR_ALIGNMENT, std::string(who) + ": rank " + std::to_string(k) +
                                         " buffer not 16-byte aligned");
  }
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, std::string(who) + ": cannot select the plan's device");
  grs::ReduceLaunch l;
  const void* ranks[GRS_MAX_WORLD] = {};
  for (int32_t k = 0; k < p->world; ++k) ranks[k] = (k < nread) ? rank_grads[k] : rank_grads[0];
  l.ranks = ranks;
  l.acc = acc;
  l.partials = emit ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + grs::ws_partials_offset())
                    : nullptr;
  l.unit_begin = unit_begin;
  l.unit_end = unit_end;
  l.state_base = state_base;
  l.rank_base = rank_base;
  l.state_len = state_len;
  l.rank_len = rank_len;
  l.accumulate = accumulate ? 1 : 0;
  l.max_ctas = max_ctas;
  if (used_mask != nullptr) {
    l.used_mask = used_mask;
    l.tile_tensor = p->d_red_tile_tensor;
  }
  if (wait_event != nullptr) {
    const cudaError_t we = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream),
                                               static_cast<cudaEvent_t>(wait_event), 0);
    if (we != cudaSuccess) return cuda_fail(we, who);
  }
  const int e = grs::launch_reduce(p, l, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), who);
  return GRS_OK;
}

grs_status grs_reduce_bucket(const grs_plan* p, int32_t b, const void* const* rank_grads, float* acc,
                             int32_t accumulate, int32_t emit, void* workspace, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_reduce_bucket");
  if (st != GRS_OK) return st;
  if (b < 0 || b >= static_cast<int32_t>(p->buckets.size()))
    return fail(GRS_ERR_INVALID_ARG, "grs_reduce_bucket: bucket index out of range");
  const grs::Bucket& bk = p->buckets[b];
  return reduce_common(p, rank_grads, acc, accumulate, emit, workspace, stream, bk.unit0,
                       bk.unit0 + bk.copies, bk.state_off, bk.rank_off, int64_t(bk.copies) * bk.padded,
                       bk.padded, bk.tag, "grs_reduce_bucket");
}

grs_status grs_reduce_bucket_ex(const grs_plan* p, int32_t b, const void* const* rank_grads, float* acc,
                                int32_t accumulate, int32_t emit, void* workspace, int32_t max_ctas,
                                void* wait_event, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_reduce_bucket_ex");
  if (st != GRS_OK) return st;
  if (b < 0 || b >= static_cast<int32_t>(p->buckets.size()))
    return fail(GRS_ERR_INVALID_ARG, "grs_reduce_bucket_ex: bucket index out of range");
  if (max_ctas < 0) return fail(GRS_ERR_INVALID_ARG, "grs_reduce_bucket_ex: max_ctas must be >= 0");
  const grs::Bucket& bk = p->buckets[b];
  return reduce_common(p, rank_grads, acc, accumulate, emit, workspace, stream, bk.unit0,
                       bk.unit0 + bk.copies, bk.state_off, bk.rank_off, int64_t(bk.copies) * bk.padded,
                       bk.padded, bk.tag, "grs_reduce_bucket_ex", max_ctas, wait_event);
}

grs_status grs_reduce_all(const grs_plan* p, const void* const* rank_grads, float* acc,
                          int32_t accumulate, int32_t emit, void* workspace, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_reduce_all");
  if (st != GRS_OK) return st;
  bool only_ar = true;
  for (const auto& bk : p->buckets) only_ar = only_ar && bk.tag == GRS_ALREADY_REDUCED;
  return reduce_common(p, rank_grads, acc, accumulate, emit, workspace, stream, 0,
                       static_cast<int32_t>(p->units.size()), 0, 0, p->n_state_pad, p->n_rank_pad,
                       only_ar ? GRS_ALREADY_REDUCED : GRS_REPLICA_AVG, "grs_reduce_all");
}

grs_status grs_reduce_all_masked(const grs_plan* p, const void* const* rank_grads, float* acc,
                                 int32_t accumulate, int32_t emit, const uint8_t* d_tensor_used,
                                 void* workspace, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_reduce_all_masked");
  if (st != GRS_OK) return st;
  if (d_tensor_used == nullptr) return fail(GRS_ERR_INVALID_ARG, "grs_reduce_all_masked: d_tensor_used is NULL");
  // The CTAs of the persistent grid each take ceil(tiles / grid) tiles, one
  // skip bit per tile in shared memory.
  const int64_t grid = p->n_red_tiles < int64_t(p->sm_count) * GRS_RED_CTAS_PER_SM ? p->n_red_tiles
                                                                                  : int64_t(p->sm_count) * GRS_RED_CTAS_PER_SM;
  if (grid > 0 && (p->n_red_tiles + grid - 1) / grid > int64_t(grs::RED_SKIP_WORDS) * 32)
    return fail(GRS_ERR_SHAPE, "grs_reduce_all_masked: more than " + std::to_string(grs::RED_SKIP_WORDS * 32) +
                                   " reduction tiles per SM");
  bool only_ar = true;
  for (const auto& bk : p->buckets) only_ar = only_ar && bk.tag == GRS_ALREADY_REDUCED;
  return reduce_common(p, rank_grads, acc, accumulate, emit, workspace, stream, 0, static_cast<int32_t>(p->units.size()),
                       0, 0, p->n_state_pad, p->n_rank_pad, only_ar ? GRS_ALREADY_REDUCED : GRS_REPLICA_AVG,
                       "grs_reduce_all_masked", 0, nullptr, d_tensor_used);
}

grs_status grs_accumulate(const grs_plan* p, int32_t b, float* acc, const float* mb, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  if (b < 0 || b >= static_cast<int32_t>(p->buckets.size()))
    return fail(GRS_ERR_INVALID_ARG, "grs_accumulate: bucket index out of range");
  if (acc == nullptr || mb == nullptr) return fail(GRS_ERR_INVALID_ARG, "grs_accumulate: NULL buffer");
  if (!aligned16(acc) || !aligned16(mb)) return fail(GRS_ERR_ALIGNMENT, "grs_accumulate: not 16-byte aligned");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_accumulate: cannot select the plan's device");
  const int e = grs::launch_accumulate(p, b, acc, mb, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_accumulate");
  return GRS_OK;
}

grs_status grs_grad_norm_sq(const grs_plan* p, const float* acc, int32_t n_micro, void* workspace,
                            int32_t partials_ready, double* d_norm_sq, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  if (workspace == nullptr || d_norm_sq == nullptr || (!partials_ready && acc == nullptr))
    return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq: NULL argument");
  if (n_micro < 1) return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq: n_micro must be >= 1");
  if (partials_ready && p->view_shard >= 0)
    return fail(GRS_ERR_UNSUPPORTED_COMPOSITION,
                "grs_grad_norm_sq: a shard view has no reduction to emit partials (partials_ready must be 0)");
  if (!aligned16(workspace) || (acc != nullptr && !aligned16(acc)) ||
      (reinterpret_cast<uintptr_t>(d_norm_sq) & 7u) != 0)
    return fail(GRS_ERR_ALIGNMENT, "grs_grad_norm_sq: misaligned pointer");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_grad_norm_sq: cannot select the plan's device");
  const int e = grs::launch_norm(p, acc, n_micro, workspace, partials_ready, d_norm_sq, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_grad_norm_sq");
  return GRS_OK;
}

grs_status grs_clip_adamw_step(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq,
                               const float* acc, float* master, float* m, float* v,
                               uint16_t* params_bf16, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  if (hp == nullptr || acc == nullptr || master == nullptr || m == nullptr || v == nullptr ||
      params_bf16 == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step: NULL argument");
  if (hp->step < 1 || hp->n_micro < 1)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step: step and n_micro must be >= 1");
  if (hp->max_norm > 0.0f && d_norm_sq == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step: clipping needs d_norm_sq");
  if (!aligned16(acc) || !aligned16(master) || !aligned16(m) || !aligned16(v) || !aligned16(params_bf16))
    return fail(GRS_ERR_ALIGNMENT, "grs_clip_adamw_step: buffer not 16-byte aligned");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_clip_adamw_step: cannot select the plan's device");
  const int e = grs::launch_update(p, hp, d_norm_sq, acc, master, m, v, params_bf16, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_clip_adamw_step");
  return GRS_OK;
}

grs_status grs_clip_adamw_step_to_tensors(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq,
                                          const float* acc, float* master, float* m, float* v,
                                          uint16_t* params_bf16, uint16_t* const* d_tensor_ptrs, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_clip_adamw_step_to_tensors");
  if (st != GRS_OK) return st;
  if (hp == nullptr || acc == nullptr || master == nullptr || m == nullptr || v == nullptr ||
      d_tensor_ptrs == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step_to_tensors: NULL argument");
  if (hp->step < 1 || hp->n_micro < 1)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step_to_tensors: step and n_micro must be >= 1");
  if (hp->max_norm > 0.0f && d_norm_sq == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step_to_tensors: clipping needs d_norm_sq");
  if (!aligned16(acc) || !aligned16(master) || !aligned16(m) || !aligned16(v) ||
      (params_bf16 != nullptr && !aligned16(params_bf16)) ||
      (reinterpret_cast<uintptr_t>(d_tensor_ptrs) & 7u) != 0)
    return fail(GRS_ERR_ALIGNMENT, "grs_clip_adamw_step_to_tensors: buffer not 16-byte aligned "
                                   "(or the pointer table not 8-byte aligned)");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_clip_adamw_step_to_tensors: cannot select the plan's device");
  const int e = grs::launch_update_to_tensors(p, hp, d_norm_sq, acc, master, m, v, params_bf16, d_tensor_ptrs,
                                              stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_clip_adamw_step_to_tensors");
  return GRS_OK;
}

grs_status grs_update_small(const grs_plan* p, const grs_adamw* hp, const void* const* rank_grads, float* acc,
                            float* master, float* m, float* v, uint16_t* params_bf16, double* d_norm_sq,
                            void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_update_small");
  if (st != GRS_OK) return st;
  if (hp == nullptr || rank_grads == nullptr || acc == nullptr || master == nullptr || m == nullptr ||
      v == nullptr || params_bf16 == nullptr || d_norm_sq == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_update_small: NULL argument");
  if (hp->step < 1 || hp->n_micro < 1)
    return fail(GRS_ERR_INVALID_ARG, "grs_update_small: step and n_micro must be >= 1");
  if (p->n_red_tiles > GRS_SMALL_MAX_TILES || static_cast<int64_t>(p->units.size()) > GRS_SMALL_MAX_TILES)
    return fail(GRS_ERR_SHAPE, "grs_update_small: the plan has " + std::to_string(p->n_red_tiles) +
                                   " reduction tiles in " + std::to_string(p->units.size()) +
                                   " bucket rows; the single-launch path takes at most " +
                                   std::to_string(GRS_SMALL_MAX_TILES) + " of each");
  const int64_t nbuf = int64_t(hp->n_micro) * p->world;
  if (nbuf > GRS_SMALL_MAX_BUFFERS)
    return fail(GRS_ERR_SHAPE, "grs_update_small: n_micro x world = " + std::to_string(nbuf) +
                                   " gradient buffers; the single-launch path takes at most " +
                                   std::to_string(GRS_SMALL_MAX_BUFFERS));
  for (int64_t k = 0; k < nbuf; ++k) {
    if (rank_grads[k] == nullptr)
      return fail(GRS_ERR_INVALID_ARG, "grs_update_small: gradient buffer " + std::to_string(k) + " is NULL");
    if (!aligned16(rank_grads[k]))
      return fail(GRS_ERR_ALIGNMENT, "grs_update_small: gradient buffer " + std::to_string(k) +
                                         " not 16-byte aligned");
  }
  if (!aligned16(acc) || !aligned16(master) || !aligned16(m) || !aligned16(v) || !aligned16(params_bf16) ||
      (reinterpret_cast<uintptr_t>(d_norm_sq) & 7u) != 0)
    return fail(GRS_ERR_ALIGNMENT, "grs_update_small: buffer not 16-byte aligned");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_update_small: cannot select the plan's device");
  const int e = grs::launch_update_small(p, hp, rank_grads, acc, master, m, v, params_bf16, d_norm_sq, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_update_small");
  return GRS_OK;
}

grs_status grs_gather_params(const grs_plan* p, const uint16_t* params_bf16, uint16_t* const* tensor_ptrs,
                             void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_gather_params");
  if (st != GRS_OK) return st;
  if (params_bf16 == nullptr || tensor_ptrs == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_gather_params: NULL argument");
  if (!aligned16(params_bf16)) return fail(GRS_ERR_ALIGNMENT, "grs_gather_params: params not 16-byte aligned");
  for (size_t i = 0; i < p->numel.size(); ++i)
    if (tensor_ptrs[i] != nullptr && (reinterpret_cast<uintptr_t>(tensor_ptrs[i]) & 1u) != 0)
      return fail(GRS_ERR_ALIGNMENT, "grs_gather_params: tensor pointer not 2-byte aligned");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_gather_params: cannot select the plan's device");
  const int e = grs::launch_gather(p, params_bf16, tensor_ptrs, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_gather_params");
  return GRS_OK;
}

grs_status grs_grad_norm_sq_masked(const grs_plan* p, const float* acc, int32_t n_micro,
                                   const uint8_t* d_tensor_used, void* workspace, double* d_norm_sq,
                                   void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_grad_norm_sq_masked");
  if (st != GRS_OK) return st;
  if (acc == nullptr || d_tensor_used == nullptr || workspace == nullptr || d_norm_sq == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq_masked: NULL argument");
  if (n_micro < 1) return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq_masked: n_micro must be >= 1");
  if (!aligned16(acc) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(d_norm_sq) & 7u) != 0)
    return fail(GRS_ERR_ALIGNMENT, "grs_grad_norm_sq_masked: misaligned pointer");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_grad_norm_sq_masked: cannot select the plan's device");
  const int e = grs::launch_norm_masked(p, acc, n_micro, d_tensor_used, workspace, d_norm_sq, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_grad_norm_sq_masked");
  return GRS_OK;
}

grs_status grs_clip_adamw_step_masked(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq,
                                      const float* acc, float* master, float* m, float* v,
                                      uint16_t* params_bf16, const uint8_t* d_tensor_used,
                                      int32_t* d_tensor_steps, void* workspace, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_clip_adamw_step_masked");
  if (st != GRS_OK) return st;
  if (hp == nullptr || acc == nullptr || master == nullptr || m == nullptr || v == nullptr ||
      params_bf16 == nullptr || d_tensor_used == nullptr || d_tensor_steps == nullptr || workspace == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step_masked: NULL argument");
  if (hp->n_micro < 1) return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step_masked: n_micro must be >= 1");
  if (hp->max_norm > 0.0f && d_norm_sq == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_clip_adamw_step_masked: clipping needs d_norm_sq");
  if (!aligned16(acc) || !aligned16(master) || !aligned16(m) || !aligned16(v) || !aligned16(params_bf16) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(d_tensor_steps) & 3u) != 0)
    return fail(GRS_ERR_ALIGNMENT, "grs_clip_adamw_step_masked: misaligned pointer");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_clip_adamw_step_masked: cannot select the plan's device");
  const int e = grs::launch_update_masked(p, hp, d_norm_sq, acc, master, m, v, params_bf16, d_tensor_used,
                                          d_tensor_steps, workspace, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_clip_adamw_step_masked");
  return GRS_OK;
}

static grs_status state_logical_common(const grs_plan* p, const float* a, float* b, bool to_logical,
                                       void* stream, const char* who) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_state_to_logical / grs_state_from_logical");
  if (st != GRS_OK) return st;
  if (a == nullptr || b == nullptr) return fail(GRS_ERR_INVALID_ARG, std::string(who) + ": NULL argument");
  if ((reinterpret_cast<uintptr_t>(a) & 3u) != 0 || (reinterpret_cast<uintptr_t>(b) & 3u) != 0)
    return fail(GRS_ERR_ALIGNMENT, std::string(who) + ": pointer not 4-byte aligned");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, std::string(who) + ": cannot select the plan's device");
  const int e = to_logical ? grs::launch_state_to_logical(p, a, b, stream)
                           : grs::launch_state_from_logical(p, a, b, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), who);
  return GRS_OK;
}

grs_status grs_state_to_logical(const grs_plan* p, const float* state, float* logical, void* stream) {
  return state_logical_common(p, state, logical, true, stream, "grs_state_to_logical");
}

grs_status grs_state_from_logical(const grs_plan* p, const float* logical, float* state, void* stream) {
  return state_logical_common(p, logical, state, false, stream, "grs_state_from_logical");
}

grs_status grs_check_already_reduced(const grs_plan* p, const void* const* rank_grads, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  st = check_not_view(p, "grs_check_already_reduced");
  if (st != GRS_OK) return st;
  if (rank_grads == nullptr) return fail(GRS_ERR_INVALID_ARG, "grs_check_already_reduced: NULL argument");
  for (int32_t k = 0; k < p->world; ++k)
    if (rank_grads[k] == nullptr)
      return fail(GRS_ERR_INVALID_ARG, "grs_check_already_reduced: rank " + std::to_string(k) + " buffer is NULL");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_check_already_reduced: cannot select the plan's device");
  const int e = grs::launch_check_already_reduced(p, rank_grads, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_check_already_reduced");
  return GRS_OK;
}

grs_status grs_selftest_bounded_wait(const grs_plan* p, int64_t limit_ns, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  if (limit_ns < 1000 || limit_ns > 2000000000LL)
    return fail(GRS_ERR_INVALID_ARG, "grs_selftest_bounded_wait: limit_ns must be in [1 us, 2 s]");
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_selftest_bounded_wait: cannot select the plan's device");
  const int e = grs::launch_bounded_wait_selftest(p, static_cast<uint64_t>(limit_ns), stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "grs_selftest_bounded_wait");
  return GRS_OK;
}

grs_status grs_check_device_errors(const grs_plan* p, void* stream) {
  grs_status st = check_plan_device(p);
  if (st != GRS_OK) return st;
  DeviceGuard g(p->device);
  if (!g.ok()) return fail(GRS_ERR_CUDA, "grs_check_device_errors: cannot select the plan's device");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "grs_check_device_errors: stream");
  int h[grs::FLAG_COUNT] = {};
  e = cudaMemcpy(h, p->d_flags, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "grs_check_device_errors: flags");
  // Cleared on the caller's stream and waited for, so that no later launch
  // on that stream (a non-blocking one included) can race with the clear.
  e = cudaMemsetAsync(p->d_flags, 0, sizeof(h), static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "grs_check_device_errors: clear flags");
  if (h[grs::FLAG_BOUNDS]) {
    static const char* const kSite[grs::SITE_COUNT] = {
        "?", "reduce_kernel", "norm_pass1_kernel", "update_kernel", "accumulate_kernel", "gather_kernel",
        "state_logical_kernel", "norm_pass1_masked_kernel", "update_masked_kernel",
        "check_already_reduced_kernel", "small_update_kernel", "update_kernel (per-tensor parameters)"};
    const int site = h[grs::FLAG_BOUNDS] > 0 && h[grs::FLAG_BOUNDS] < grs::SITE_COUNT ? h[grs::FLAG_BOUNDS] : 0;
    return fail(GRS_ERR_BOUNDS, std::string("checked build: an index left its buffer in ") + kSite[site]);
  }
  if (h[grs::FLAG_TIMEOUT]) return fail(GRS_ERR_TIMEOUT, "a bounded device wait timed out");
  if (h[grs::FLAG_NONFINITE]) return fail(GRS_ERR_NONFINITE, "global gradient norm is not finite");
  if (h[grs::FLAG_AR_MISMATCH])
    return fail(GRS_ERR_INVALID_ARG,
                "an ALREADY_REDUCED gradient differs across ranks: it was not reduced by its owner");
  return GRS_OK;
}

const char* grs_last_error(void) { return g_last_error.c_str(); }

uint32_t grs_build_features(void) { return GRS_CHECKED ? GRS_FEATURE_CHECKED : 0u; }

}  // extern "C"
