// grs_step_from_host: one whole update from host-resident rank gradients.
//
// Gradients arrive per bucket, as a backward pass produces them ("refactor
// (distributed): establish shared native TP replica ownership", "Preserved
// prototype and evidence": an asynchronous FP32 reduction hook; "Proposed
// scope": overlap during backward).  Here the host-to-device copy of bucket
// b+1 (on the plan's own copy stream) overlaps the reduction of bucket b (on
// the caller's stream): one cudaMemcpyAsync per rank row read by the bucket's
// owner group (rank 0 only for ALREADY_REDUCED), an event per bucket and
// staging half, two staging halves alternating across microbatches.  Then
// the norm finish, clip + AdamW + bf16, and the copies back to the host.
#include <cuda_runtime.h>

#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace {

std::mutex g_res_mu;

struct Resources {
  cudaStream_t copy = nullptr;
  cudaEvent_t start = nullptr;       // the caller's stream at the first call's entry
  cudaEvent_t prev_done = nullptr;   // after the last reduction of the previous call
  bool have_prev = false;            // prev_done was recorded by a call that succeeded
  std::vector<cudaEvent_t> copied;   // [2][n_buckets]
  std::vector<cudaEvent_t> reduced;  // [2][n_buckets]
};

Resources* resources(const grs_plan* p) { return static_cast<Resources*>(p->host_step_resources); }

grs_status fail(grs_status s, const std::string& msg) {
  grs::set_last_error(msg);
  return s;
}

grs_status ensure_resources(grs_plan* p) {
  std::lock_guard<std::mutex> lock(g_res_mu);
  if (p->host_step_resources != nullptr) return GRS_OK;
  Resources* r = new Resources();
  const size_t ne = 2 * p->buckets.size();
  cudaError_t e = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->prev_done, cudaEventDisableTiming);
  for (size_t i = 0; i < ne && e == cudaSuccess; ++i) {
    cudaEvent_t a = nullptr, b = nullptr;
    e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
    r->copied.push_back(a);
    r->reduced.push_back(b);
  }
  if (e != cudaSuccess) {
    for (auto ev : r->copied) if (ev) cudaEventDestroy(ev);
    for (auto ev : r->reduced) if (ev) cudaEventDestroy(ev);
    if (r->start) cudaEventDestroy(r->start);
    if (r->prev_done) cudaEventDestroy(r->prev_done);
    if (r->copy) cudaStreamDestroy(r->copy);
    delete r;
    return fail(GRS_ERR_CUDA, std::string("grs_step_from_host: stream/event creation: ") + cudaGetErrorString(e));
  }
  p->host_step_resources = r;
  return GRS_OK;
}

}  // namespace

namespace grs {
void destroy_host_step_resources(grs_plan* p) {
  Resources* r = resources(p);
  if (r == nullptr) return;
  if (r->copy) cudaStreamSynchronize(r->copy);
  for (auto ev : r->copied) cudaEventDestroy(ev);
  for (auto ev : r->reduced) cudaEventDestroy(ev);
  if (r->start) cudaEventDestroy(r->start);
  if (r->prev_done) cudaEventDestroy(r->prev_done);
  if (r->copy) cudaStreamDestroy(r->copy);
  delete r;
  p->host_step_resources = nullptr;
}
}  // namespace grs

extern "C" grs_status grs_step_from_host(const grs_plan* pc, const grs_adamw* hp,
                                         const void* const* host_grads, void* const* dev_stage,
                                         float* acc, float* master, float* m, float* v,
                                         uint16_t* params_bf16, void* workspace, double* d_norm_sq,
                                         uint16_t* host_params, double* host_norm_sq, void* stream) {
  grs_plan* p = const_cast<grs_plan*>(pc);
  if (p == nullptr || hp == nullptr || host_grads == nullptr || dev_stage == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_step_from_host: NULL argument");
  if (p->device < 0) return fail(GRS_ERR_NO_DEVICE, "grs_step_from_host: plan was created with GRS_PLAN_HOST_ONLY");
  if (p->view_shard >= 0)
    return fail(GRS_ERR_UNSUPPORTED_COMPOSITION, "grs_step_from_host: not defined on a shard view");
  if (hp->n_micro < 1 || hp->step < 1)
    return fail(GRS_ERR_INVALID_ARG, "grs_step_from_host: step and n_micro must be >= 1");
  const int32_t M = hp->n_micro, W = p->world;
  for (int32_t j = 0; j < M; ++j)
    for (int32_t k = 0; k < W; ++k)
      if (host_grads[size_t(j) * W + k] == nullptr)
        return fail(GRS_ERR_INVALID_ARG, "grs_step_from_host: host gradient pointer is NULL");
  for (int32_t s = 0; s < (M > 1 ? 2 : 1); ++s)
    for (int32_t k = 0; k < W; ++k) {
      const void* d = dev_stage[size_t(s) * W + k];
      if (d == nullptr) return fail(GRS_ERR_INVALID_ARG, "grs_step_from_host: staging pointer is NULL");
      if ((reinterpret_cast<uintptr_t>(d) & 15u) != 0)
        return fail(GRS_ERR_ALIGNMENT, "grs_step_from_host: staging buffer not 16-byte aligned");
    }
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return fail(GRS_ERR_CUDA, "grs_step_from_host: cudaGetDevice");
  if (prev != p->device && cudaSetDevice(p->device) != cudaSuccess)
    return fail(GRS_ERR_CUDA, "grs_step_from_host: cannot select the plan's device");
  grs_status st = ensure_resources(p);
  Resources* r = resources(p);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t nb = p->buckets.size();
  // The copies only write the staging halves.  On the first call they wait
  // for everything the caller queued before; afterwards only for the
  // previous call's reductions (the last readers of the staging halves), so
  // this step's host-to-device copies overlap the previous step's update and
  // read-back.
  if (st == GRS_OK) {
    cudaError_t e = cudaSuccess;
    if (!r->have_prev) {
      e = cudaEventRecord(r->start, cs);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(r->copy, r->start, 0);
    } else {
      e = cudaStreamWaitEvent(r->copy, r->prev_done, 0);
    }
    if (e != cudaSuccess) st = fail(GRS_ERR_CUDA, std::string("grs_step_from_host: ") + cudaGetErrorString(e));
  }
  for (int32_t j = 0; j < M && st == GRS_OK; ++j) {
    const int32_t half = j & 1;
    for (size_t b = 0; b < nb && st == GRS_OK; ++b) {
      const grs::Bucket& bk = p->buckets[b];
      cudaEvent_t ev_copy = r->copied[half * nb + b];
      cudaEvent_t ev_red = r->reduced[half * nb + b];
      cudaError_t e = cudaSuccess;
      if (j >= 2) e = cudaStreamWaitEvent(r->copy, ev_red, 0);  // staging half is free again
      const int32_t nread = bk.tag == GRS_ALREADY_REDUCED ? 1 : W;
      const size_t es = static_cast<size_t>(p->grad_esize);
      const size_t bytes = size_t(bk.padded) * es;
      const size_t boff = size_t(bk.rank_off) * es;
      for (int32_t k = 0; k < nread && e == cudaSuccess && bytes > 0; ++k)
        e = cudaMemcpyAsync(static_cast<uint8_t*>(dev_stage[size_t(half) * W + k]) + boff,
                            static_cast<const uint8_t*>(host_grads[size_t(j) * W + k]) + boff, bytes,
                            cudaMemcpyHostToDevice, r->copy);
      if (e == cudaSuccess) e = cudaEventRecord(ev_copy, r->copy);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev_copy, 0);
      if (e != cudaSuccess) {
        st = fail(GRS_ERR_CUDA, std::string("grs_step_from_host: copy: ") + cudaGetErrorString(e));
        break;
      }
      const void* ranks[GRS_MAX_WORLD] = {};
      for (int32_t k = 0; k < W; ++k)
        ranks[k] = static_cast<const uint8_t*>(dev_stage[size_t(half) * W + (k < nread ? k : 0)]) + boff;
      st = grs_reduce_bucket(p, static_cast<int32_t>(b), ranks, acc + bk.state_off, j > 0 ? 1 : 0,
                             j == M - 1 ? 1 : 0, workspace, stream);
      if (st != GRS_OK) break;
      e = cudaEventRecord(ev_red, cs);
      if (e != cudaSuccess) st = fail(GRS_ERR_CUDA, std::string("grs_step_from_host: ") + cudaGetErrorString(e));
    }
  }
  if (st == GRS_OK) {
    const cudaError_t e = cudaEventRecord(r->prev_done, cs);
    if (e != cudaSuccess) st = fail(GRS_ERR_CUDA, std::string("grs_step_from_host: ") + cudaGetErrorString(e));
  }
  // A call that failed part-way may have left reductions queued; the next
  // call then waits for all work on its stream again.
  if (r != nullptr) r->have_prev = st == GRS_OK;
  if (st == GRS_OK) st = grs_grad_norm_sq(p, acc, M, workspace, 1, d_norm_sq, stream);
  if (st == GRS_OK) st = grs_clip_adamw_step(p, hp, d_norm_sq, acc, master, m, v, params_bf16, stream);
  if (st == GRS_OK && host_params != nullptr) {
    const cudaError_t e = cudaMemcpyAsync(host_params, params_bf16, size_t(p->n_state_pad) * 2,
                                          cudaMemcpyDeviceToHost, cs);
    if (e != cudaSuccess) st = fail(GRS_ERR_CUDA, std::string("grs_step_from_host: D2H: ") + cudaGetErrorString(e));
  }
  if (st == GRS_OK && host_norm_sq != nullptr) {
    const cudaError_t e = cudaMemcpyAsync(host_norm_sq, d_norm_sq, sizeof(double), cudaMemcpyDeviceToHost, cs);
    if (e != cudaSuccess) st = fail(GRS_ERR_CUDA, std::string("grs_step_from_host: D2H: ") + cudaGetErrorString(e));
  }
  if (prev != p->device) cudaSetDevice(prev);
  return st;
}
