// Gather of bf16 parameters from the bucket-ordered full-parameter buffer
// back into per-tensor storage ("Cosmos 3 ... distributed parallelism",
// section 2: parameters are all-gathered across shards for the forward;
// LOCAL_SHARD tensors are reassembled from their tp rows in dim-0 order).
//
// A segmented copy: the plan holds one job per (tensor, state row) and, per
// GATHER_CHUNK slice of a job, the job's index (one load finds a block's
// job).  Each block copies one chunk.  Tensors are packed back to back
// inside buckets, so source and destination alignments differ per job:
// when both are 16-byte co-aligned the body moves 16-byte vectors, the whole
// chunk's loads issued before its stores; otherwise 4-byte or 2-byte words.
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace grs {

namespace {

constexpr int GATHER_THREADS = 256;
constexpr int GATHER_MAX_PTRS = 256;  // tensor pointers per launch (2 KB of parameters)

// Block-wide copy of n elements of T (2 or 4 bytes).  The 16-byte body puts
// a whole chunk's loads in flight per thread (GATHER_CHUNK·sizeof(T)/16 over
// the block) before storing, so a block costs one memory round trip.
template <typename T>
__device__ __forceinline__ void block_copy(const T* __restrict__ src, T* __restrict__ dst, int64_t n) {
  constexpr int U = static_cast<int>(GATHER_CHUNK * sizeof(T) / 16 / GATHER_THREADS);
  constexpr int PER_VEC = 16 / static_cast<int>(sizeof(T));
  static_assert(U >= 1, "chunk smaller than one vector per thread");
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
  const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
  if (((sa ^ da) & 15) == 0) {
    const int64_t h = static_cast<int64_t>(((16 - (sa & 15)) & 15) / sizeof(T));
    const int64_t head = h < n ? h : n;
    for (int64_t i = threadIdx.x; i < head; i += GATHER_THREADS) dst[i] = src[i];
    const int64_t nv = (n - head) / PER_VEC;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + head);
    uint4* d4 = reinterpret_cast<uint4*>(dst + head);
    int64_t i = threadIdx.x;
    for (; i + int64_t(U - 1) * GATHER_THREADS < nv; i += int64_t(U) * GATHER_THREADS) {
      uint4 r[U];
#pragma unroll
      for (int u = 0; u < U; ++u) r[u] = __ldcs(s4 + i + u * GATHER_THREADS);
#pragma unroll
      for (int u = 0; u < U; ++u) d4[i + u * GATHER_THREADS] = r[u];
    }
    for (; i < nv; i += GATHER_THREADS) d4[i] = __ldcs(s4 + i);
    for (int64_t k = head + nv * PER_VEC + threadIdx.x; k < n; k += GATHER_THREADS) dst[k] = src[k];
  } else if (sizeof(T) == 2 && ((sa ^ da) & 3) == 0) {
    const int64_t head = ((sa & 3) != 0 && n > 0) ? 1 : 0;
    if (threadIdx.x == 0 && head) dst[0] = src[0];
    const int64_t nw = (n - head) >> 1;
    const uint32_t* s2 = reinterpret_cast<const uint32_t*>(src + head);
    uint32_t* d2 = reinterpret_cast<uint32_t*>(dst + head);
    for (int64_t i = threadIdx.x; i < nw; i += GATHER_THREADS) d2[i] = s2[i];
    if (threadIdx.x == 0 && head + nw * 2 < n) dst[n - 1] = src[n - 1];
  } else {
    for (int64_t i = threadIdx.x; i < n; i += GATHER_THREADS) dst[i] = src[i];
  }
}

struct GatherArgs {
  uint16_t* dst[GATHER_MAX_PTRS];
  const uint16_t* params;
  const GatherJob* jobs;
  const int32_t* chunk_job;
  int* flags;
  int64_t n_state;       // elements of params
  int32_t n_jobs;
  int32_t tensor_begin;  // dst[0] is this tensor
  int32_t tensor_end;
  int64_t chunk_begin;
};

__global__ void __launch_bounds__(GATHER_THREADS) gather_kernel(const __grid_constant__ GatherArgs a) {
  const int64_t chunk = a.chunk_begin + blockIdx.x;
  const int32_t j = a.chunk_job[chunk];
  if (!GRS_CHECK(j >= 0 && j < a.n_jobs, a.flags, SITE_GATHER)) return;
  const GatherJob jb = a.jobs[j];
  if (!GRS_CHECK(jb.tensor >= a.tensor_begin && jb.tensor < a.tensor_end, a.flags, SITE_GATHER)) return;
  uint16_t* dbase = a.dst[jb.tensor - a.tensor_begin];
  if (dbase == nullptr) return;
  const int64_t off = (chunk - jb.chunk0) * GATHER_CHUNK;
  const int64_t rem = jb.len - off;
  if (!GRS_CHECK(off >= 0 && rem > 0 && jb.dst >= 0 && jb.src >= 0 &&
                     jb.src + off + (rem < GATHER_CHUNK ? rem : GATHER_CHUNK) <= a.n_state,
                 a.flags, SITE_GATHER))
    return;
  block_copy(a.params + jb.src + off, dbase + jb.dst + off, rem < GATHER_CHUNK ? rem : GATHER_CHUNK);
}

// fp32 state <-> canonical logical order: the same segmented jobs and
// chunks, one block per chunk.
template <bool kToLogical>
__global__ void __launch_bounds__(GATHER_THREADS) state_logical_kernel(const GatherJob* __restrict__ jobs,
                                                                        const int32_t* __restrict__ chunk_job,
                                                                        const float* __restrict__ src_base,
                                                                        float* __restrict__ dst_base, int32_t n_jobs,
                                                                        int64_t n_state, int64_t n_logical,
                                                                        int* __restrict__ flags) {
  const int64_t chunk = blockIdx.x;
  const int32_t j = chunk_job[chunk];
  if (!GRS_CHECK(j >= 0 && j < n_jobs, flags, SITE_STATE_LOGICAL)) return;
  const GatherJob jb = jobs[j];
  const int64_t off = (chunk - jb.chunk0) * GATHER_CHUNK;
  const int64_t rem = jb.len - off;
  if (!GRS_CHECK(off >= 0 && rem > 0 && jb.src >= 0 && jb.logical >= 0 &&
                     jb.src + off + (rem < GATHER_CHUNK ? rem : GATHER_CHUNK) <= n_state &&
                     jb.logical + off + (rem < GATHER_CHUNK ? rem : GATHER_CHUNK) <= n_logical,
                 flags, SITE_STATE_LOGICAL))
    return;
  block_copy(src_base + (kToLogical ? jb.src : jb.logical) + off,
             dst_base + (kToLogical ? jb.logical : jb.src) + off, rem < GATHER_CHUNK ? rem : GATHER_CHUNK);
}

// The padding of every state row, [used, padded), set to exact zeros: the
// only state elements that no layout job writes (segments tile [0, used)).
// One block per row; a row's padding is under 8 * dp_shard elements.
__global__ void __launch_bounds__(256) zero_padding_kernel(const UnitDesc* __restrict__ units, int32_t n_units,
                                                           float* __restrict__ state, int64_t n_state,
                                                           int* __restrict__ flags) {
  if (static_cast<int32_t>(blockIdx.x) >= n_units) return;
  const UnitDesc ud = units[blockIdx.x];
  const int64_t lo = ud.state_off + ud.used;
  const int64_t hi = ud.state_off + ud.padded;
  if (!GRS_CHECK(ud.state_off >= 0 && ud.used >= 0 && ud.used <= ud.padded && hi <= n_state, flags,
                 SITE_STATE_LOGICAL))
    return;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) state[i] = 0.0f;
}

// Self-test of the bounded wait: one thread arms an mbarrier that nothing
// will ever complete and waits on it through the same routine the
// reduction's producer and consumers use.
__global__ void bounded_wait_selftest_kernel(int* flags, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait_bounded(&bar, 0, flags, &abort_flag, limit_ns);
}

// ALREADY_REDUCED check: every rank's copy of an already-reduced bucket
// must equal rank 0's bit for bit (it was reduced by its owner before it
// reached us, so all ranks hold the same values).  16-byte words compared;
// padding included (callers may leave it unset, so only [0, used) counts).
struct ArCheckArgs {
  const void* ranks[GRS_MAX_WORLD];
  const UnitDesc* unit;  // the ALREADY_REDUCED bucket's (single) row
  int64_t rank_len;      // elements of each rank buffer
  int32_t world;
  int32_t esize;
  int* flags;
};

__global__ void __launch_bounds__(256) check_already_reduced_kernel(const __grid_constant__ ArCheckArgs a) {
  const UnitDesc* ud = a.unit;
  const int64_t el = static_cast<int64_t>(blockIdx.x) * UPD_T + int64_t(threadIdx.x) * 8;
  if (el >= ud->used) return;
  const int64_t n = ud->used - el < 8 ? ud->used - el : 8;
  if (!GRS_CHECK(el >= 0 && ud->rank_off >= 0 && ud->rank_off + el + n <= a.rank_len, a.flags, SITE_AR_CHECK))
    return;
  const int64_t base = (ud->rank_off + el) * a.esize;
  const uint8_t* r0 = static_cast<const uint8_t*>(a.ranks[0]) + base;
  bool same = true;
  for (int k = 1; k < a.world && same; ++k) {
    const uint8_t* rk = static_cast<const uint8_t*>(a.ranks[k]) + base;
    for (int64_t i = 0; i < n * a.esize; ++i) same = same && (r0[i] == rk[i]);
  }
  if (!same) atomicOr(a.flags + FLAG_AR_MISMATCH, 1);
}

}  // namespace

int launch_check_already_reduced(const grs_plan* p, const void* const* ranks, void* stream) {
  ArCheckArgs a;
  for (int k = 0; k < GRS_MAX_WORLD; ++k) a.ranks[k] = k < p->world ? ranks[k] : nullptr;
  a.world = p->world;
  a.esize = p->grad_esize;
  a.flags = p->d_flags;
  a.rank_len = p->n_rank_pad;
  for (const Bucket& bk : p->buckets) {
    if (bk.tag != GRS_ALREADY_REDUCED || bk.used == 0) continue;
    a.unit = p->d_units + bk.unit0;
    const int64_t tiles = (bk.used + UPD_T - 1) / UPD_T;
    check_already_reduced_kernel<<<static_cast<unsigned>(tiles), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  return 0;
}

int launch_bounded_wait_selftest(const grs_plan* p, uint64_t limit_ns, void* stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(p->d_flags, limit_ns);
  return static_cast<int>(cudaGetLastError());
}

int launch_state_to_logical(const grs_plan* p, const float* state, float* logical, void* stream) {
  if (p->n_gather_chunks <= 0) return 0;
  state_logical_kernel<true><<<static_cast<unsigned>(p->n_gather_chunks), GATHER_THREADS, 0,
                               static_cast<cudaStream_t>(stream)>>>(
      p->d_jobs, p->d_chunk_job, state, logical, static_cast<int32_t>(p->jobs.size()), p->n_state_pad,
      p->n_unique, p->d_flags);
  return static_cast<int>(cudaGetLastError());
}

int launch_state_from_logical(const grs_plan* p, const float* logical, float* state, void* stream) {
  const int32_t n_units = static_cast<int32_t>(p->units.size());
  if (n_units > 0) {
    zero_padding_kernel<<<static_cast<unsigned>(n_units), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        p->d_units, n_units, state, p->n_state_pad, p->d_flags);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  if (p->n_gather_chunks <= 0) return 0;
  state_logical_kernel<false><<<static_cast<unsigned>(p->n_gather_chunks), GATHER_THREADS, 0,
                                static_cast<cudaStream_t>(stream)>>>(
      p->d_jobs, p->d_chunk_job, logical, state, static_cast<int32_t>(p->jobs.size()), p->n_state_pad,
      p->n_unique, p->d_flags);
  return static_cast<int>(cudaGetLastError());
}

int launch_gather(const grs_plan* p, const uint16_t* params, uint16_t* const* tensor_ptrs,
                  void* stream) {
  const int32_t n = static_cast<int32_t>(p->numel.size());
  for (int32_t t0 = 0; t0 < n; t0 += GATHER_MAX_PTRS) {
    const int32_t t1 = t0 + GATHER_MAX_PTRS < n ? t0 + GATHER_MAX_PTRS : n;
    GatherArgs a;
    bool any = false;
    for (int32_t i = 0; i < GATHER_MAX_PTRS; ++i) {
      a.dst[i] = (t0 + i < t1) ? tensor_ptrs[t0 + i] : nullptr;
      any = any || a.dst[i] != nullptr;
    }
    if (!any) continue;
    a.params = params;
    a.jobs = p->d_jobs;
    a.chunk_job = p->d_chunk_job;
    a.flags = p->d_flags;
    a.n_state = p->n_state_pad;
    a.n_jobs = static_cast<int32_t>(p->jobs.size());
    a.tensor_begin = t0;
    a.tensor_end = t1;
    const int32_t job_begin = p->tensor_job0[t0];
    const int32_t job_end = p->tensor_job0[t1];
    if (job_end <= job_begin) continue;
    a.chunk_begin = p->jobs[job_begin].chunk0;
    const int64_t chunk_end =
        job_end < static_cast<int32_t>(p->jobs.size()) ? p->jobs[job_end].chunk0 : p->n_gather_chunks;
    if (chunk_end <= a.chunk_begin) continue;
    gather_kernel<<<static_cast<unsigned>(chunk_end - a.chunk_begin), GATHER_THREADS, 0,
                    static_cast<cudaStream_t>(stream)>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  return 0;
}

}  // namespace grs
