// Global norm (deterministic, two levels), fused clip + AdamW + bf16 cast,
// and the fp32 accumulate kernel.
//
// Norm ("refactor(distributed): establish shared native TP replica
// ownership", "Proposed scope": global norms and clipping): per-tile fp32
// partial sums of acc^2 (written by the reduction's epilogue, or here by
// pass 1 in the very same order), then fp64 across tiles in a fixed tree.
// The grid never changes a partial, so the norm is bit-reproducible.
//
// Update: AdamW with decoupled weight decay (Loshchilov & Hutter, in the
// form torch.optim.AdamW documents it) on the clipped, microbatch-averaged
// gradient, fp32 state, bf16 round-to-nearest-even output in the
// bucket-ordered full-parameter layout and/or (the gather fused in) straight
// into each tensor's own storage.  Each thread streams 8 elements: 2 x 16 B
// of every fp32 array in, 2 x 16 B of each state array and 16 B of bf16 out
// (30 bytes per element, the kernel's whole traffic).
#include <cuda_bf16.h>
#include <cmath>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "launch.cuh"

namespace grs {

namespace {

constexpr int NORM1_THREADS = 256;  // 8 warps, one reduction tile each at a time
constexpr int NORM1_BLOCKS_PER_SM = 8;
constexpr int NORM2_THREADS = 256;
constexpr int UPD_THREADS = 256;
static_assert(UPD_T == UPD_THREADS * 8, "one 8-element group per thread per tile");

// ----------------------------------------------------------------- norm pass 1
// One warp per reduction tile (tile_partial_warp): the same per-tile partial,
// bit for bit, as the reduction's fused epilogue.  Warps take tiles
// gw, gw + (all warps), ...
__global__ void __launch_bounds__(NORM1_THREADS) norm_pass1_kernel(const float* __restrict__ acc,
                                                                   const UnitDesc* __restrict__ units,
                                                                   const int32_t* __restrict__ tile_unit,
                                                                   int32_t n_units, int64_t n_tiles,
                                                                   float* __restrict__ partials, int64_t n_state,
                                                                   int* __restrict__ flags) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const int64_t n_warps = int64_t(gridDim.x) * (NORM1_THREADS / 32);
  KeepAll all;
  for (int64_t tile = int64_t(blockIdx.x) * (NORM1_THREADS / 32) + (threadIdx.x >> 5); tile < n_tiles;
       tile += n_warps) {
    const int u = __ldg(tile_unit + tile);
    if (!GRS_CHECK(u >= 0 && u < n_units, flags, SITE_NORM1)) continue;  // (warp-uniform)
    const UnitDesc* ud = units + u;
    const int64_t T = ud->red_T;
    const int64_t e0 = (tile - ud->red_tile0) * T;
    const int64_t rem = ud->padded - e0;
    int n = static_cast<int>(rem < T ? rem : T);
    // (uniform over the warp: the same tile)
    if (!GRS_CHECK(e0 >= 0 && n > 0 && ud->state_off + e0 + n <= n_state, flags, SITE_NORM1)) n = 0;
    const float s = tile_partial_warp(acc + ud->state_off + e0, n >> 3, lane, all);
    if (lane == 0) partials[tile] = s;
  }
}

// ----------------------------------------------------------------- norm pass 2
// Block b of NORM_L2_BLOCKS sums its contiguous range of tile partials in
// fp64: thread t takes indices t, t+256, ... in order, then a fixed tree.
__device__ __forceinline__ double block_sum_fixed(double x, double* red) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  x = warp_sum(x);
  if (lane == 0) red[w] = x;
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0) {
    s = red[0];
    for (int k = 1; k < static_cast<int>(blockDim.x >> 5); ++k) s = __dadd_rn(s, red[k]);
  }
  return s;
}

// One launch: block b sums its contiguous range of tile partials in fp64
// (thread t takes indices t, t+256, ... in order, then a fixed tree) into
// level2[b]; the block that finishes last (a ticket counter in the
// workspace, reset by that block) sums level2[0..NORM_L2_BLOCKS) in a fixed
// tree.  Which block is last varies, the order of every addition does not.
__global__ void __launch_bounds__(NORM2_THREADS) norm_finish_kernel(const float* __restrict__ partials,
                                                                    int64_t n, double* __restrict__ level2,
                                                                    unsigned int* __restrict__ ticket,
                                                                    double inv_m2, double* __restrict__ out,
                                                                    int* __restrict__ flags) {
  __shared__ double red[NORM2_THREADS / 32];
  __shared__ bool last;
  pdl_wait();  // the partials come from the previous kernel
  pdl_trigger();
  const int64_t chunk = (n + NORM_L2_BLOCKS - 1) / NORM_L2_BLOCKS;
  const int64_t lo = blockIdx.x * chunk;
  const int64_t hi = lo + chunk < n ? lo + chunk : n;
  double s = 0.0;
  for (int64_t i = lo + threadIdx.x; i < hi; i += NORM2_THREADS)
    s = __dadd_rn(s, static_cast<double>(partials[i]));
  s = block_sum_fixed(s, red);
  if (threadIdx.x == 0) {
    level2[blockIdx.x] = s;
    __threadfence();
    last = atomicAdd(ticket, 1u) == NORM_L2_BLOCKS - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  double x = threadIdx.x < NORM_L2_BLOCKS ? __ldcg(level2 + threadIdx.x) : 0.0;
  __syncthreads();  // red[] is reused
  x = block_sum_fixed(x, red);
  if (threadIdx.x == 0) {
    x = __dmul_rn(x, inv_m2);
    *out = x;
    if (!isfinite(x)) atomicOr(flags + FLAG_NONFINITE, 1);
    *ticket = 0u;
  }
}

// ----------------------------------------------------------------- update
struct UpdateArgs {
  const float* acc;
  float* master;
  float* m;
  float* v;
  uint16_t* params;
  const double* norm_sq;
  const UnitDesc* units;
  const int32_t* tile_unit;  // [tiles]: the unit of each update tile
  int* flags;
  int64_t n_state;   // elements of acc, master, m, v and params
  int32_t n_units;
  // Per-tensor bf16 output (the fused update + gather only): the device
  // table of tensor pointers, the gather jobs in state order and each update
  // tile's first job.
  uint16_t* const* tensor_ptrs;
  const GatherJob* sjobs;
  const int32_t* tile_job;     // [tiles + 1]
  const UpdTileInfo* tile_info;  // [tiles]: unit, sole tensor (or -1), offset in it
  int32_t n_tensors;
  int32_t n_sjobs;
  AdamwK k;
  float step_size;   // lr / (1 - beta1^t)
  float inv_bc2_sqrt;// 1 / sqrt(1 - beta2^t)
  float max_norm;    // <= 0: no clipping
  float inv_m;       // 1 / n_micro
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The last state-ordered job in [lo, hi) that starts at or before state
// element e (lo itself when none does); lo < hi.
__device__ __forceinline__ int32_t find_job(const UpdateArgs& a, int32_t lo, int32_t hi, int64_t e) {
  while (hi - lo > 1) {
    const int32_t mid = lo + ((hi - lo) >> 1);
    if (a.sjobs[mid].src <= e) lo = mid; else hi = mid;
  }
  return lo;
}

// Stores one element's bf16 bits into its tensor, if a job covers state
// element e (padding belongs to none) and its tensor has a destination.
__device__ __forceinline__ void store_to_tensor(const UpdateArgs& a, int32_t lo, int32_t hi, int64_t e,
                                                uint16_t bits) {
  const GatherJob jb = a.sjobs[find_job(a, lo, hi, e)];
  if (jb.src > e || e >= jb.src + jb.len) return;
  uint16_t* d = a.tensor_ptrs[jb.tensor];
  if (d != nullptr) d[jb.dst + (e - jb.src)] = bits;
}

// kTensors: the bf16 parameters also go straight to per-tensor storage (the
// gather fused into the update); the bucket-ordered copy is then optional.
// Four blocks per SM are pinned (at most 64 registers): measured on the 3.2B
// plan, the per-tensor instance compiled for one block per SM took 70
// registers (3 blocks per SM) and 14.40 instead of 13.58 ms, and bounds of 5
// or 6 blocks per SM spill (14.35 and 15.68 ms for the plain update against
// 13.52).
template <bool kTensors>
__global__ void __launch_bounds__(UPD_THREADS, 4) update_kernel(const __grid_constant__ UpdateArgs a) {
  // Tiles run in reverse order: the reduction wrote its last tiles last, so
  // their accumulator values are the ones still in L2.
  const unsigned tile = GRS_UPD_REVERSE ? gridDim.x - 1u - blockIdx.x : blockIdx.x;
  // Per-tensor output: one 16-byte load gives the tile's unit, the tensor
  // holding the whole tile and the offset inside it, so that the caller's
  // pointer table is read in parallel with the unit descriptor (the same
  // depth of dependent loads as the plain update).  A tile that spans
  // tensors or reaches padding takes the job search after its stores.
  int32_t u_info = -1, t_sole = -1;
  uint16_t* t_dst = nullptr;
  if (kTensors) {
    const int4 w = __ldg(reinterpret_cast<const int4*>(a.tile_info + tile));
    u_info = w.x;
    const int64_t off = (static_cast<int64_t>(static_cast<uint32_t>(w.w)) << 32) | static_cast<uint32_t>(w.z);
    t_sole = off >= 0 ? w.y : -1;
    if (t_sole >= 0 && GRS_CHECK(t_sole < a.n_tensors, a.flags, SITE_UPDATE_TENSORS)) {
      t_dst = a.tensor_ptrs[t_sole];
      if (t_dst != nullptr) t_dst += off;
    } else {
      t_sole = -1;
    }
  }
  pdl_wait();  // S and acc come from the kernels before
  pdl_trigger();
  // Clip coefficient from the device-resident S, evaluated by every thread.
  const float gscale = a.max_norm > 0.0f ? clip_gscale(*a.norm_sq, a.max_norm, a.inv_m) : a.inv_m;
  const int u = kTensors ? u_info : __ldg(a.tile_unit + tile);
  if (!GRS_CHECK(u >= 0 && u < a.n_units, a.flags, SITE_UPDATE)) return;
  const UnitDesc* ud = a.units + u;
  const int64_t e0 = (static_cast<int64_t>(tile) - ud->upd_tile0) * UPD_T;
  const int64_t el = e0 + int64_t(threadIdx.x) * 8;  // element within the unit
  if (el >= ud->padded) return;
  const int64_t i = ud->state_off + el;
  const int64_t used = ud->used;
  if (!GRS_CHECK(e0 >= 0 && i >= 0 && i + 8 <= a.n_state, a.flags, SITE_UPDATE)) return;
  const float4 g0 = __ldcs(reinterpret_cast<const float4*>(a.acc + i));
  const float4 g1 = __ldcs(reinterpret_cast<const float4*>(a.acc + i + 4));
  const float4 p0 = __ldcs(reinterpret_cast<const float4*>(a.master + i));
  const float4 p1 = __ldcs(reinterpret_cast<const float4*>(a.master + i + 4));
  const float4 m0 = __ldcs(reinterpret_cast<const float4*>(a.m + i));
  const float4 m1 = __ldcs(reinterpret_cast<const float4*>(a.m + i + 4));
  const float4 v0 = __ldcs(reinterpret_cast<const float4*>(a.v + i));
  const float4 v1 = __ldcs(reinterpret_cast<const float4*>(a.v + i + 4));
  float G[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  float P[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  float M[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float V[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    adamw_elem(G[q], gscale, a.step_size, a.inv_bc2_sqrt, a.k, P[q], M[q], V[q]);
    if (el + q >= used) P[q] = M[q] = V[q] = 0.0f;  // padding
  }
  __stcs(reinterpret_cast<float4*>(a.master + i), make_float4(P[0], P[1], P[2], P[3]));
  __stcs(reinterpret_cast<float4*>(a.master + i + 4), make_float4(P[4], P[5], P[6], P[7]));
  __stcs(reinterpret_cast<float4*>(a.m + i), make_float4(M[0], M[1], M[2], M[3]));
  __stcs(reinterpret_cast<float4*>(a.m + i + 4), make_float4(M[4], M[5], M[6], M[7]));
  __stcs(reinterpret_cast<float4*>(a.v + i), make_float4(V[0], V[1], V[2], V[3]));
  __stcs(reinterpret_cast<float4*>(a.v + i + 4), make_float4(V[4], V[5], V[6], V[7]));
  uint4 h;
  h.x = pack_bf16x2(P[0], P[1]);
  h.y = pack_bf16x2(P[2], P[3]);
  h.z = pack_bf16x2(P[4], P[5]);
  h.w = pack_bf16x2(P[6], P[7]);
  if (!kTensors || a.params != nullptr) __stcs(reinterpret_cast<uint4*>(a.params + i), h);
  if (kTensors) {
    // Common case: a tile inside one tensor.
    if (t_sole >= 0) {
      if (t_dst == nullptr) return;
      uint16_t* dst = t_dst + (el - e0);
      const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
      if ((da & 15u) == 0) {
        __stcs(reinterpret_cast<uint4*>(dst), h);
      } else if ((da & 3u) == 0) {
        uint32_t* d4 = reinterpret_cast<uint32_t*>(dst);
        d4[0] = h.x; d4[1] = h.y; d4[2] = h.z; d4[3] = h.w;
      } else {
        const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = static_cast<uint16_t>(w[q >> 1] >> (16 * (q & 1)));
      }
      return;
    }
    // Tile spanning several tensors (or reaching the padding): element by element.
    const int32_t j_lo = __ldg(a.tile_job + tile);
    int32_t j_hi = __ldg(a.tile_job + tile + 1) + 1;
    if (j_hi > a.n_sjobs) j_hi = a.n_sjobs;
    if (j_lo >= a.n_sjobs) return;  // past the last tensor: padding only
    if (!GRS_CHECK(j_lo >= 0 && j_lo < j_hi && j_hi <= a.n_sjobs, a.flags, SITE_UPDATE_TENSORS)) return;
    const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (el + q < used) store_to_tensor(a, j_lo, j_hi, i + q, static_cast<uint16_t>(w[q >> 1] >> (16 * (q & 1))));
  }
}

// ----------------------------------------------------------------- accumulate
__global__ void __launch_bounds__(UPD_THREADS) accumulate_kernel(float* __restrict__ acc,
                                                                 const float* __restrict__ mb,
                                                                 const UnitDesc* __restrict__ units,
                                                                 const int32_t* __restrict__ tile_unit,
                                                                 int32_t unit_begin, int32_t unit_end,
                                                                 int64_t tile_begin, int64_t state_base,
                                                                 int64_t state_len, int* __restrict__ flags) {
  const int64_t tile = tile_begin + blockIdx.x;
  // The plan's tables are read before the dependent-launch wait (which
  // waits only when the build enables dependent launch); acc and mb after.
  const int u = __ldg(tile_unit + tile);
  if (!GRS_CHECK(u >= unit_begin && u < unit_end, flags, SITE_ACCUMULATE)) return;
  const UnitDesc* ud = units + u;
  const int64_t el = (tile - ud->upd_tile0) * UPD_T + int64_t(threadIdx.x) * 8;
  const int64_t padded = ud->padded, used = ud->used;
  const int64_t i = ud->state_off - state_base + el;
  pdl_wait();
  pdl_trigger();
  if (el >= padded) return;
  if (!GRS_CHECK(el >= 0 && i >= 0 && i + 8 <= state_len, flags, SITE_ACCUMULATE)) return;
  float4* a4 = reinterpret_cast<float4*>(acc + i);
  const float4* b4 = reinterpret_cast<const float4*>(mb + i);
  float4 x0 = a4[0], x1 = a4[1];
  const float4 y0 = __ldg(b4), y1 = __ldg(b4 + 1);
  float o[8] = {__fadd_rn(x0.x, y0.x), __fadd_rn(x0.y, y0.y), __fadd_rn(x0.z, y0.z),
                __fadd_rn(x0.w, y0.w), __fadd_rn(x1.x, y1.x), __fadd_rn(x1.y, y1.y),
                __fadd_rn(x1.z, y1.z), __fadd_rn(x1.w, y1.w)};
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (el + q >= used) o[q] = 0.0f;
  a4[0] = make_float4(o[0], o[1], o[2], o[3]);
  a4[1] = make_float4(o[4], o[5], o[6], o[7]);
}

}  // namespace

int launch_norm(const grs_plan* p, const float* acc, int32_t n_micro, void* workspace,
                int32_t partials_ready, double* d_norm_sq, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_partials_offset());
  if (!partials_ready && p->n_red_tiles > 0) {
    const int64_t tiles_per_block = NORM1_THREADS / 32;
    const int64_t need = (p->n_red_tiles + tiles_per_block - 1) / tiles_per_block;
    const int64_t cap = int64_t(p->sm_count) * NORM1_BLOCKS_PER_SM;
    const int64_t grid = need < cap ? need : cap;
    const int e = static_cast<int>(launch_k(norm_pass1_kernel, dim3(unsigned(grid)), dim3(NORM1_THREADS), 0, s,
                                            acc, static_cast<const UnitDesc*>(p->d_units),
                                            static_cast<const int32_t*>(p->d_red_tile_unit),
                                            static_cast<int32_t>(p->units.size()), p->n_red_tiles, partials,
                                            p->n_state_pad, p->d_flags));
    if (e != 0) return e;
  }
  return launch_norm_finish(p, n_micro, workspace, d_norm_sq, stream);
}

int launch_norm_finish(const grs_plan* p, int32_t n_micro, void* workspace, double* d_norm_sq,
                       void* stream) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* partials = reinterpret_cast<float*>(ws + ws_partials_offset());
  double* level2 = reinterpret_cast<double*>(ws + ws_level2_offset(p->n_red_tiles));
  unsigned int* ticket = reinterpret_cast<unsigned int*>(ws + ws_ticket_offset(p->n_red_tiles));
  const double inv_m = 1.0 / static_cast<double>(n_micro);
  return static_cast<int>(launch_k(norm_finish_kernel, dim3(NORM_L2_BLOCKS), dim3(NORM2_THREADS), 0, stream,
                                   static_cast<const float*>(partials), p->n_red_tiles, level2, ticket,
                                   inv_m * inv_m, d_norm_sq, p->d_flags));
}

AdamwK adamw_consts(const grs_adamw* hp) {
  AdamwK k;
  const double lr = hp->lr, wd = hp->weight_decay;
  k.decay = static_cast<float>(1.0 - lr * wd);
  k.b1 = hp->beta1;
  k.omb1 = static_cast<float>(1.0 - static_cast<double>(hp->beta1));
  k.b2 = hp->beta2;
  k.omb2 = static_cast<float>(1.0 - static_cast<double>(hp->beta2));
  k.eps = hp->eps;
  return k;
}

void bias_factors(const grs_adamw* hp, int32_t step, float* step_size, float* inv_bc2_sqrt) {
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2;
  const double bc1 = 1.0 - std::pow(b1, static_cast<double>(step));
  const double bc2 = 1.0 - std::pow(b2, static_cast<double>(step));
  *step_size = static_cast<float>(lr / bc1);
  *inv_bc2_sqrt = static_cast<float>(1.0 / std::sqrt(bc2));
}

namespace {

UpdateArgs update_args(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq, const float* acc,
                       float* master, float* m, float* v, uint16_t* params) {
  UpdateArgs a{};
  a.acc = acc;
  a.master = master;
  a.m = m;
  a.v = v;
  a.params = params;
  a.norm_sq = d_norm_sq;
  a.units = p->d_units;
  a.tile_unit = p->d_upd_tile_unit;
  a.flags = p->d_flags;
  a.n_state = p->n_state_pad;
  a.n_units = static_cast<int32_t>(p->units.size());
  a.k = adamw_consts(hp);
  bias_factors(hp, hp->step, &a.step_size, &a.inv_bc2_sqrt);
  a.max_norm = hp->max_norm > 0.0f ? hp->max_norm : 0.0f;
  a.inv_m = static_cast<float>(1.0 / static_cast<double>(hp->n_micro));
  return a;
}

}  // namespace

int launch_update(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq, const float* acc,
                  float* master, float* m, float* v, uint16_t* params, void* stream) {
  if (p->n_upd_tiles <= 0) return 0;
  const UpdateArgs a = update_args(p, hp, d_norm_sq, acc, master, m, v, params);
  return static_cast<int>(
      launch_k(update_kernel<false>, dim3(unsigned(p->n_upd_tiles)), dim3(UPD_THREADS), 0, stream, a));
}

int launch_update_to_tensors(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq, const float* acc,
                             float* master, float* m, float* v, uint16_t* params,
                             uint16_t* const* d_tensor_ptrs, void* stream) {
  if (p->n_upd_tiles <= 0) return 0;
  UpdateArgs a = update_args(p, hp, d_norm_sq, acc, master, m, v, params);
  a.tensor_ptrs = d_tensor_ptrs;
  a.sjobs = p->d_state_jobs;
  a.tile_job = p->d_upd_tile_job;
  a.tile_info = p->d_upd_tile_info;
  a.n_tensors = static_cast<int32_t>(p->numel.size());
  a.n_sjobs = static_cast<int32_t>(p->state_jobs.size());
  return static_cast<int>(
      launch_k(update_kernel<true>, dim3(unsigned(p->n_upd_tiles)), dim3(UPD_THREADS), 0, stream, a));
}

int launch_accumulate(const grs_plan* p, int32_t bucket, float* acc, const float* mb, void* stream) {
  const Bucket& bk = p->buckets[bucket];
  const int32_t ub = bk.unit0, ue = bk.unit0 + bk.copies;
  const int64_t t0 = p->upd_prefix[ub], t1 = p->upd_prefix[ue];
  if (t1 <= t0) return 0;
  return static_cast<int>(launch_k(accumulate_kernel, dim3(static_cast<unsigned>(t1 - t0)), dim3(UPD_THREADS), 0,
                                   stream, acc, mb, static_cast<const UnitDesc*>(p->d_units),
                                   static_cast<const int32_t*>(p->d_upd_tile_unit), ub, ue, t0, bk.state_off,
                                   int64_t(bk.copies) * bk.padded, p->d_flags));
}

}  // namespace grs
