// Per-step tensor masks: parameters without a gradient this step.
//
// "refactor(distributed): establish shared native TP replica ownership",
// "Proposed scope": validate frozen/unused parameters.  A parameter whose
// gradient is absent this step (PyTorch's grad None) is skipped the way
// clip_grad_norm_ and torch.optim.AdamW skip it: it adds nothing to the
// global norm, and its master, moments, bf16 copy and step count stay as
// they are.  Every other tensor advances its own step count, so its bias
// correction follows the number of updates it actually received.
//
// Element -> tensor: each bucket row holds its tensors back to back; the
// plan's segment table (start offset, tensor) per bucket is searched once
// per thread and then walked forward.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "device.cuh"
#include "internal.h"

namespace grs {

namespace {

constexpr int MNORM_THREADS = 256;  // 8 warps, one reduction tile each (as the unmasked pass)
constexpr int MNORM_BLOCKS_PER_SM = 8;
constexpr int MUPD_THREADS = 256;
// Resident blocks per SM the masked update is compiled for (register cap):
// 4 (64 registers, a few bytes spilled) measured 8% faster than 3 (75).
#ifndef GRS_MUPD_MIN_BLOCKS
#define GRS_MUPD_MIN_BLOCKS 4
#endif
static_assert(UPD_T == MUPD_THREADS * 8, "one 8-element group per thread per tile");

// The masked norm pass: one warp per reduction tile, the same partials as
// the unmasked pass (tile_partial_warp) with elements of tensors without a
// gradient counted as zero.  The tile's loads do not wait for the mask.
__global__ void __launch_bounds__(MNORM_THREADS, 3) norm_pass1_masked_kernel(
    const float* __restrict__ acc, const UnitDesc* __restrict__ units, const int32_t* __restrict__ tile_unit,
    int32_t n_units, int64_t n_tiles, Segs sg, const uint8_t* __restrict__ used_mask,
    const int32_t* __restrict__ tile_tensor, float* __restrict__ partials, int64_t n_state,
    int* __restrict__ flags) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = int64_t(gridDim.x) * (MNORM_THREADS / 32);
  for (int64_t tile = int64_t(blockIdx.x) * (MNORM_THREADS / 32) + (threadIdx.x >> 5); tile < n_tiles;
       tile += n_warps) {
    const int u = __ldg(tile_unit + tile);
    if (!GRS_CHECK(u >= 0 && u < n_units, flags, SITE_NORM1_MASKED)) continue;  // (warp-uniform)
    const UnitDesc* ud = units + u;
    const int64_t T = ud->red_T;
    const int64_t e0 = (tile - ud->red_tile0) * T;
    const int64_t rem = ud->padded - e0;
    int n = static_cast<int>(rem < T ? rem : T);
    if (!GRS_CHECK(e0 >= 0 && n > 0 && ud->state_off + e0 + n <= n_state, flags, SITE_NORM1_MASKED)) n = 0;
    // A tile inside one tensor: its mask bit decides the whole tile (a tile
    // without a gradient is not read: its partial is +0, as when summed).
    const int32_t sole = __ldg(tile_tensor + tile);
    float s = 0.0f;
    if (sole >= 0 && GRS_CHECK(sole < sg.n_tensors, flags, SITE_NORM1_MASKED)) {
      if (__ldg(used_mask + sole) != 0) {
        KeepAll all;
        s = tile_partial_warp(acc + ud->state_off + e0, n >> 3, lane, all);
      }
    } else if (sole < 0) {
      const int lo = __ldg(sg.bucket_seg0 + ud->bucket), hi = __ldg(sg.bucket_seg0 + ud->bucket + 1);
      MaskKeep keep{sg, used_mask, lo, hi, e0, ud->used, flags, SITE_NORM1_MASKED, SegCursor{lo, hi, 0, -1, false}, 0};
      // (two chunk loads in flight per lane: the cursor needs the registers)
      s = tile_partial_warp<2>(acc + ud->state_off + e0, n >> 3, lane, keep);
    }
    if (lane == 0) partials[tile] = s;
  }
}

// Per tensor: advance the step count of tensors with a gradient and derive
// their bias-corrected factors (lr / (1 - b1^t), 1 / sqrt(1 - b2^t)).  A
// tensor whose new step equals the caller's step takes the factors the host
// computed for it (the plain update's, bit for bit); any other is computed
// here in fp64 (slow on this GPU's fp64 units, so only for tensors that
// skipped updates).
__global__ void tensor_factors_kernel(int32_t n, const uint8_t* __restrict__ live,
                                      const uint8_t* __restrict__ used_mask, int32_t* __restrict__ steps,
                                      float2* __restrict__ factors, double lr, double b1, double b2,
                                      int32_t hint_step, float2 hint) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (live[i] && used_mask[i]) {
    const int t = steps[i] + 1;
    steps[i] = t;
    if (t == hint_step) {
      factors[i] = hint;
      return;
    }
    const double bc1 = 1.0 - pow(b1, static_cast<double>(t));
    const double bc2 = 1.0 - pow(b2, static_cast<double>(t));
    factors[i] = make_float2(static_cast<float>(lr / bc1), static_cast<float>(1.0 / sqrt(bc2)));
  } else {
    factors[i] = make_float2(0.0f, 0.0f);
  }
}

struct MaskedArgs {
  const float* acc;
  float* master;
  float* m;
  float* v;
  uint16_t* params;
  const double* norm_sq;
  const UnitDesc* units;
  const int32_t* tile_unit;    // per update tile: its unit
  Segs sg;
  const uint8_t* used_mask;
  const int32_t* tile_tensor;  // per update tile: the tensor holding it whole, or -1
  const float2* factors;
  int* flags;
  int64_t n_state;  // elements of acc, master, m, v and params
  int32_t n_units;
  AdamwK k;
  float max_norm;
  float inv_m;
};

__device__ __forceinline__ uint16_t bf16_rn(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

__global__ void __launch_bounds__(MUPD_THREADS, GRS_MUPD_MIN_BLOCKS) update_masked_kernel(const __grid_constant__ MaskedArgs a) {
  // Tiles in reverse order, as the unmasked update (the reduction's last
  // accumulator tiles are the ones still in L2).
  const unsigned tile = gridDim.x - 1u - blockIdx.x;
  // A tile inside one tensor (the common case): one mask bit and one factor
  // pair for the whole block; a tile without a gradient is neither read nor
  // written.
  // (The tile's unit and tensor load together.)
  const int32_t sole = __ldg(a.tile_tensor + tile);
  const int u = __ldg(a.tile_unit + tile);
  if (!GRS_CHECK(u >= 0 && u < a.n_units, a.flags, SITE_UPDATE_MASKED)) return;
  const UnitDesc* ud = a.units + u;
  const int64_t el = (static_cast<int64_t>(tile) - ud->upd_tile0) * UPD_T + int64_t(threadIdx.x) * 8;
  const int64_t padded = ud->padded;
  const int64_t i = ud->state_off + el;
  const int64_t used = ud->used;
  const bool whole = sole >= 0 && GRS_CHECK(sole < a.sg.n_tensors, a.flags, SITE_UPDATE_MASKED);
  float2 f = make_float2(0.0f, 0.0f);
  uint8_t on = 1;
  if (whole) {
    on = __ldg(a.used_mask + sole);
    f = __ldg(a.factors + sole);
  }
  if (on == 0 || el >= padded) return;
  if (!GRS_CHECK(i >= 0 && i + 8 <= a.n_state, a.flags, SITE_UPDATE_MASKED)) return;
  const float gscale = a.max_norm > 0.0f ? clip_gscale(*a.norm_sq, a.max_norm, a.inv_m) : a.inv_m;

  // Otherwise: which of the eight elements change — padding (rewritten as
  // zeros) and elements of tensors with a gradient this step.  A group that
  // lies wholly in tensors without a gradient is neither read nor written.
  uint32_t wmask = 0xffu;  // bit q: element el + q is written (a whole tile holds no padding)
  SegCursor cur0;
  cur0.s = 0;
  cur0.hi = 0;
  cur0.end = INT64_MAX;
  cur0.t = sole;
  cur0.on = true;
  if (!whole) {
    const int lo = __ldg(a.sg.bucket_seg0 + ud->bucket), hi = __ldg(a.sg.bucket_seg0 + ud->bucket + 1);
    cur0.s = lo;
    cur0.hi = hi;
    cur0.end = 0;
    cur0.t = -1;
    cur0.on = false;
    if (el < used) cur0 = seg_at(a.sg, a.used_mask, lo, hi, el, used, a.flags, SITE_UPDATE_MASKED);
    SegCursor cur = cur0;
    wmask = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int64_t e = el + q;
      bool w = true;  // padding
      if (e < used) {
        if (e >= cur.end) seg_advance(cur, a.sg, a.used_mask, e, used, a.flags, SITE_UPDATE_MASKED);
        w = cur.on;
      }
      wmask |= (w ? 1u : 0u) << q;
    }
    if (wmask == 0) return;
    if (cur0.t >= 0) f = __ldg(a.factors + cur0.t);
  }
  const bool all = wmask == 0xffu;

  const float4 g0 = __ldcs(reinterpret_cast<const float4*>(a.acc + i));
  const float4 g1 = __ldcs(reinterpret_cast<const float4*>(a.acc + i + 4));
  const float4 p0 = __ldcs(reinterpret_cast<const float4*>(a.master + i));
  const float4 p1 = __ldcs(reinterpret_cast<const float4*>(a.master + i + 4));
  const float4 m0 = __ldcs(reinterpret_cast<const float4*>(a.m + i));
  const float4 m1 = __ldcs(reinterpret_cast<const float4*>(a.m + i + 4));
  const float4 v0 = __ldcs(reinterpret_cast<const float4*>(a.v + i));
  const float4 v1 = __ldcs(reinterpret_cast<const float4*>(a.v + i + 4));
  const float G[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  float P[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  float M[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float V[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  SegCursor cur = cur0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int64_t e = el + q;
    if (e >= used) {  // padding: exact zeros
      P[q] = M[q] = V[q] = 0.0f;
      continue;
    }
    if (!((wmask >> q) & 1u)) continue;  // no gradient this step: state stays
    if (e >= cur.end) {
      seg_advance(cur, a.sg, a.used_mask, e, used, a.flags, SITE_UPDATE_MASKED);
      f = __ldg(a.factors + cur.t);
    }
    adamw_elem(G[q], gscale, f.x, f.y, a.k, P[q], M[q], V[q]);
  }
  if (all) {
    __stcs(reinterpret_cast<float4*>(a.master + i), make_float4(P[0], P[1], P[2], P[3]));
    __stcs(reinterpret_cast<float4*>(a.master + i + 4), make_float4(P[4], P[5], P[6], P[7]));
    __stcs(reinterpret_cast<float4*>(a.m + i), make_float4(M[0], M[1], M[2], M[3]));
    __stcs(reinterpret_cast<float4*>(a.m + i + 4), make_float4(M[4], M[5], M[6], M[7]));
    __stcs(reinterpret_cast<float4*>(a.v + i), make_float4(V[0], V[1], V[2], V[3]));
    __stcs(reinterpret_cast<float4*>(a.v + i + 4), make_float4(V[4], V[5], V[6], V[7]));
    uint4 h;
    h.x = uint32_t(bf16_rn(P[0])) | (uint32_t(bf16_rn(P[1])) << 16);
    h.y = uint32_t(bf16_rn(P[2])) | (uint32_t(bf16_rn(P[3])) << 16);
    h.z = uint32_t(bf16_rn(P[4])) | (uint32_t(bf16_rn(P[5])) << 16);
    h.w = uint32_t(bf16_rn(P[6])) | (uint32_t(bf16_rn(P[7])) << 16);
    __stcs(reinterpret_cast<uint4*>(a.params + i), h);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (!((wmask >> q) & 1u)) continue;
      a.master[i + q] = P[q];
      a.m[i + q] = M[q];
      a.v[i + q] = V[q];
      a.params[i + q] = bf16_rn(P[q]);
    }
  }
}

}  // namespace

int launch_norm_masked(const grs_plan* p, const float* acc, int32_t n_micro, const uint8_t* used,
                       void* workspace, double* d_norm_sq, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_partials_offset());
  if (p->n_red_tiles > 0) {
    const int64_t tiles_per_block = MNORM_THREADS / 32;
    const int64_t need = (p->n_red_tiles + tiles_per_block - 1) / tiles_per_block;
    const int64_t cap = int64_t(p->sm_count) * MNORM_BLOCKS_PER_SM;
    const int64_t grid = need < cap ? need : cap;
    norm_pass1_masked_kernel<<<static_cast<unsigned>(grid), MNORM_THREADS, 0, s>>>(
        acc, p->d_units, p->d_red_tile_unit, static_cast<int32_t>(p->units.size()), p->n_red_tiles,
        Segs{p->d_seg_start, p->d_seg_tensor, p->d_bucket_seg0, static_cast<int32_t>(p->numel.size())}, used,
        p->d_red_tile_tensor, partials,
        p->n_state_pad, p->d_flags);
    const int e = static_cast<int>(cudaGetLastError());
    if (e != 0) return e;
  }
  return launch_norm_finish(p, n_micro, workspace, d_norm_sq, stream);
}

int launch_update_masked(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq,
                         const float* acc, float* master, float* m, float* v, uint16_t* params,
                         const uint8_t* used, int32_t* steps, void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t n = static_cast<int32_t>(p->numel.size());
  float2* factors = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + ws_factors_offset(p->n_red_tiles));
  float2 hint = make_float2(0.0f, 0.0f);
  const int32_t hint_step = hp->step >= 1 ? hp->step : 0;
  if (hint_step >= 1) bias_factors(hp, hint_step, &hint.x, &hint.y);
  tensor_factors_kernel<<<(n + 255) / 256, 256, 0, s>>>(n, p->d_tensor_live, used, steps, factors, hp->lr,
                                                         hp->beta1, hp->beta2, hint_step, hint);
  int e = static_cast<int>(cudaGetLastError());
  if (e != 0 || p->n_upd_tiles <= 0) return e;
  MaskedArgs a;
  a.acc = acc;
  a.master = master;
  a.m = m;
  a.v = v;
  a.params = params;
  a.norm_sq = d_norm_sq;
  a.units = p->d_units;
  a.tile_unit = p->d_upd_tile_unit;
  a.sg = Segs{p->d_seg_start, p->d_seg_tensor, p->d_bucket_seg0, static_cast<int32_t>(p->numel.size())};
  a.used_mask = used;
  a.tile_tensor = p->d_upd_tile_tensor;
  a.factors = factors;
  a.flags = p->d_flags;
  a.n_state = p->n_state_pad;
  a.n_units = static_cast<int32_t>(p->units.size());
  a.k = adamw_consts(hp);
  a.max_norm = hp->max_norm > 0.0f ? hp->max_norm : 0.0f;
  a.inv_m = static_cast<float>(1.0 / static_cast<double>(hp->n_micro));
  update_masked_kernel<<<static_cast<unsigned>(p->n_upd_tiles), MUPD_THREADS, 0, s>>>(a);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace grs
