// Owner-tagged reduction of R simulated ranks' bf16 gradients into an fp32
// accumulator, with the reduce-scatter's shard layout, microbatch
// accumulation and an optional fused norm epilogue.
//
// What it computes ("refactor(distributed): establish shared native TP
// replica ownership", "Why this needs separate work" and "Preserved
// prototype and evidence" — FP32 reduction of BF16 gradients): for each
// element e of a state row,
//     acc[e] (= | +=) scale * sum_{k in group, ascending} float(g_k[e])
// and, on the last microbatch, per-tile partial sums of acc^2 for the
// global norm.
//
// Input: bf16 gradients, or fp32 ones for plans created with
// GRS_PLAN_FP32_GRADS (tiles sized for 4-byte elements).
//
// How (GB300): a persistent grid, one CTA per SM.  Warp 0 is a TMA producer:
// for every tile it issues one 1-D bulk copy (cp.async.bulk) per rank row of
// the tile's reduction group, plus the old accumulator tile when
// accumulating, into a shared-memory ring (as many stages of the largest
// tile as fit in the ring budget, at most 8) guarded by mbarriers.  Unit tables
// are walked forward, never searched, and the consumers get each tile's
// metadata through shared memory.
// The consumer warps take a stage: 16-byte shared loads of 8 bf16 per rank,
// fp32 adds in rank order, scale (and fused add of the old value), padding
// masked to zero, coalesced 16-byte stores, and a fixed-order warp
// butterfly for the norm partial.  The producer folds the consumer warps'
// partials of a tile into one fp32 value in fixed order when the stage is
// recycled, so the partial of a tile never depends on the grid size.
// All mbarrier waits are bounded (device.cuh).
#include <cuda_runtime.h>

#include <atomic>

#include "device.cuh"
#include "internal.h"
#include "launch.cuh"

namespace grs {

namespace {

#ifndef GRS_RED_MAX_STAGES
#define GRS_RED_MAX_STAGES 8
#endif
constexpr int RED_CTHREADS = 32 * RED_CWARPS;
constexpr int RED_THREADS = 32 + RED_CTHREADS;
constexpr int RED_MAX_STAGES = GRS_RED_MAX_STAGES;

// Everything a consumer needs about the tile in one stage (written by the
// producer before it arms the stage's barrier, so consumers touch no global
// tables).
struct StageMeta {
  int64_t tile;
  int64_t out_off;  // acc element offset of the tile's first element
  int32_t n;        // elements in the tile (multiple of 8)
  int32_t valid;    // elements before the padding starts (0..n)
  int32_t gc;       // rank rows in the stage
  float scale;
  // Masked instantiation with norm partials, a tile spanning several
  // tensors: its bucket row's segments [seg_lo, seg_hi) (seg_hi == seg_lo
  // for every other tile), its first element in the row and the row's used
  // count.
  int64_t e0;
  int64_t used;
  int32_t seg_lo;
  int32_t seg_hi;
};

constexpr size_t RED_SMEM_TAIL = 2 * RED_MAX_STAGES * sizeof(uint64_t)        // full/empty
                                 + RED_MAX_STAGES * sizeof(StageMeta)          // tile metadata
                                 + RED_MAX_STAGES * RED_CWARPS * sizeof(float) // warp partials
                                 + 16;                                          // abort flag
// The masked instantiation's largest shared-memory request (ring, tail and
// its two tile bitmaps) within the 227 KB a CTA may opt into.
static_assert(RED_RING_BYTES + RED_SMEM_TAIL + size_t(RED_SKIP_WORDS) * 8 <= 227 * 1024,
              "reduce_kernel shared memory above the per-CTA limit");

struct ReduceArgs {
  const void* ranks[GRS_MAX_WORLD];  // bf16 bits or fp32, by the plan
  float* acc;
  float* partials;
  const UnitDesc* units;
  const int64_t* prefix;
  int* flags;
  int64_t state_base;
  int64_t rank_base;
  int64_t state_len;    // elements reachable from acc
  int64_t rank_len;     // elements reachable from each rank pointer
  int64_t n_partials;   // tiles of the plan (the partials array's length)
  int32_t world;
  int64_t tile_begin;
  int64_t tile_end;
  int32_t unit_begin;
  int32_t unit_end;
  int32_t accumulate;
  int32_t stages;       // ring depth (<= RED_MAX_STAGES)
  int32_t stage_bytes;  // bytes per stage (multiple of 128)
  const uint8_t* used_mask;    // masked instantiation only
  const int32_t* tile_tensor;  // masked instantiation only
  int32_t skip_words;          // masked instantiation only: words of each bitmap after the tail
  int32_t n_tensors;           // masked instantiation only: entries of used_mask
  Segs sg;                     // masked instantiation only: the plan's tensor segments
};

__device__ __forceinline__ float fold_partials(const float* wp) {
  float s = wp[0];
#pragma unroll
  for (int w = 1; w < RED_CWARPS; ++w) s = __fadd_rn(s, wp[w]);
  return s;
}

// kMasked: the masked instantiation (grs_reduce_all_masked).  Before the
// pipeline starts, the CTA marks which of its tiles lie wholly inside a
// tensor without a gradient this step (one bit per tile, from the plan's
// per-tile tensor table and the caller's mask); producer and consumers both
// pass over those tiles, so they are neither read nor written and take no
// stage (their norm partial is +0).  A second bitmap marks the tiles that
// span several tensors: with norm partials wanted, their elements of tensors
// without a gradient count as zero in the partial (a segment cursor per
// consumer thread), which makes the partials those of the masked norm pass
// bit for bit.  The plain instantiation has none of this.
template <typename E, bool kMasked>
__global__ void __launch_bounds__(RED_THREADS, GRS_RED_CTAS_PER_SM) reduce_kernel(const __grid_constant__ ReduceArgs a) {
  constexpr uint32_t ESZ = sizeof(E);
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = a.stages;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * a.stage_bytes);
  uint64_t* empty = full + RED_MAX_STAGES;
  StageMeta* meta = reinterpret_cast<StageMeta*>(empty + RED_MAX_STAGES);
  float* wp = reinterpret_cast<float*>(meta + RED_MAX_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(wp + RED_MAX_STAGES * RED_CWARPS);
  uint32_t* skip = reinterpret_cast<uint32_t*>(smem + size_t(S) * a.stage_bytes + RED_SMEM_TAIL);
  uint32_t* multi = skip + a.skip_words;  // masked: tiles spanning several tensors

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();     // the previous kernel on the stream may still read acc
  pdl_trigger();  // the norm finish / update may start launching
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], RED_CWARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  const int64_t stride = gridDim.x;
  if constexpr (kMasked) {
    // Bit k of the bitmaps: this CTA's k-th tile (tile_begin + blockIdx.x + k * stride)
    // lies in one tensor whose mask entry is 0 (skip), or spans several (multi).
    for (int w = warp; w < a.skip_words; w += RED_THREADS / 32) {
      const int64_t k = int64_t(w) * 32 + lane;
      const int64_t tile = a.tile_begin + blockIdx.x + k * stride;
      bool sk = false, mt = false;
      if (tile < a.tile_end && GRS_CHECK(tile < a.n_partials, a.flags, SITE_REDUCE)) {
        const int32_t t = __ldg(a.tile_tensor + tile);
        sk = t >= 0 && GRS_CHECK(t < a.n_tensors, a.flags, SITE_REDUCE) && __ldg(a.used_mask + t) == 0;
        mt = t < 0;
      }
      const uint32_t bits = __ballot_sync(0xffffffffu, sk);
      const uint32_t mbits = __ballot_sync(0xffffffffu, mt);
      if (lane == 0) {
        skip[w] = bits;
        multi[w] = mbits;
      }
    }
  }
  __syncthreads();
  // Tiles of this CTA it passes over (masked instantiation only).
  auto skipped = [&](int64_t k) -> bool {
    if constexpr (kMasked) return (skip[k >> 5] >> (k & 31)) & 1u;
    return false;
  };
  auto spans = [&](int64_t k) -> bool {
    if constexpr (kMasked) return (multi[k >> 5] >> (k & 31)) & 1u;
    return false;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    const uint64_t pol = GRS_RED_EVICT_FIRST ? l2_policy_evict_first() : l2_policy_evict_normal();
    int64_t iter = 0;
    bool ok = true;
    // The CTA's tiles increase monotonically, so the unit only moves forward.
    int u = a.unit_begin;
    int64_t u_next = __ldg(a.prefix + u + 1);
    UnitDesc ud = a.units[u];
    int32_t seg_lo = 0, seg_hi = 0;  // the unit's bucket segments (masked, with partials)
    const bool seg_need = kMasked && a.partials != nullptr;
    if (seg_need) {
      seg_lo = __ldg(a.sg.bucket_seg0 + ud.bucket);
      seg_hi = __ldg(a.sg.bucket_seg0 + ud.bucket + 1);
    }
    int64_t k = 0;
    for (int64_t tile = a.tile_begin + blockIdx.x; tile < a.tile_end; tile += stride, ++k) {
      if (skipped(k)) {
        if (a.partials != nullptr && lane == 0) a.partials[tile] = 0.0f;
        continue;
      }
      const int s = static_cast<int>(iter % S);
      const uint32_t ph = static_cast<uint32_t>((iter / S) & 1);
      if (tile >= u_next) {
        do {
          ++u;
          u_next = __ldg(a.prefix + u + 1);
        } while (tile >= u_next && (!GRS_CHECKED || u + 1 < a.unit_end));
        ud = a.units[u];
        if (seg_need) {
          seg_lo = __ldg(a.sg.bucket_seg0 + ud.bucket);
          seg_hi = __ldg(a.sg.bucket_seg0 + ud.bucket + 1);
        }
      }
      const int64_t T = ud.red_T;
      const int64_t e0 = (tile - ud.red_tile0) * T;
      const int64_t rem = ud.padded - e0;
      const int32_t n = static_cast<int32_t>(rem < T ? rem : T);
      const int64_t vrem = ud.used - e0;
      const int32_t valid = static_cast<int32_t>(vrem <= 0 ? 0 : (vrem < n ? vrem : n));
      const uint32_t grad_bytes = static_cast<uint32_t>(ud.g_count) * static_cast<uint32_t>(n) * ESZ;
      const uint32_t bytes = grad_bytes + (a.accumulate ? static_cast<uint32_t>(n) * 4u : 0u);
      const int64_t out_off = ud.state_off - a.state_base + e0;
      const int64_t roff = ud.rank_off - a.rank_base + e0;
#if GRS_CHECKED
      {
        // Uniform across the warp: every lane leaves together.
        const int64_t last_rank = int64_t(ud.g_start) + int64_t(ud.g_count - 1) * ud.g_stride;
        const bool in = u < a.unit_end && e0 >= 0 && n > 0 && (n & 7) == 0 && e0 + n <= ud.padded &&
                        bytes <= static_cast<uint32_t>(a.stage_bytes) && out_off >= 0 &&
                        out_off + n <= a.state_len && roff >= 0 && roff + n <= a.rank_len && ud.g_count >= 1 &&
                        ud.g_start >= 0 && last_rank < a.world && (a.partials == nullptr || tile < a.n_partials);
        if (!GRS_CHECK(in, a.flags, SITE_REDUCE)) {
          if (lane == 0) *abort_flag = 1;  // consumers leave their waits
          ok = false;
          break;
        }
      }
#endif
      int good = 1;
      if (lane == 0) good = mbar_wait_bounded(&empty[s], ph ^ 1u, a.flags, abort_flag) ? 1 : 0;
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      uint8_t* st = ring + size_t(s) * a.stage_bytes;
      if (lane == 0) {
        if (a.partials != nullptr && iter >= S) a.partials[meta[s].tile] = fold_partials(wp + s * RED_CWARPS);
        StageMeta& md = meta[s];
        md.tile = tile;
        md.out_off = out_off;
        md.n = n;
        md.valid = valid;
        md.gc = ud.g_count;
        md.scale = ud.scale;
        const bool mixed = seg_need && spans(k);
        md.e0 = e0;
        md.used = ud.used;
        md.seg_lo = mixed ? seg_lo : 0;
        md.seg_hi = mixed ? seg_hi : 0;
        mbar_arrive_expect_tx(&full[s], bytes);
      }
      __syncwarp();
      for (int i = lane; i < ud.g_count; i += 32)
        bulk_g2s(st + size_t(i) * n * ESZ, static_cast<const E*>(a.ranks[ud.g_start + i * ud.g_stride]) + roff,
                 static_cast<uint32_t>(n) * ESZ, &full[s], pol);
      if (a.accumulate && lane == 0)
        bulk_g2s(st + grad_bytes, a.acc + out_off, static_cast<uint32_t>(n) * 4u, &full[s]);
      ++iter;
    }
    if (lane == 0) {
      const int64_t first = iter > S ? iter - S : 0;
      if (ok) {
        // Drain: the last stages' partials become final once consumers release them.
        for (int64_t k = first; k < iter; ++k) {
          const int s = static_cast<int>(k % S);
          if (!mbar_wait_bounded(&empty[s], static_cast<uint32_t>((k / S) & 1), a.flags, abort_flag))
            break;
          if (a.partials != nullptr) a.partials[meta[s].tile] = fold_partials(wp + s * RED_CWARPS);
        }
      }
      if (*abort_flag) {
        // Let every copy this CTA issued land before the CTA exits.
        volatile int no_abort = 0;
        for (int64_t k = first; k < iter; ++k) {
          const int s = static_cast<int>(k % S);
          if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((k / S) & 1), a.flags, &no_abort))
            break;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int ct = threadIdx.x - 32;
    const int cw = ct >> 5;
    int64_t iter = 0;
    int64_t k = 0;
    for (int64_t tile = a.tile_begin + blockIdx.x; tile < a.tile_end; tile += stride, ++k) {
      if (skipped(k)) continue;
      const int s = static_cast<int>(iter % S);
      const uint32_t ph = static_cast<uint32_t>((iter++ / S) & 1);
      if (!mbar_wait_bounded(&full[s], ph, a.flags, abort_flag)) break;
      const StageMeta md = meta[s];
      const int32_t gc = md.gc;
      const int32_t n = md.n;
      float* out = a.acc + md.out_off;
      const uint8_t* st = ring + size_t(s) * a.stage_bytes;
      const size_t row = size_t(n) * ESZ;
      const float* old = reinterpret_cast<const float*>(st + size_t(gc) * row);
      float psum = 0.0f;
      // Masked, tile spanning several tensors: elements of tensors without a
      // gradient add +0 to the partial (the stored values are unspecified).
      const bool mixed = kMasked && md.seg_hi > md.seg_lo;
      MaskKeep keep{a.sg, a.used_mask, md.seg_lo, md.seg_hi, md.e0, md.used, a.flags, SITE_REDUCE,
                    SegCursor{md.seg_lo, md.seg_hi, 0, -1, false}, 0};
      for (int c = ct; c < (n >> 3); c += RED_CTHREADS) {
        const uint8_t* p = st + size_t(c) * 8 * ESZ;
        Sum8<E> sum;
        sum.set(p);
#pragma unroll 4
        for (int i = 1; i < gc; ++i) sum.add(p + i * row);
        float v[8];
        sum.finish(v);
        float o[8];
        if (a.accumulate) {
          const uint4 q0 = lds128(old + c * 8);
          const uint4 q1 = lds128(old + c * 8 + 4);
          const float ov[8] = {__uint_as_float(q0.x), __uint_as_float(q0.y), __uint_as_float(q0.z),
                               __uint_as_float(q0.w), __uint_as_float(q1.x), __uint_as_float(q1.y),
                               __uint_as_float(q1.z), __uint_as_float(q1.w)};
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = __fmaf_rn(v[q], md.scale, ov[q]);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = __fmul_rn(v[q], md.scale);
        }
        const int el = c * 8;
        if (el + 8 > md.valid) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (el + q >= md.valid) o[q] = 0.0f;
        }
        float4* o4 = reinterpret_cast<float4*>(out + el);
        o4[0] = make_float4(o[0], o[1], o[2], o[3]);
        o4[1] = make_float4(o[4], o[5], o[6], o[7]);
        if (mixed) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float x = keep(c, q) ? o[q] : 0.0f;
            psum = __fmaf_rn(x, x, psum);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) psum = __fmaf_rn(o[q], o[q], psum);
        }
      }
      if (a.partials != nullptr) {
        psum = warp_sum(psum);
        if (lane == 0) wp[s * RED_CWARPS + cw] = psum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// Whether the dynamic shared-memory cap is raised, per (gradient type,
// device); plans on several host threads may launch at once.
std::atomic<bool> g_attr_set[2][2][64] = {};

}  // namespace

int launch_reduce(const grs_plan* p, const ReduceLaunch& l, void* stream) {
  ReduceArgs a;
  for (int k = 0; k < GRS_MAX_WORLD; ++k) a.ranks[k] = k < p->world ? l.ranks[k] : nullptr;
  a.acc = l.acc;
  a.partials = l.partials;
  a.units = p->d_units;
  a.prefix = p->d_red_prefix;
  a.flags = p->d_flags;
  a.state_base = l.state_base;
  a.rank_base = l.rank_base;
  a.state_len = l.state_len;
  a.rank_len = l.rank_len;
  a.n_partials = p->n_red_tiles;
  a.world = p->world;
  a.unit_begin = l.unit_begin;
  a.unit_end = l.unit_end;
  a.tile_begin = p->red_prefix[l.unit_begin];
  a.tile_end = p->red_prefix[l.unit_end];
  a.accumulate = l.accumulate;
  const bool masked = l.used_mask != nullptr;
  a.used_mask = l.used_mask;
  a.tile_tensor = l.tile_tensor;
  a.n_tensors = static_cast<int32_t>(p->numel.size());
  a.sg = Segs{p->d_seg_start, p->d_seg_tensor, p->d_bucket_seg0, a.n_tensors};
  const int64_t tiles = a.tile_end - a.tile_begin;
  if (tiles <= 0) return 0;
  // Stage size: the largest tile of the launched units (rank rows plus the
  // old accumulator tile when accumulating), rounded to 128 bytes.
  int64_t need = 128;
  for (int32_t u = l.unit_begin; u < l.unit_end; ++u) {
    const UnitDesc& d = p->units[u];
    const int64_t b = int64_t(d.g_count) * d.red_T * p->grad_esize + (l.accumulate ? int64_t(d.red_T) * 4 : 0);
    need = b > need ? b : need;
  }
  need = (need + 127) / 128 * 128;
  int stages = static_cast<int>(RED_RING_BYTES / need);  // >= 2 by the plan's tile cap
  stages = stages > RED_MAX_STAGES ? RED_MAX_STAGES : stages;
  // Plans with few rank rows per element: a shallower ring for the plain
  // reduction (grs_plan::red_stage_cap, RED_FEW_ROWS_*).
  if (!masked && p->red_stage_cap > 0 && stages > p->red_stage_cap) stages = p->red_stage_cap;
  if (stages < 2) return static_cast<int>(cudaErrorInvalidConfiguration);
  a.stages = stages;
  a.stage_bytes = static_cast<int32_t>(need);
  int64_t cap = int64_t(p->sm_count) * GRS_RED_CTAS_PER_SM;
  if (l.max_ctas > 0 && l.max_ctas < cap) cap = l.max_ctas;
  const int64_t grid = tiles < cap ? tiles : cap;
  const int64_t per_cta = (tiles + grid - 1) / grid;
  a.skip_words = masked ? static_cast<int32_t>((per_cta + 31) / 32) : 0;
  if (a.skip_words > RED_SKIP_WORDS) return static_cast<int>(cudaErrorInvalidValue);
  const size_t smem = size_t(stages) * need + RED_SMEM_TAIL + size_t(a.skip_words) * 8;  // two bitmaps
  const int f32 = p->grad_esize == 4 ? 1 : 0;
  const int mk = masked ? 1 : 0;
  if (p->device >= 0 && p->device < 64 && !g_attr_set[f32][mk][p->device].load(std::memory_order_acquire)) {
    const int bytes = static_cast<int>(RED_RING_BYTES + RED_SMEM_TAIL + (masked ? RED_SKIP_WORDS * 8 : 0));
    cudaError_t e;
    if (f32)
      e = masked ? cudaFuncSetAttribute(reduce_kernel<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
                 : cudaFuncSetAttribute(reduce_kernel<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    else
      e = masked ? cudaFuncSetAttribute(reduce_kernel<uint16_t, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
                 : cudaFuncSetAttribute(reduce_kernel<uint16_t, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_attr_set[f32][mk][p->device].store(true, std::memory_order_release);
  }
  const dim3 gd(static_cast<unsigned>(grid));
  const dim3 bd(static_cast<unsigned>(RED_THREADS));
  cudaError_t e;
  if (f32)
    e = masked ? launch_k(reduce_kernel<float, true>, gd, bd, smem, stream, a)
               : launch_k(reduce_kernel<float, false>, gd, bd, smem, stream, a);
  else
    e = masked ? launch_k(reduce_kernel<uint16_t, true>, gd, bd, smem, stream, a)
               : launch_k(reduce_kernel<uint16_t, false>, gd, bd, smem, stream, a);
  return static_cast<int>(e);
}

}  // namespace grs
