// Device helpers for sm_103a: mbarriers with bounded waits, 1-D bulk TMA
// copies, bf16 unpacking, flags.  Inline PTX written for this library.
#pragma once

#include <cstdint>

#include "internal.h"

namespace grs {

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor on the stream is still
// running; pdl_wait() blocks until the predecessor has completed and its
// writes are visible (a no-op for an ordinary launch), pdl_trigger() lets
// this kernel's own successor start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Index checks of checked builds: GRS_CHECK(cond, flags, site) is `cond`,
// and when it is false the site is recorded in flags[FLAG_BOUNDS] (the first
// failure wins).  In ordinary builds it is `true` and compiles away.
__device__ __forceinline__ bool check_or_flag(bool ok, int* flags, int site) {
  if (!ok) atomicCAS(flags + FLAG_BOUNDS, 0, site);
  return ok;
}
#if GRS_CHECKED
#define GRS_CHECK(cond, flags, site) (::grs::check_or_flag((cond), (flags), (site)))
#else
#define GRS_CHECK(cond, flags, site) true
#endif

// A device wait gives up after this long and raises FLAG_TIMEOUT.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with `parity` has completed.  Gives up (returns
// false, raises FLAG_TIMEOUT) after `limit_ns` or when *abort is set by
// another thread of the block.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* flags,
                                                  volatile int* abort, uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(flags + FLAG_TIMEOUT, 1);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// bf16 pair in one 32-bit word -> two floats (exact: bf16 is the high half
// of binary32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void add_bf16x8(float (&a)[8], const uint4& w) {
  a[0] = __fadd_rn(a[0], bf16_lo(w.x));
  a[1] = __fadd_rn(a[1], bf16_hi(w.x));
  a[2] = __fadd_rn(a[2], bf16_lo(w.y));
  a[3] = __fadd_rn(a[3], bf16_hi(w.y));
  a[4] = __fadd_rn(a[4], bf16_lo(w.z));
  a[5] = __fadd_rn(a[5], bf16_hi(w.z));
  a[6] = __fadd_rn(a[6], bf16_lo(w.w));
  a[7] = __fadd_rn(a[7], bf16_hi(w.w));
}

__device__ __forceinline__ void set_bf16x8(float (&a)[8], const uint4& w) {
  a[0] = bf16_lo(w.x);
  a[1] = bf16_hi(w.x);
  a[2] = bf16_lo(w.y);
  a[3] = bf16_hi(w.y);
  a[4] = bf16_lo(w.z);
  a[5] = bf16_hi(w.z);
  a[6] = bf16_lo(w.w);
  a[7] = bf16_hi(w.w);
}

// Sum of eight elements over the rank rows, in rank order: set() takes the
// first rank's 8 elements, add() each further rank's, finish() the sums.
// The rows come from shared memory (set/add: the reduction's TMA stages) or
// global memory (set_g/add_g: 16-byte loads); the arithmetic is the same.
// bf16 rows (16 bytes per 8 elements): plain fp32 adds — a sum of bf16
// values is exact in fp32 unless an input is 2^24 times smaller than the
// largest, so the result is the correctly rounded sum in practice.
// fp32 rows (32 bytes): Knuth's TwoSum keeps each add's rounding error in a
// compensation term added at the end, so the sum is accurate relative to
// the result, not to the operands (where gradients nearly cancel, AdamW's
// g / (|g| + eps) would otherwise magnify an operand-relative error).
template <typename E>
struct Sum8;
template <>
struct Sum8<uint16_t> {
  float v[8];
  __device__ __forceinline__ void set(const uint8_t* p) { set_bf16x8(v, lds128(p)); }
  __device__ __forceinline__ void add(const uint8_t* p) { add_bf16x8(v, lds128(p)); }
  __device__ __forceinline__ void set_g(const uint16_t* p) { set_bf16x8(v, __ldg(reinterpret_cast<const uint4*>(p))); }
  __device__ __forceinline__ void add_g(const uint16_t* p) { add_bf16x8(v, __ldg(reinterpret_cast<const uint4*>(p))); }
  __device__ __forceinline__ void finish(float (&o)[8]) const {
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = v[q];
  }
};
template <>
struct Sum8<float> {
  float v[8], c[8];
  __device__ __forceinline__ void set_w(const uint4& a, const uint4& b) {
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
#pragma unroll
    for (int q = 0; q < 8; ++q) c[q] = 0.0f;
  }
  __device__ __forceinline__ void two_sum(int q, float x) {
    const float t = __fadd_rn(v[q], x);
    const float z = __fsub_rn(t, v[q]);
    const float err = __fadd_rn(__fsub_rn(v[q], __fsub_rn(t, z)), __fsub_rn(x, z));
    c[q] = __fadd_rn(c[q], err);
    v[q] = t;
  }
  __device__ __forceinline__ void add_w(const uint4& a, const uint4& b) {
    two_sum(0, __uint_as_float(a.x)); two_sum(1, __uint_as_float(a.y));
    two_sum(2, __uint_as_float(a.z)); two_sum(3, __uint_as_float(a.w));
    two_sum(4, __uint_as_float(b.x)); two_sum(5, __uint_as_float(b.y));
    two_sum(6, __uint_as_float(b.z)); two_sum(7, __uint_as_float(b.w));
  }
  __device__ __forceinline__ void set(const uint8_t* p) { set_w(lds128(p), lds128(p + 16)); }
  __device__ __forceinline__ void add(const uint8_t* p) { add_w(lds128(p), lds128(p + 16)); }
  __device__ __forceinline__ void set_g(const float* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    set_w(__ldg(q), __ldg(q + 1));
  }
  __device__ __forceinline__ void add_g(const float* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    add_w(__ldg(q), __ldg(q + 1));
  }
  __device__ __forceinline__ void finish(float (&o)[8]) const {
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = __fadd_rn(v[q], c[q]);
  }
};

// Gradient scale of the update: 1/M times the clip coefficient
// c = min(1, max_norm / (sqrt(S) + 1e-6)) (NaN kept), evaluated in fp32 from
// the device-resident S; max_norm <= 0 turns clipping off.  Every update
// kernel uses this one expression.
__device__ __forceinline__ float clip_gscale(double norm_sq, float max_norm, float inv_m) {
  if (!(max_norm > 0.0f)) return inv_m;
  const float cr = max_norm / (sqrtf(static_cast<float>(norm_sq)) + 1e-6f);
  return __fmul_rn((cr < 1.0f || isnan(cr)) ? cr : 1.0f, inv_m);
}

// One AdamW step on one element, in place: torch.optim.AdamW's order of
// operations (decoupled decay, moments, bias-corrected step) in fp32 with
// explicit roundings.  step_size = lr / (1 - beta1^t), inv_bc2_sqrt =
// 1 / sqrt(1 - beta2^t).  Every update kernel uses this one routine.
__device__ __forceinline__ void adamw_elem(float G, float gscale, float step_size, float inv_bc2_sqrt,
                                           const AdamwK& k, float& P, float& M, float& V) {
  const float g = __fmul_rn(G, gscale);
  const float p = __fmul_rn(P, k.decay);
  const float mm = __fmaf_rn(k.b1, M, __fmul_rn(k.omb1, g));
  const float vv = __fmaf_rn(k.b2, V, __fmul_rn(__fmul_rn(k.omb2, g), g));
  const float denom = __fadd_rn(__fmul_rn(__fsqrt_rn(vv), inv_bc2_sqrt), k.eps);
  P = __fsub_rn(p, __fmul_rn(step_size, __fdiv_rn(mm, denom)));
  M = mm;
  V = vv;
}

// Sum over the warp with a fixed butterfly (every lane gets the result).
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = __dadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Every element of a tile counts (the unmasked norm pass).
// ---------------------------------------------------------------- segments
// Element -> tensor inside a bucket row: the row holds its tensors back to
// back; the plan's segment table (start offset, tensor) per bucket is
// searched once and then walked forward.  Used by the passes that take a
// per-step mask of tensors without a gradient.

// Last segment in [lo, hi) whose start is <= e (the first segment starts at 0).
__device__ __forceinline__ int find_seg(const int64_t* __restrict__ start, int lo, int hi, int64_t e) {
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(start + mid) <= e)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

struct Segs {
  const int64_t* start;
  const int32_t* tensor;
  const int32_t* bucket_seg0;
  int32_t n_tensors;  // length of the per-tensor arrays (used mask, steps, factors)
};

// The tensor segment under a forward-moving bucket element: its index, end,
// tensor and whether that tensor has a gradient this step.  Loaded once per
// segment, not once per element.
struct SegCursor {
  int s;
  int hi;         // one past the bucket's last segment
  int64_t end;    // first element after segment s (the bucket's used count for the last)
  int32_t t;      // tensor of segment s (-1 when out of range in a checked build)
  bool on;        // tensor t has a gradient this step
};

__device__ __forceinline__ void seg_load(SegCursor& c, const Segs& sg, const uint8_t* __restrict__ used_mask,
                                         int64_t used, int* flags, int site) {
  c.end = c.s + 1 < c.hi ? __ldg(sg.start + c.s + 1) : used;
  const int32_t t = __ldg(sg.tensor + c.s);
  const bool ok = GRS_CHECK(t >= 0 && t < sg.n_tensors, flags, site);
  c.t = ok ? t : -1;
  c.on = ok && __ldg(used_mask + t) != 0;
}

// Cursor at element e (< used) of a bucket row whose segments are [lo, hi).
__device__ __forceinline__ SegCursor seg_at(const Segs& sg, const uint8_t* __restrict__ used_mask, int lo, int hi,
                                            int64_t e, int64_t used, int* flags, int site) {
  SegCursor c;
  c.s = find_seg(sg.start, lo, hi, e);
  c.hi = hi;
  seg_load(c, sg, used_mask, used, flags, site);
  return c;
}

// Move the cursor forward to element e (< used); zero-length segments
// (zero-size tensors) are stepped over.
__device__ __forceinline__ void seg_advance(SegCursor& c, const Segs& sg, const uint8_t* __restrict__ used_mask,
                                            int64_t e, int64_t used, int* flags, int site) {
  while (e >= c.end && c.s + 1 < c.hi) {
    ++c.s;
    seg_load(c, sg, used_mask, used, flags, site);
  }
}

// Element 8c + q of a tile counts iff it lies in [0, used) of its bucket row
// and in a tensor with a gradient this step.  The cursor keeps the segment
// of the last element asked for ([begin, end)) and seeks again (a binary
// search) only when an element falls outside it.
struct MaskKeep {
  const Segs& sg;
  const uint8_t* __restrict__ used_mask;
  int lo, hi;
  int64_t e0, used;
  int* flags;
  int site;
  SegCursor cur;
  int64_t begin;

  __device__ __forceinline__ bool operator()(int c, int q) {
    const int64_t e = e0 + 8 * int64_t(c) + q;
    if (e >= used) return false;
    if (e < begin || e >= cur.end) {
      cur = seg_at(sg, used_mask, lo, hi, e, used, flags, site);
      begin = __ldg(sg.start + cur.s);
    }
    return cur.on;
  }
};

struct KeepAll {
  __device__ __forceinline__ bool operator()(int, int) const { return true; }
};

// Norm partial (sum of squares) of one reduction tile of nch 8-element
// chunks, computed by ONE warp and bit-identical to the reduction's fused
// epilogue, where RED_CWARPS consumer warps of 32 lanes share the tile:
// consumer thread t = 32 v + l sums, in order, the chunks t, t + 32
// RED_CWARPS, ... with fmaf(x, x, psum) over each chunk's 8 elements; each
// warp's lanes are combined by warp_sum and the warps' sums folded in order
// v = 0, 1, ...  Here the warp plays the consumer warps one after another
// ("virtual warps"), BATCH of them with their loads in flight at once; KE
// is the number of chunks a consumer thread has at most in this tile.  The
// batch changes only how many loads are in flight, never the order of the
// arithmetic.  keep(c, q) == false zeros element 8c + q (a masked pass);
// virtual warps without a chunk add +0 and are skipped.
template <int BATCH, int KE, typename Keep>
__device__ __forceinline__ float tile_partial_warp_k(const float* __restrict__ src, int nch, int lane, Keep& keep) {
  constexpr int CT = 32 * RED_CWARPS;
  float s = 0.0f;
  for (int v0 = 0; v0 < RED_CWARPS && 32 * v0 < nch; v0 += BATCH) {
    float4 x[BATCH][KE][2];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
#pragma unroll
      for (int k = 0; k < KE; ++k) {
        const int c = 32 * (v0 + b) + lane + CT * k;
        if (v0 + b < RED_CWARPS && c < nch) {
          x[b][k][0] = __ldcs(reinterpret_cast<const float4*>(src + 8 * int64_t(c)));
          x[b][k][1] = __ldcs(reinterpret_cast<const float4*>(src + 8 * int64_t(c) + 4));
        } else {
          x[b][k][0] = x[b][k][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int v = v0 + b;
      if (v >= RED_CWARPS || 32 * v >= nch) break;  // warp-uniform
      float psum = 0.0f;
#pragma unroll
      for (int k = 0; k < KE; ++k) {
        const int c = 32 * v + lane + CT * k;
        if (c < nch) {
          float o[8] = {x[b][k][0].x, x[b][k][0].y, x[b][k][0].z, x[b][k][0].w,
                        x[b][k][1].x, x[b][k][1].y, x[b][k][1].z, x[b][k][1].w};
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (!keep(c, q)) o[q] = 0.0f;
#pragma unroll
          for (int q = 0; q < 8; ++q) psum = __fmaf_rn(o[q], o[q], psum);
        }
      }
      psum = warp_sum(psum);
      s = v == 0 ? psum : __fadd_rn(s, psum);
    }
  }
  return s;
}

// SLOTS chunk loads in flight per lane: tiles of at most one chunk per
// consumer thread (nch <= 32 RED_CWARPS, every tile of 4096 elements or
// fewer) play SLOTS virtual warps at a time, larger tiles SLOTS / KMAX.
template <int SLOTS = 8, typename Keep>
__device__ __forceinline__ float tile_partial_warp(const float* __restrict__ src, int nch, int lane, Keep& keep) {
  constexpr int CT = 32 * RED_CWARPS;
  constexpr int KMAX = static_cast<int>(RED_MAX_T / 8 / CT);  // chunks per consumer thread at most
  static_assert(KMAX >= 1 && RED_MAX_T % (8 * CT) == 0, "tile cap must be whole rounds of the consumer threads");
  static_assert(SLOTS % KMAX == 0, "a batch holds whole consumer threads");
  if (KMAX == 1 || nch <= CT) return tile_partial_warp_k<SLOTS, 1>(src, nch, lane, keep);
  return tile_partial_warp_k<SLOTS / KMAX, KMAX>(src, nch, lane, keep);
}

}  // namespace grs
