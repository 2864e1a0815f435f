// The whole update of a small plan in one launch: every microbatch's
// owner-tagged reduction, the global norm, clip and AdamW with the bf16
// cast ("refactor(distributed): establish shared native TP replica
// ownership", "Preserved prototype and evidence" and "Proposed scope": FP32
// reduction, accumulation, global-norm clipping, optimizer update).
//
// For plans of at most GRS_SMALL_MAX_TILES reduction tiles, where the
// multi-kernel path is bound by its four launches rather than by memory.
// One thread-block cluster of 16 CTAs, in four phases separated by cluster
// barriers:
//  1. every thread of the cluster reduces 8-element chunks of every tile
//     over all microbatches (the reduction kernel's arithmetic: ranks in
//     group order, fp32 sums or compensated fp32 sums, fmul by the tag's
//     scale on the first microbatch and fma onto the running value after)
//     and writes the accumulator;
//  2. CTA t % 16 forms tile t's norm partial in the fused epilogue's order
//     (its 16 warps play the reduction's 16 consumer warps, lanes combined
//     by the same butterfly, warps folded in order) into its shared memory;
//  3. every CTA reads the partials from the owners' shared memory
//     (distributed shared memory) and folds them in the norm finish
//     kernel's order, which for at most 128 tiles gives each second-level
//     sum exactly one partial;
//  4. every thread updates 8-element chunks with the update kernel's
//     arithmetic.
// Results equal the multi-kernel path bit for bit.  Accumulator values
// written by another CTA are read through L2 (ld.global.cg) after the
// barrier that publishes them.
//
// No thread leaves before the three cluster barriers: every loop before
// them is bounded by the plan's tile count, and checked builds skip
// accesses instead of returning.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "device.cuh"
#include "internal.h"

namespace grs {

namespace {

constexpr int SMALL_THREADS = 512;
// CTAs in the cluster: 16, beyond the portable 8, measured fastest on GB300
// (one tiny-plan update: 12.3 us against 14.4 with 8, 18.8 with 4).
#ifndef GRS_SMALL_CLUSTER
#define GRS_SMALL_CLUSTER 16
#endif
constexpr int SMALL_MAX_CLUSTER = GRS_SMALL_CLUSTER;
static_assert(GRS_SMALL_MAX_TILES <= NORM_L2_BLOCKS,
              "the norm replay assumes one partial per second-level block");

struct SmallArgs {
  const void* ranks[GRS_SMALL_MAX_BUFFERS];  // [j * world + k]
  float* acc;
  float* master;
  float* m;
  float* v;
  uint16_t* params;
  double* norm_out;
  const UnitDesc* units;
  const int64_t* prefix;
  int* flags;
  int64_t n_state;
  int64_t rank_len;
  int32_t n_tiles;
  int32_t n_units;
  int32_t world;
  int32_t n_micro;
  double inv_m2;
  AdamwK k;
  float step_size, inv_bc2_sqrt;
  float max_norm;
  float inv_m;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

// Every thread of every CTA of the cluster arrives and waits: writes before
// it (shared, global) are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float in the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float x;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(remote) : "memory");
  return x;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// What the phases need of one reduction tile, gathered once per CTA.
struct SmallTile {
  int64_t out;    // first accumulator / state element
  int64_t roff;   // first element in each rank buffer
  int64_t e0;     // first element within its unit (row)
  int64_t used;   // the unit's valid elements
  int32_t n;      // elements (multiple of 8; 0 when a checked build rejects the tile)
  int32_t valid;  // elements before the padding
  int32_t g_start, g_stride, g_count;
  float scale;
};

template <typename E>
__global__ void __launch_bounds__(SMALL_THREADS) small_update_kernel(const __grid_constant__ SmallArgs a) {
  __shared__ float part[GRS_SMALL_MAX_TILES];  // this CTA's tiles' partials, at their plan index
  __shared__ float vsum[RED_CWARPS];           // one tile's virtual-warp sums
  __shared__ double s_norm;
  __shared__ int64_t s_prefix[GRS_SMALL_MAX_TILES + 1];  // the plan's first tile per unit
  __shared__ int64_t s_c0[GRS_SMALL_MAX_TILES + 1];      // first chunk of each tile
  __shared__ SmallTile s_tile[GRS_SMALL_MAX_TILES];
  __shared__ UnitDesc s_units[GRS_SMALL_MAX_TILES];
  const uint32_t crank = cluster_rank();
  const uint32_t csize = cluster_size();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t gthread = int64_t(crank) * SMALL_THREADS + threadIdx.x;  // thread index in the cluster
  const int64_t gstride = int64_t(csize) * SMALL_THREADS;
  const int32_t n_tiles = a.n_tiles;

  // ---- 0. the tile table: the unit prefix and descriptors in one round of
  // coalesced reads, then each thread t < n_tiles describes tile t; a prefix
  // sum gives chunk offsets
  for (int i = threadIdx.x; i <= a.n_units; i += SMALL_THREADS) s_prefix[i] = __ldg(a.prefix + i);
  {
    constexpr int W = static_cast<int>(sizeof(UnitDesc) / 8);
    const int64_t* src = reinterpret_cast<const int64_t*>(a.units);
    int64_t* dst = reinterpret_cast<int64_t*>(s_units);
    for (int i = threadIdx.x; i < a.n_units * W; i += SMALL_THREADS) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < n_tiles; t += SMALL_THREADS) {
    int u = 0, uh = a.n_units;  // the unit holding tile t: last u with s_prefix[u] <= t
    while (uh - u > 1) {
      const int mid = (u + uh) >> 1;
      if (s_prefix[mid] <= t) u = mid; else uh = mid;
    }
    const UnitDesc& ud = s_units[u];
    SmallTile st;
    st.e0 = (t - ud.red_tile0) * int64_t(ud.red_T);
    const int64_t rem = ud.padded - st.e0;
    st.n = static_cast<int32_t>(rem < ud.red_T ? rem : ud.red_T);
    st.out = ud.state_off + st.e0;
    st.roff = ud.rank_off + st.e0;
    st.used = ud.used;
    const int64_t vrem = ud.used - st.e0;
    st.valid = static_cast<int32_t>(vrem <= 0 ? 0 : (vrem < st.n ? vrem : st.n));
    st.g_start = ud.g_start;
    st.g_stride = ud.g_stride;
    st.g_count = ud.g_count;
    st.scale = ud.scale;
    if (!GRS_CHECK(st.e0 >= 0 && st.n > 0 && (st.n & 7) == 0 && st.out + st.n <= a.n_state &&
                       st.roff + st.n <= a.rank_len && ud.g_count >= 1 &&
                       ud.g_start + int64_t(ud.g_count - 1) * ud.g_stride < a.world,
                   a.flags, SITE_SMALL))
      st.n = 0;
    s_tile[t] = st;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t c0 = 0;
    for (int t = 0; t < n_tiles; ++t) {
      s_c0[t] = c0;
      c0 += s_tile[t].n >> 3;
    }
    s_c0[n_tiles] = c0;
  }
  __syncthreads();
  const int64_t n_chunks = s_c0[n_tiles];
  // The optimizer state this thread updates in phase 4, fetched into L2 now
  // (nothing waits for it) so that phase 4 does not wait on memory.
  for (int64_t g = gthread; g < n_chunks; g += gstride) {
    int lo = 0, hi = n_tiles;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_c0[mid] <= g) lo = mid; else hi = mid;
    }
    const int64_t i = s_tile[lo].out + 8 * (g - s_c0[lo]);
    prefetch_l2(a.master + i);
    prefetch_l2(a.m + i);
    prefetch_l2(a.v + i);
  }

  // ---- 1. reduction over the microbatches into the accumulator: the
  // cluster's threads take the plan's 8-element chunks in turn
  for (int64_t g = gthread; g < n_chunks; g += gstride) {
    int lo = 0, hi = n_tiles;  // the tile holding chunk g: last t with s_c0[t] <= g
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_c0[mid] <= g) lo = mid; else hi = mid;
    }
    const SmallTile& st = s_tile[lo];
    const int64_t c = g - s_c0[lo];
    float accv[8];
    for (int32_t j = 0; j < a.n_micro; ++j) {
      const void* const* rk = a.ranks + int64_t(j) * a.world;
      Sum8<E> sum;
      sum.set_g(static_cast<const E*>(rk[st.g_start]) + st.roff + 8 * c);
#pragma unroll 4
      for (int i = 1; i < st.g_count; ++i)
        sum.add_g(static_cast<const E*>(rk[st.g_start + i * st.g_stride]) + st.roff + 8 * c);
      float s8[8];
      sum.finish(s8);
#pragma unroll
      for (int q = 0; q < 8; ++q) accv[q] = j == 0 ? __fmul_rn(s8[q], st.scale) : __fmaf_rn(s8[q], st.scale, accv[q]);
    }
    const int64_t el = 8 * c;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (el + q >= st.valid) accv[q] = 0.0f;
    float4* o4 = reinterpret_cast<float4*>(a.acc + st.out + el);
    o4[0] = make_float4(accv[0], accv[1], accv[2], accv[3]);
    o4[1] = make_float4(accv[4], accv[5], accv[6], accv[7]);
  }
  cluster_sync_all();  // the whole accumulator is written

  // ---- 2. tile partials, the fused epilogue's order: CTA t % C owns tile
  // t; its warp v plays consumer warp v (chunks 32 v + lane + 32 RED_CWARPS k,
  // in k order), lanes combined by warp_sum, warps folded in order.
  constexpr int CT = 32 * RED_CWARPS;
  constexpr int KMAX = static_cast<int>(RED_MAX_T / 8 / CT);
  static_assert(SMALL_THREADS == CT, "one warp per consumer warp of the reduction");
  for (int32_t tile = static_cast<int32_t>(crank); tile < n_tiles; tile += static_cast<int32_t>(csize)) {
    const SmallTile& st = s_tile[tile];
    const float* src = a.acc + st.out;
    float psum = 0.0f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int c = 32 * warp + lane + CT * k;
      if (c < (st.n >> 3)) {
        const float4 x0 = __ldcg(reinterpret_cast<const float4*>(src + 8 * c));
        const float4 x1 = __ldcg(reinterpret_cast<const float4*>(src + 8 * c + 4));
        const float o[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) psum = __fmaf_rn(o[q], o[q], psum);
      }
    }
    psum = warp_sum(psum);
    if (lane == 0) vsum[warp] = psum;
    __syncthreads();
    if (threadIdx.x == 0) {
      float f = vsum[0];
#pragma unroll
      for (int w = 1; w < RED_CWARPS; ++w) f = __fadd_rn(f, vsum[w]);
      part[tile] = f;
    }
    __syncthreads();
  }
  cluster_sync_all();  // every tile's partial is published

  // ---- 3. global norm: the finish kernel's order.  With at most 128 tiles
  // its second-level block b holds partial b alone (or nothing), and its
  // last block sums the 128 second-level values with 8 warp butterflies
  // folded in order; the warps past tile 127 add +0 and are skipped.
  if (warp == 0) {
    double s = 0.0;
    for (int w = 0; 32 * w < n_tiles; ++w) {
      const int t = 32 * w + lane;
      const double x = t < n_tiles ? static_cast<double>(ld_cluster_f32(&part[t], static_cast<uint32_t>(t) % csize))
                                   : 0.0;
      const double r = warp_sum(x);
      s = w == 0 ? r : __dadd_rn(s, r);
    }
    if (lane == 0) s_norm = __dmul_rn(s, a.inv_m2);
  }
  cluster_sync_all();  // every remote read is done before any CTA moves on

  const double S = s_norm;
  if (crank == 0 && threadIdx.x == 0) {
    *a.norm_out = S;
    if (!isfinite(S)) atomicOr(a.flags + FLAG_NONFINITE, 1);
  }

  // ---- 4. clip + AdamW + bf16, the cluster's threads on the chunks in turn
  const float gscale = clip_gscale(S, a.max_norm, a.inv_m);
  for (int64_t g = gthread; g < n_chunks; g += gstride) {
    int lo = 0, hi = n_tiles;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_c0[mid] <= g) lo = mid; else hi = mid;
    }
    const SmallTile& st = s_tile[lo];
    const int64_t c = g - s_c0[lo];
    const int64_t el = st.e0 + 8 * c;  // element within the unit
    const int64_t i = st.out + 8 * c;
    const float4 g0 = __ldcg(reinterpret_cast<const float4*>(a.acc + i));
    const float4 g1 = __ldcg(reinterpret_cast<const float4*>(a.acc + i + 4));
    const float4 p0 = reinterpret_cast<const float4*>(a.master + i)[0];
    const float4 p1 = reinterpret_cast<const float4*>(a.master + i + 4)[0];
    const float4 m0 = reinterpret_cast<const float4*>(a.m + i)[0];
    const float4 m1 = reinterpret_cast<const float4*>(a.m + i + 4)[0];
    const float4 v0 = reinterpret_cast<const float4*>(a.v + i)[0];
    const float4 v1 = reinterpret_cast<const float4*>(a.v + i + 4)[0];
    const float G[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float P[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    float M[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float V[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      adamw_elem(G[q], gscale, a.step_size, a.inv_bc2_sqrt, a.k, P[q], M[q], V[q]);
      if (el + q >= st.used) P[q] = M[q] = V[q] = 0.0f;  // padding
    }
    reinterpret_cast<float4*>(a.master + i)[0] = make_float4(P[0], P[1], P[2], P[3]);
    reinterpret_cast<float4*>(a.master + i + 4)[0] = make_float4(P[4], P[5], P[6], P[7]);
    reinterpret_cast<float4*>(a.m + i)[0] = make_float4(M[0], M[1], M[2], M[3]);
    reinterpret_cast<float4*>(a.m + i + 4)[0] = make_float4(M[4], M[5], M[6], M[7]);
    reinterpret_cast<float4*>(a.v + i)[0] = make_float4(V[0], V[1], V[2], V[3]);
    reinterpret_cast<float4*>(a.v + i + 4)[0] = make_float4(V[4], V[5], V[6], V[7]);
    uint4 h;
    h.x = pack_bf16x2(P[0], P[1]);
    h.y = pack_bf16x2(P[2], P[3]);
    h.z = pack_bf16x2(P[4], P[5]);
    h.w = pack_bf16x2(P[6], P[7]);
    reinterpret_cast<uint4*>(a.params + i)[0] = h;
  }
}

// Whether the non-portable cluster size is allowed yet, per (gradient
// type, device).
std::atomic<bool> g_cluster_attr_set[2][64] = {};

}  // namespace

int launch_update_small(const grs_plan* p, const grs_adamw* hp, const void* const* rank_grads, float* acc,
                        float* master, float* m, float* v, uint16_t* params, double* d_norm_sq, void* stream) {
  SmallArgs a;
  const int64_t nbuf = int64_t(hp->n_micro) * p->world;
  for (int64_t k = 0; k < GRS_SMALL_MAX_BUFFERS; ++k) a.ranks[k] = k < nbuf ? rank_grads[k] : nullptr;
  a.acc = acc;
  a.master = master;
  a.m = m;
  a.v = v;
  a.params = params;
  a.norm_out = d_norm_sq;
  a.units = p->d_units;
  a.prefix = p->d_red_prefix;
  a.flags = p->d_flags;
  a.n_state = p->n_state_pad;
  a.rank_len = p->n_rank_pad;
  a.n_tiles = static_cast<int32_t>(p->n_red_tiles);
  a.n_units = static_cast<int32_t>(p->units.size());
  a.world = p->world;
  a.n_micro = hp->n_micro;
  const double inv_m = 1.0 / static_cast<double>(hp->n_micro);
  a.inv_m2 = inv_m * inv_m;
  a.k = adamw_consts(hp);
  bias_factors(hp, hp->step, &a.step_size, &a.inv_bc2_sqrt);
  a.max_norm = hp->max_norm > 0.0f ? hp->max_norm : 0.0f;
  a.inv_m = static_cast<float>(inv_m);

  const unsigned csize = SMALL_MAX_CLUSTER;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(SMALL_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int f32 = p->grad_esize == 4 ? 1 : 0;
  if (SMALL_MAX_CLUSTER > 8 && p->device >= 0 && p->device < 64 &&
      !g_cluster_attr_set[f32][p->device].load(std::memory_order_acquire)) {  // beyond the portable size
    const cudaError_t ea = f32 ? cudaFuncSetAttribute(small_update_kernel<float>,
                                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1)
                               : cudaFuncSetAttribute(small_update_kernel<uint16_t>,
                                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (ea != cudaSuccess) return static_cast<int>(ea);
    g_cluster_attr_set[f32][p->device].store(true, std::memory_order_release);
  }
  const cudaError_t e = p->grad_esize == 4 ? cudaLaunchKernelEx(&cfg, small_update_kernel<float>, a)
                                           : cudaLaunchKernelEx(&cfg, small_update_kernel<uint16_t>, a);
  return static_cast<int>(e);
}

}  // namespace grs
