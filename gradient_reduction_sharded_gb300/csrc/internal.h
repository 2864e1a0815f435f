// Internal types shared by the host plan builder, the C-ABI layer and the
// CUDA launchers of libgrs.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "grs.h"

namespace grs {

// Checked build: every kernel verifies the indices it derives against the
// extents of the buffers they address (the sizes the C ABI documents),
// skips a failing access and records the kernel in FLAG_BOUNDS.
#ifndef GRS_CHECKED
#define GRS_CHECKED 0
#endif

// Reduction tiles: a tile carries STAGE_GRAD_BYTES of gradient input (all the
// group's rank rows for T elements), so T = STAGE_GRAD_BYTES / (esize * group),
// capped at RED_MAX_T, a multiple of 8, and small enough that two stages
// (rank rows plus the old accumulator tile) fit in the shared-memory ring.
// Measured on GB300: each rank row of a tile is one bulk copy, and copies
// of 4 KB and more keep HBM busy where 1-2 KB copies do not.
#ifndef GRS_STAGE_GRAD_BYTES
#define GRS_STAGE_GRAD_BYTES 65536
#endif
#ifndef GRS_RED_MAX_T
#define GRS_RED_MAX_T 8192
#endif
#ifndef GRS_RED_CWARPS
#define GRS_RED_CWARPS 16
#endif
#ifndef GRS_RED_RING_KB
#define GRS_RED_RING_KB 216
#endif
#ifndef GRS_RED_CTAS_PER_SM
#define GRS_RED_CTAS_PER_SM 1
#endif
// L2 policy of the gradient reads: evict-first measured slower than the
// default policy on every workload (most on the accumulating ones, -2.7%).
#ifndef GRS_RED_EVICT_FIRST
#define GRS_RED_EVICT_FIRST 0
#endif
constexpr int64_t RED_RING_BYTES = int64_t(GRS_RED_RING_KB) * 1024;
// Plans whose buckets all reduce at most RED_FEW_ROWS_GROUP bf16 rank rows
// per element (e.g. 4 simulated ranks) run the plain reduction with at most
// RED_FEW_ROWS_STAGES stages in flight per CTA.  Measured on the 3.2B,
// world-4 plan (8192-element tiles of 4 rows): 5.43 ms per launch with 2
// stages against 5.74 with 3 (and 5.51-6.09 for two CTAs per SM with
// smaller rings); the 67M world-16 plan is 5% slower with 2 stages (0.333
// against 0.316 ms) and the 1.1B world-8 one about equal, so wider groups
// keep the ring's full depth.
#ifndef GRS_RED_FEW_ROWS_GROUP
#define GRS_RED_FEW_ROWS_GROUP 4
#endif
#ifndef GRS_RED_FEW_ROWS_STAGES
#define GRS_RED_FEW_ROWS_STAGES 2
#endif
constexpr int RED_FEW_ROWS_GROUP = GRS_RED_FEW_ROWS_GROUP;
constexpr int RED_FEW_ROWS_STAGES = GRS_RED_FEW_ROWS_STAGES;
constexpr int64_t STAGE_GRAD_BYTES = GRS_STAGE_GRAD_BYTES;
constexpr int64_t RED_MAX_T = GRS_RED_MAX_T;
// Consumer warps of the reduction; the norm pass over acc uses the same
// count so that both produce bit-identical per-tile partials.
constexpr int RED_CWARPS = GRS_RED_CWARPS;
// Update (clip + AdamW) and accumulate tiles.
constexpr int64_t UPD_T = 2048;

// One "unit" is one state row of one bucket: bucket b, tp row t.
struct UnitDesc {
  int64_t state_off;  // first element in the state arrays
  int64_t rank_off;   // first element in each rank's gradient buffer
  int64_t padded;     // P: elements of the row (multiple of 8)
  int64_t used;       // valid elements; [used, padded) is padding
  int64_t red_tile0;  // first global reduction tile
  int64_t upd_tile0;  // first global update tile
  int32_t red_T;      // elements per reduction tile
  int32_t g_start;    // group ranks: g_start + i * g_stride, i < g_count
  int32_t g_stride;
  int32_t g_count;
  float scale;        // 1/R, 1/dp or 1 by tag
  int32_t bucket;
};
static_assert(sizeof(UnitDesc) == 72, "UnitDesc layout");

struct Bucket {
  int32_t tag = 0;
  int32_t copies = 1;
  int32_t group_size = 1;
  int32_t n_tensors = 0;
  int64_t used = 0;
  int64_t padded = 0;
  int64_t shard_len = 0;
  int64_t rank_off = 0;
  int64_t state_off = 0;
  int32_t unit0 = 0;  // first unit of the bucket (copies consecutive units)
};

// Segmented-copy job of the gather: `len` elements from state offset
// `src` to element `dst` of tensor `tensor`.
struct GatherJob {
  int64_t src;      // state offset
  int64_t dst;      // offset inside the logical tensor
  int64_t len;
  int64_t chunk0;   // first global chunk of this job
  int64_t logical;  // offset in the canonical logical order (all live tensors, model order)
  int32_t tensor;
  int32_t pad_;
};
// Per update tile, for the update that writes bf16 parameters straight into
// per-tensor storage: the tile's unit, the tensor holding the whole tile
// (-1 when it spans tensors or reaches padding) and the offset of the tile's
// first element inside that tensor; 16 bytes, read in one load.
struct alignas(16) UpdTileInfo {
  int32_t unit;
  int32_t tensor;
  int64_t dst;
};
static_assert(sizeof(UpdTileInfo) == 16, "UpdTileInfo layout");

// Elements per gather / layout chunk (one block each).
#ifndef GRS_GATHER_CHUNK
#define GRS_GATHER_CHUNK 16384
#endif
constexpr int64_t GATHER_CHUNK = GRS_GATHER_CHUNK;

}  // namespace grs

struct grs_plan {
  // inputs
  std::vector<int64_t> numel;
  std::vector<int32_t> owner;
  std::vector<uint32_t> tensor_flags;  // GRS_TENSOR_* per tensor
  std::vector<uint8_t> tensor_live;    // 1 unless frozen (has state in the plan)
  int32_t world = 0, tp = 0, dp_replicate = 0, dp_shard = 0, dp = 0;
  int32_t grad_esize = 2;  // bytes per gradient element: 2 (bf16) or 4 (fp32)
  int32_t red_stage_cap = 0;  // plain bf16 reduction: at most this many stages per CTA (0: no cap)
  // A shard view (grs_plan_shard_view): the state layout of one rank (shard
  // view_shard, tp index view_tp) of a parent plan; -1 for an ordinary plan.
  int32_t view_shard = -1, view_tp = -1;
  int64_t bucket_bytes = 0;
  // layout
  std::vector<int32_t> t_bucket;
  std::vector<int64_t> t_offset;
  std::vector<grs::Bucket> buckets;
  std::vector<grs::UnitDesc> units;
  std::vector<int64_t> red_prefix;  // [n_units + 1] first reduction tile per unit
  std::vector<int64_t> upd_prefix;  // [n_units + 1] first update tile per unit
  std::vector<grs::GatherJob> jobs; // by tensor, LOCAL_SHARD: tp jobs
  std::vector<int32_t> chunk_job;   // [n_gather_chunks]: the job each gather chunk belongs to
  // Tensor segments of every bucket in offset order: segments
  // [bucket_seg0[b], bucket_seg0[b+1]) start at seg_start[] (per-rank element
  // offset inside the bucket) and belong to tensor seg_tensor[].
  std::vector<int64_t> seg_start;
  std::vector<int32_t> seg_tensor;
  std::vector<int32_t> bucket_seg0;
  std::vector<int32_t> tensor_job0; // [n_tensors + 1]
  // Per reduction tile / per update tile: the tensor holding the whole tile,
  // or -1 (the masked passes look a tile's mask bit up in one load).
  std::vector<int32_t> red_tile_tensor;  // [n_red_tiles]
  std::vector<int32_t> upd_tile_tensor;  // [n_upd_tiles]
  // Per reduction tile / per update tile: its unit (the norm, update and
  // accumulate kernels look it up in one load instead of searching the tile
  // prefix).
  std::vector<int32_t> red_tile_unit;    // [n_red_tiles]
  std::vector<int32_t> upd_tile_unit;    // [n_upd_tiles]
  // The gather jobs sorted by state offset, and per update tile the first
  // of them ending after the tile's first element ([n_upd_tiles + 1], the
  // last entry = state_jobs.size()): the fused update + gather's map from a
  // state element to its tensor.
  std::vector<grs::GatherJob> state_jobs;
  std::vector<int32_t> upd_tile_job;
  std::vector<grs::UpdTileInfo> upd_tile_info;  // [n_upd_tiles]
  int64_t n_unique = 0, n_rank_pad = 0, n_state_pad = 0;
  int64_t n_red_tiles = 0, n_upd_tiles = 0, n_gather_chunks = 0;
  int64_t workspace_bytes = 0;
  // device side (absent for host-only plans)
  int device = -1;
  int sm_count = 0;
  grs::UnitDesc* d_units = nullptr;
  int64_t* d_red_prefix = nullptr;
  grs::GatherJob* d_jobs = nullptr;
  int32_t* d_chunk_job = nullptr;
  int64_t* d_seg_start = nullptr;
  int32_t* d_seg_tensor = nullptr;
  int32_t* d_bucket_seg0 = nullptr;
  uint8_t* d_tensor_live = nullptr;
  int32_t* d_red_tile_tensor = nullptr;
  int32_t* d_upd_tile_tensor = nullptr;
  int32_t* d_red_tile_unit = nullptr;
  int32_t* d_upd_tile_unit = nullptr;
  grs::GatherJob* d_state_jobs = nullptr;
  int32_t* d_upd_tile_job = nullptr;
  grs::UpdTileInfo* d_upd_tile_info = nullptr;
  int* d_flags = nullptr;  // [4]: timeout, nonfinite, reserved
  void* host_step_resources = nullptr;  // copy stream + events of grs_step_from_host
};

namespace grs {

// Workspace layout: [n_red_tiles floats: per-tile partial sums of acc^2]
//                   [NORM_L2_BLOCKS doubles: second-level partials]
//                   [one 32-bit ticket counter, zero between calls]
constexpr int NORM_L2_BLOCKS = 128;
inline int64_t ws_partials_offset() { return 0; }
inline int64_t ws_level2_offset(int64_t n_red_tiles) {
  return ((n_red_tiles * 4 + 255) / 256) * 256;
}
inline int64_t ws_ticket_offset(int64_t n_red_tiles) {
  return ws_level2_offset(n_red_tiles) + NORM_L2_BLOCKS * 8;
}
// Bytes the norm needs (partials, level 2, ticket).
inline int64_t ws_bytes(int64_t n_red_tiles) { return ws_ticket_offset(n_red_tiles) + 256; }
// Per-tensor update factors of the masked update ([n_tensors] float2) follow.
inline int64_t ws_factors_offset(int64_t n_red_tiles) { return ws_bytes(n_red_tiles); }

// Device flags
enum : int { FLAG_TIMEOUT = 0, FLAG_NONFINITE = 1, FLAG_AR_MISMATCH = 2, FLAG_BOUNDS = 3, FLAG_COUNT = 4 };

// Kernels of checked builds (GRS_CHECKED=1) record the first failed index
// check as one of these in FLAG_BOUNDS.
enum : int {
  SITE_REDUCE = 1,
  SITE_NORM1 = 2,
  SITE_UPDATE = 3,
  SITE_ACCUMULATE = 4,
  SITE_GATHER = 5,
  SITE_STATE_LOGICAL = 6,
  SITE_NORM1_MASKED = 7,
  SITE_UPDATE_MASKED = 8,
  SITE_AR_CHECK = 9,
  SITE_SMALL = 10,
  SITE_UPDATE_TENSORS = 11,
  SITE_COUNT = 12
};

// Programmatic dependent launch between the path's kernels: measured on
// GB300 (67M workload, back-to-back steps) at 0.6248 ms/step against 0.6214
// without it, so it is off; the kernels keep their griddepcontrol points.
#ifndef GRS_PDL
#define GRS_PDL 0
#endif
#ifndef GRS_UPD_REVERSE
#define GRS_UPD_REVERSE 1
#endif

// Sets the message grs_last_error() returns on this thread (api.cu).
void set_last_error(const std::string& msg);
// Frees the copy stream and events grs_step_from_host created (host_step.cu).
void destroy_host_step_resources(grs_plan* p);

// Host tables of the shard view (shard, tp_index) of `parent` (plan.cpp).
void build_shard_view(const grs_plan& parent, int32_t shard, int32_t tp_index, grs_plan* v);

// host plan builder (plan.cpp)
grs_status build_plan(const int64_t* numels, const int32_t* owners, const uint32_t* tensor_flags,
                      int32_t n, int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                      int64_t bucket_bytes, int32_t grad_esize, grs_plan* p, std::string* why);

// launchers (kernels_*.cu); all return cudaGetLastError() as int
struct ReduceLaunch {
  const void* const* ranks;  // host array [world]
  float* acc;
  float* partials;  // nullptr: no norm epilogue
  int32_t unit_begin, unit_end;
  int64_t state_base, rank_base;
  int64_t state_len, rank_len;  // elements reachable from acc and from each rank pointer
  int32_t accumulate;
  int32_t max_ctas = 0;  // cap on the persistent grid (0: one CTA per SM)
  // Masked reduction (both set, or both null): tiles lying wholly inside a
  // tensor whose used_mask entry is 0 are neither read nor written.
  const uint8_t* used_mask = nullptr;   // device [n_tensors]
  const int32_t* tile_tensor = nullptr; // device [n_red_tiles]: the plan's red_tile_tensor
};
// Skip bits of a masked reduction: one per tile a CTA takes, at most
// RED_SKIP_WORDS * 32 tiles per CTA.
constexpr int RED_SKIP_WORDS = 1024;
int launch_reduce(const grs_plan* p, const ReduceLaunch& a, void* stream);
int launch_norm(const grs_plan* p, const float* acc, int32_t n_micro, void* workspace,
                int32_t partials_ready, double* d_norm_sq, void* stream);
// The AdamW constants of one update (fp32, as the kernels apply them).
struct AdamwK {
  float decay;       // 1 - lr * wd
  float b1, omb1;    // beta1, 1 - beta1
  float b2, omb2;    // beta2, 1 - beta2
  float eps;
};
AdamwK adamw_consts(const grs_adamw* hp);

// Bias-corrected AdamW factors of step `step` computed on the host in fp64
// and rounded to fp32: lr / (1 - beta1^step) and 1 / sqrt(1 - beta2^step).
void bias_factors(const grs_adamw* hp, int32_t step, float* step_size, float* inv_bc2_sqrt);
int launch_update(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq, const float* acc,
                  float* master, float* m, float* v, uint16_t* params, void* stream);
// The update with the bf16 parameters also written to per-tensor storage:
// params (bucket-ordered, may be null) and d_tensor_ptrs (device array of
// one device pointer per tensor, null entries skipped).
int launch_update_to_tensors(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq, const float* acc,
                             float* master, float* m, float* v, uint16_t* params,
                             uint16_t* const* d_tensor_ptrs, void* stream);
int launch_accumulate(const grs_plan* p, int32_t bucket, float* acc, const float* mb, void* stream);
int launch_update_small(const grs_plan* p, const grs_adamw* hp, const void* const* rank_grads, float* acc,
                        float* master, float* m, float* v, uint16_t* params, double* d_norm_sq, void* stream);
int launch_gather(const grs_plan* p, const uint16_t* params, uint16_t* const* tensor_ptrs,
                  void* stream);
int launch_bounded_wait_selftest(const grs_plan* p, uint64_t limit_ns, void* stream);
int launch_check_already_reduced(const grs_plan* p, const void* const* ranks, void* stream);
// fp32 state arrays: bucket layout <-> canonical logical order.
int launch_state_to_logical(const grs_plan* p, const float* state, float* logical, void* stream);
int launch_state_from_logical(const grs_plan* p, const float* logical, float* state, void* stream);
// Second half of the norm: tile partials in `workspace` -> *d_norm_sq.
int launch_norm_finish(const grs_plan* p, int32_t n_micro, void* workspace, double* d_norm_sq,
                       void* stream);
int launch_norm_masked(const grs_plan* p, const float* acc, int32_t n_micro, const uint8_t* used,
                       void* workspace, double* d_norm_sq, void* stream);
int launch_update_masked(const grs_plan* p, const grs_adamw* hp, const double* d_norm_sq,
                         const float* acc, float* master, float* m, float* v, uint16_t* params,
                         const uint8_t* used, int32_t* steps, void* workspace, void* stream);

}  // namespace grs
