// Host-side reduction plan: owner routing, buckets, padding, shards, tile
// tables.  Pure C++ (no CUDA); the C-ABI layer uploads the tables.
//
// Rules ("refactor(distributed): establish shared native TP replica
// ownership", "Why this needs separate work" and "Proposed scope": one
// owner per parameter, unsupported compositions rejected; "Cosmos 3 ...
// distributed parallelism", section 1: dp_replicate x dp_shard = world,
// dp_shard = -1 auto; Mixle "Distributed Transformer Training", "Optimizer
// and checkpoint semantics": plan from the logical parameter list):
//  * buckets are tag-homogeneous, in tag order RA, PS, LS, AR, model order
//    within a tag, greedy on per-rank bf16 bytes (2 bytes per element, also
//    for fp32 gradient plans, so both share one layout), tensors never split;
//  * a LOCAL_SHARD tensor holds numel/tp elements per rank;
//  * buckets are padded to a multiple of 8 * dp_shard elements so every
//    shard starts on a 16-byte boundary;
//  * state rows: tp per LOCAL_SHARD bucket, one otherwise.
#include <algorithm>
#include <string>

#include "internal.h"

namespace grs {

namespace {

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

// Tiles of T elements over one row of bucket b: for each, the tensor whose
// segment holds the whole tile, or -1.  The bucket's segments tile [0, used)
// in offset order (zero-size tensors give empty segments, stepped over).
void sole_tensors(const grs_plan& p, int32_t b, int64_t T, std::vector<int32_t>& out) {
  const int32_t s0 = p.bucket_seg0[b], s1 = p.bucket_seg0[b + 1];
  const int64_t used = p.buckets[b].used, padded = p.buckets[b].padded;
  int32_t s = s0;
  for (int64_t e0 = 0; e0 < padded; e0 += T) {
    const int64_t e1 = std::min(padded, e0 + T);
    int32_t sole = -1;
    if (e1 <= used && s0 < s1) {
      while (s + 1 < s1 && p.seg_start[s + 1] <= e0) ++s;  // the segment holding e0
      const int64_t end = s + 1 < s1 ? p.seg_start[s + 1] : used;
      if (e1 <= end) sole = p.seg_tensor[s];
    }
    out.push_back(sole);
  }
}

int32_t group_size_of(int32_t tag, const grs_plan& p) {
  switch (tag) {
    case GRS_REPLICA_AVG:
    case GRS_PARTIAL_SUM:
      return p.world;
    case GRS_LOCAL_SHARD:
      return p.dp;
    default:
      return 1;
  }
}

}  // namespace

grs_status build_plan(const int64_t* numels, const int32_t* owners, const uint32_t* tensor_flags,
                      int32_t n, int32_t world, int32_t tp, int32_t dp_replicate, int32_t dp_shard,
                      int64_t bucket_bytes, int32_t grad_esize, grs_plan* p, std::string* why) {
  if (n <= 0 || numels == nullptr || owners == nullptr) {
    *why = "plan needs at least one tensor (numels/owners non-null)";
    return GRS_ERR_INVALID_ARG;
  }
  if (bucket_bytes <= 0) {
    *why = "bucket_bytes must be positive";
    return GRS_ERR_INVALID_ARG;
  }
  if (world <= 0 || world > GRS_MAX_WORLD || tp <= 0 || dp_replicate <= 0 ||
      (dp_shard <= 0 && dp_shard != -1)) {
    *why = "degrees must be positive (dp_shard may be -1) and world <= GRS_MAX_WORLD";
    return GRS_ERR_INVALID_ARG;
  }
  if (dp_shard == -1) {
    if (world % (tp * dp_replicate) != 0) {
      *why = "dp_shard=-1: world is not a multiple of tp * dp_replicate";
      return GRS_ERR_UNSUPPORTED_COMPOSITION;
    }
    dp_shard = world / (tp * dp_replicate);
  }
  if (static_cast<int64_t>(tp) * dp_replicate * dp_shard != world) {
    *why = "tp * dp_replicate * dp_shard != world";
    return GRS_ERR_UNSUPPORTED_COMPOSITION;
  }
  for (int32_t i = 0; i < n; ++i) {
    if (owners[i] < GRS_REPLICA_AVG || owners[i] > GRS_ALREADY_REDUCED) {
      *why = "tensor " + std::to_string(i) + ": unknown owner tag " + std::to_string(owners[i]);
      return GRS_ERR_INVALID_ARG;
    }
    if (numels[i] < 0) {
      *why = "tensor " + std::to_string(i) + ": negative numel";
      return GRS_ERR_SHAPE;
    }
    if (owners[i] == GRS_LOCAL_SHARD && numels[i] % tp != 0) {
      *why = "tensor " + std::to_string(i) + ": LOCAL_SHARD numel not divisible by tp";
      return GRS_ERR_SHAPE;
    }
    if (tensor_flags != nullptr && (tensor_flags[i] & ~GRS_TENSOR_FROZEN) != 0) {
      *why = "tensor " + std::to_string(i) + ": unknown tensor flag bits";
      return GRS_ERR_INVALID_ARG;
    }
  }
  // A frozen tensor (no gradient, no optimizer state) takes no place in the plan.
  auto frozen = [&](int32_t i) { return tensor_flags != nullptr && (tensor_flags[i] & GRS_TENSOR_FROZEN) != 0; };

  p->numel.assign(numels, numels + n);
  p->owner.assign(owners, owners + n);
  p->tensor_flags.assign(n, 0u);
  if (tensor_flags != nullptr) p->tensor_flags.assign(tensor_flags, tensor_flags + n);
  p->tensor_live.assign(n, 1);
  for (int32_t i = 0; i < n; ++i) p->tensor_live[i] = frozen(i) ? 0 : 1;
  p->world = world;
  p->tp = tp;
  p->dp_replicate = dp_replicate;
  p->dp_shard = dp_shard;
  p->dp = dp_replicate * dp_shard;
  p->bucket_bytes = bucket_bytes;
  p->grad_esize = grad_esize;
  p->t_bucket.assign(n, -1);
  p->t_offset.assign(n, 0);
  p->buckets.clear();
  p->n_unique = 0;
  for (int32_t i = 0; i < n; ++i)
    if (!frozen(i)) p->n_unique += numels[i];

  // Greedy, tag-homogeneous buckets.
  for (int32_t tag = GRS_REPLICA_AVG; tag <= GRS_ALREADY_REDUCED; ++tag) {
    Bucket* cur = nullptr;
    for (int32_t i = 0; i < n; ++i) {
      if (owners[i] != tag || frozen(i)) continue;
      const int64_t per_rank = (tag == GRS_LOCAL_SHARD) ? numels[i] / tp : numels[i];
      if (cur != nullptr && cur->used > 0 && 2 * (cur->used + per_rank) > bucket_bytes) cur = nullptr;
      if (cur == nullptr) {
        p->buckets.emplace_back();
        cur = &p->buckets.back();
        cur->tag = tag;
        cur->copies = (tag == GRS_LOCAL_SHARD) ? tp : 1;
        cur->group_size = group_size_of(tag, *p);
      }
      p->t_bucket[i] = static_cast<int32_t>(p->buckets.size() - 1);
      p->t_offset[i] = cur->used;
      cur->used += per_rank;
      cur->n_tensors += 1;
    }
  }

  // Padding, shards, offsets, units and tiles.
  const int64_t quantum = 8 * static_cast<int64_t>(dp_shard);
  p->units.clear();
  p->red_prefix.assign(1, 0);
  p->upd_prefix.assign(1, 0);
  int64_t rank_off = 0, state_off = 0, red_tiles = 0, upd_tiles = 0;
  int32_t max_group = 0;
  for (const Bucket& bk : p->buckets) max_group = std::max(max_group, bk.group_size);
  p->red_stage_cap = (grad_esize == 2 && max_group <= RED_FEW_ROWS_GROUP) ? RED_FEW_ROWS_STAGES : 0;
  for (size_t b = 0; b < p->buckets.size(); ++b) {
    Bucket& bk = p->buckets[b];
    bk.padded = round_up(bk.used, quantum);
    bk.shard_len = bk.padded / dp_shard;
    bk.rank_off = rank_off;
    bk.state_off = state_off;
    bk.unit0 = static_cast<int32_t>(p->units.size());
    const int64_t gsz = bk.group_size;
    const int64_t es = grad_esize;
    int64_t T = std::min<int64_t>(STAGE_GRAD_BYTES / (es * gsz), RED_RING_BYTES / (2 * (es * gsz + 4)));
    T = std::min<int64_t>(RED_MAX_T, std::max<int64_t>(8, T / 8 * 8));
    for (int32_t t = 0; t < bk.copies; ++t) {
      UnitDesc u{};
      u.state_off = state_off + static_cast<int64_t>(t) * bk.padded;
      u.rank_off = rank_off;
      u.padded = bk.padded;
      u.used = bk.used;
      u.red_tile0 = red_tiles;
      u.upd_tile0 = upd_tiles;
      u.red_T = static_cast<int32_t>(T);
      u.bucket = static_cast<int32_t>(b);
      switch (bk.tag) {
        case GRS_REPLICA_AVG:  // average across TP and DP: all ranks
          u.g_start = 0; u.g_stride = 1; u.g_count = world;
          u.scale = 1.0f / static_cast<float>(world);
          break;
        case GRS_PARTIAL_SUM:  // sum across TP, average across DP
          u.g_start = 0; u.g_stride = 1; u.g_count = world;
          u.scale = 1.0f / static_cast<float>(p->dp);
          break;
        case GRS_LOCAL_SHARD:  // the DP group of tp index t only
          u.g_start = t; u.g_stride = tp; u.g_count = p->dp;
          u.scale = 1.0f / static_cast<float>(p->dp);
          break;
        default:  // ALREADY_REDUCED: canonical rank 0, no reduction
          u.g_start = 0; u.g_stride = 1; u.g_count = 1;
          u.scale = 1.0f;
          break;
      }
      red_tiles += (bk.padded + T - 1) / T;
      upd_tiles += (bk.padded + UPD_T - 1) / UPD_T;
      p->units.push_back(u);
      p->red_prefix.push_back(red_tiles);
      p->upd_prefix.push_back(upd_tiles);
    }
    rank_off += bk.padded;
    state_off += static_cast<int64_t>(bk.copies) * bk.padded;
  }
  p->n_rank_pad = rank_off;
  p->n_state_pad = state_off;
  p->n_red_tiles = red_tiles;
  p->n_upd_tiles = upd_tiles;
  p->workspace_bytes = ws_bytes(red_tiles);

  // Gather jobs: one per (tensor, state row).
  p->jobs.clear();
  p->chunk_job.clear();
  p->tensor_job0.assign(1, 0);
  int64_t chunks = 0;
  int64_t logical = 0;  // canonical order: live tensors in model order, full logical extent
  for (int32_t i = 0; i < n; ++i) {
    if (p->t_bucket[i] < 0) {  // frozen: nothing to gather
      p->tensor_job0.push_back(static_cast<int32_t>(p->jobs.size()));
      continue;
    }
    const Bucket& bk = p->buckets[p->t_bucket[i]];
    const int64_t per_rank = (owners[i] == GRS_LOCAL_SHARD) ? numels[i] / tp : numels[i];
    for (int32_t t = 0; t < bk.copies; ++t) {
      GatherJob j{};
      j.src = bk.state_off + static_cast<int64_t>(t) * bk.padded + p->t_offset[i];
      j.dst = static_cast<int64_t>(t) * per_rank;
      j.len = per_rank;
      j.chunk0 = chunks;
      j.logical = logical + static_cast<int64_t>(t) * per_rank;
      j.tensor = i;
      const int64_t nc = (per_rank + GATHER_CHUNK - 1) / GATHER_CHUNK;
      chunks += nc;
      p->chunk_job.insert(p->chunk_job.end(), static_cast<size_t>(nc), static_cast<int32_t>(p->jobs.size()));
      p->jobs.push_back(j);
    }
    logical += numels[i];
    p->tensor_job0.push_back(static_cast<int32_t>(p->jobs.size()));
  }
  p->n_gather_chunks = chunks;

  // Segments per bucket, in offset order (tensors were appended in model
  // order with increasing offsets inside each bucket).
  std::vector<std::vector<int32_t>> members(p->buckets.size());
  for (int32_t i = 0; i < n; ++i)
    if (p->t_bucket[i] >= 0) members[p->t_bucket[i]].push_back(i);
  p->seg_start.clear();
  p->seg_tensor.clear();
  p->bucket_seg0.assign(1, 0);
  for (size_t b = 0; b < members.size(); ++b) {
    for (int32_t i : members[b]) {
      p->seg_start.push_back(p->t_offset[i]);
      p->seg_tensor.push_back(i);
    }
    p->bucket_seg0.push_back(static_cast<int32_t>(p->seg_start.size()));
  }
  // The tensor that holds each reduction and update tile entirely (-1 when
  // a tile spans several tensors or reaches the padding), unit by unit.
  p->red_tile_tensor.clear();
  p->upd_tile_tensor.clear();
  p->red_tile_unit.clear();
  p->upd_tile_unit.clear();
  for (size_t ui = 0; ui < p->units.size(); ++ui) {
    const UnitDesc& u = p->units[ui];
    sole_tensors(*p, u.bucket, u.red_T, p->red_tile_tensor);
    sole_tensors(*p, u.bucket, UPD_T, p->upd_tile_tensor);
    p->red_tile_unit.insert(p->red_tile_unit.end(), static_cast<size_t>(p->red_prefix[ui + 1] - p->red_prefix[ui]),
                            static_cast<int32_t>(ui));
    p->upd_tile_unit.insert(p->upd_tile_unit.end(), static_cast<size_t>(p->upd_prefix[ui + 1] - p->upd_prefix[ui]),
                            static_cast<int32_t>(ui));
  }
  // The non-empty gather jobs in state order (they never overlap: each
  // covers one tensor's part of one bucket row, so their starts differ) and,
  // per update tile, the first of them that ends after the tile's first
  // element: the update kernel that writes the bf16 parameters straight into
  // per-tensor storage finds the destination of its elements from there.
  // (An empty job would share its start with the next tensor's.)
  p->state_jobs.clear();
  for (const GatherJob& j : p->jobs)
    if (j.len > 0) p->state_jobs.push_back(j);
  std::sort(p->state_jobs.begin(), p->state_jobs.end(),
            [](const GatherJob& a, const GatherJob& b) { return a.src < b.src; });
  // Per tile also its unit, the tensor holding the whole tile and the
  // offset of its first element inside that tensor (UpdTileInfo), so that
  // the kernel finds the destination from one per-tile load and the
  // caller's pointer table.
  p->upd_tile_job.clear();
  p->upd_tile_info.clear();
  {
    size_t j = 0;
    for (size_t ui = 0; ui < p->units.size(); ++ui) {
      const UnitDesc& u = p->units[ui];
      for (int64_t t = p->upd_prefix[ui]; t < p->upd_prefix[ui + 1]; ++t) {
        const int64_t first = u.state_off + (t - p->upd_prefix[ui]) * UPD_T;
        while (j < p->state_jobs.size() && p->state_jobs[j].src + p->state_jobs[j].len <= first) ++j;
        p->upd_tile_job.push_back(static_cast<int32_t>(j));
        const int64_t e0 = (t - p->upd_prefix[ui]) * UPD_T;
        const int64_t len = std::min<int64_t>(UPD_T, u.padded - e0);  // the unit's last tile may be short
        UpdTileInfo info{static_cast<int32_t>(ui), -1, -1};
        if (p->upd_tile_tensor[t] >= 0 && j < p->state_jobs.size()) {
          const GatherJob& jb = p->state_jobs[j];
          if (jb.tensor == p->upd_tile_tensor[t] && jb.src <= first && first + len <= jb.src + jb.len) {
            info.tensor = jb.tensor;
            info.dst = jb.dst + (first - jb.src);
          }
        }
        p->upd_tile_info.push_back(info);
      }
    }
    p->upd_tile_job.push_back(static_cast<int32_t>(p->state_jobs.size()));  // sentinel
  }
  p->workspace_bytes = ws_factors_offset(red_tiles) + (static_cast<int64_t>(n) * 8 + 255) / 256 * 256;
  return GRS_OK;
}

// The state layout of rank (r, shard, tp_index) after the reduce-scatter:
// per bucket one slice of shard_len elements, [shard * shard_len, +shard_len)
// of row tp_index (LOCAL_SHARD) or row 0 (every other tag), slices back to
// back in bucket order.  One unit per bucket; the update tiles cover every
// slice, the norm tiles only the slices this rank holds uniquely within its
// tp group (LOCAL_SHARD rows always, the others only at tp index 0), so the
// views of one replica partition the plan's unique elements.
void build_shard_view(const grs_plan& parent, int32_t shard, int32_t tp_index, grs_plan* v) {
  v->numel = parent.numel;
  v->owner = parent.owner;
  v->tensor_flags = parent.tensor_flags;
  v->tensor_live = parent.tensor_live;
  v->world = parent.world;
  v->tp = parent.tp;
  v->dp_replicate = parent.dp_replicate;
  v->dp_shard = parent.dp_shard;
  v->dp = parent.dp;
  v->grad_esize = parent.grad_esize;
  v->bucket_bytes = parent.bucket_bytes;
  v->t_bucket = parent.t_bucket;
  v->t_offset = parent.t_offset;
  v->view_shard = shard;
  v->view_tp = tp_index;
  v->buckets.clear();
  v->units.clear();
  v->red_prefix.assign(1, 0);
  v->upd_prefix.assign(1, 0);
  v->red_tile_unit.clear();
  v->upd_tile_unit.clear();
  v->bucket_seg0.assign(1, 0);
  int64_t state_off = 0, red_tiles = 0, upd_tiles = 0, unique = 0;
  for (size_t b = 0; b < parent.buckets.size(); ++b) {
    const Bucket& pb = parent.buckets[b];
    const UnitDesc& pu = parent.units[pb.unit0];
    const int64_t L = pb.shard_len;
    const int64_t used = std::max<int64_t>(0, std::min<int64_t>(L, pb.used - int64_t(shard) * L));
    Bucket bk = pb;
    bk.copies = 1;
    bk.used = used;
    bk.padded = L;
    bk.shard_len = L;
    bk.rank_off = 0;
    bk.state_off = state_off;
    bk.unit0 = static_cast<int32_t>(v->units.size());
    v->buckets.push_back(bk);
    v->bucket_seg0.push_back(0);
    UnitDesc u{};
    u.state_off = state_off;
    u.padded = L;
    u.used = used;
    u.red_tile0 = red_tiles;
    u.upd_tile0 = upd_tiles;
    u.red_T = pu.red_T;
    u.bucket = static_cast<int32_t>(b);
    const bool counts = pb.tag == GRS_LOCAL_SHARD || tp_index == 0;
    const int64_t nr = counts ? (L + pu.red_T - 1) / pu.red_T : 0;
    const int64_t nu = (L + UPD_T - 1) / UPD_T;
    v->red_tile_unit.insert(v->red_tile_unit.end(), static_cast<size_t>(nr), static_cast<int32_t>(v->units.size()));
    v->upd_tile_unit.insert(v->upd_tile_unit.end(), static_cast<size_t>(nu), static_cast<int32_t>(v->units.size()));
    red_tiles += nr;
    upd_tiles += nu;
    if (counts) unique += used;
    v->units.push_back(u);
    v->red_prefix.push_back(red_tiles);
    v->upd_prefix.push_back(upd_tiles);
    state_off += L;
  }
  v->n_unique = unique;
  v->n_rank_pad = 0;
  v->n_state_pad = state_off;
  v->n_red_tiles = red_tiles;
  v->n_upd_tiles = upd_tiles;
  v->n_gather_chunks = 0;
  v->workspace_bytes = ws_bytes(red_tiles);
}

}  // namespace grs
