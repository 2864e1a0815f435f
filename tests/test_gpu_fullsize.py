"""Full-size parity: the four large workloads, one update from the seeded
state, in exactly the launch configuration bench.py times (bench.GpuUpdate:
grs_reduce_all per microbatch with the fused norm epilogue, grs_grad_norm_sq,
grs_clip_adamw_step).

The oracle computes the exact global norm over every element (each bucket's
inputs streamed to the host through pinned buffers, one thread per core) and
the clipped AdamW update at sampled elements of every bucket row: random
interior points, the first and last valid elements, tile edges and padding.
"""
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_support import assert_bf16_cast, assert_close, assert_close_bracketed

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


def _free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 1e9


def sample_positions(rng, used, P, tile=2048, n_random=384):
    """Element indices of one bucket row: random interior points, both ends
    of the valid range, elements around tile boundaries, padding."""
    pos = set()
    if used > 0:
        pos.update(rng.integers(0, used, min(n_random, used)).tolist())
        pos.update(range(0, min(8, used)))
        pos.update(range(max(0, used - 8), used))
        for b in range(tile, used, max(tile, (used // 16) // tile * tile or tile)):
            pos.update(range(b - 2, min(b + 2, used)))
    pos.update(range(used, min(P, used + 8)))  # padding
    return np.array(sorted(p for p in pos if 0 <= p < P), np.int64)


@pytest.mark.parametrize("cid", [1, 4, 3, 2])
def test_full_size_update_matches_oracle(cid):
    import bench  # the benchmark's own update object

    w = workloads.get(cid)
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    need = (w.n_micro * w.world * op.n_rank_pad * 2 + op.n_state_pad * 18) / 1e9
    if _free_gb() < need * 1.05 + 4:
        pytest.skip(f"needs {need:.0f} GB of device memory")
    dev = torch.device("cuda")
    rng = np.random.default_rng(1000 + cid)
    u = bench.GpuUpdate(w, dev)
    try:
        M, R = w.n_micro, w.world
        # samples and their initial state, before the update overwrites it
        samples = {}
        for b in range(op.n_buckets):
            P, used = int(op.b_padded[b]), int(op.b_used[b])
            samples[b] = sample_positions(rng, used, P)
        state_idx = np.concatenate([int(op.b_state_off[b]) + t * int(op.b_padded[b]) + samples[b]
                                    for b in range(op.n_buckets) for t in range(op.copies(b))])
        sidx = torch.from_numpy(state_idx).to(dev)
        master0 = u.master[sidx].cpu().numpy()

        u.step()
        torch.cuda.synchronize()
        assert u.grs.grs_check_device_errors(u.plan, u.stream) == 0

        # ---- exact global norm: every element through the oracle, bucket by
        # bucket in chunks of at most CHUNK elements (bounded host memory)
        CHUNK = 1 << 21
        items = [(b, cs, min(CHUNK, int(op.b_padded[b]) - cs))
                 for b in range(op.n_buckets) for cs in range(0, int(op.b_padded[b]), CHUNK)]
        pinned = threading.local()

        def host_buf():
            if not hasattr(pinned, "buf"):
                pinned.buf = torch.empty(M * R * CHUNK, dtype=torch.int16).pin_memory()
            return pinned.buf

        def chunk_norm(item):
            b, cs, cl = item
            ro = int(op.b_rank_off[b]) + cs
            hb = host_buf()[:M * R * cl].view(M, R, cl)
            for j in range(M):
                for k in range(R):
                    hb[j, k].copy_(u.grads[j][k][ro:ro + cl].view(torch.int16))
            g = hb.numpy().view(np.uint16)
            used = max(0, min(cl, int(op.b_used[b]) - cs))
            acc = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, cl,
                                       used, g)
            return oracle.norm_sq(acc, M)

        threads = max(1, min(8, os.cpu_count() or 1))
        with ThreadPoolExecutor(threads) as ex:
            parts = list(ex.map(chunk_norm, items))
        s_oracle = float(np.sum(np.array(parts, np.float64)))  # (bucket, chunk) order
        s_gpu = float(u.norm.cpu()[0])
        assert_close([s_gpu], [s_oracle], f"workload {cid} norm_sq")
        c = oracle.clip_coef(s_oracle, w.adamw.max_norm)
        assert c < 1.0  # clipping is active on these workloads

        # ---- sampled accumulator and update
        a = w.adamw
        hp = (a.lr, a.beta1, a.beta2, a.eps, a.weight_decay)
        want_acc, want_p, want_m, want_v, want_bits = [], [], [], [], []
        lo_p, lo_m, lo_v, hi_p, hi_m, hi_v = [], [], [], [], [], []
        for b in range(op.n_buckets):
            pos = samples[b]
            ro, used = int(op.b_rank_off[b]), int(op.b_used[b])
            pt = torch.from_numpy(pos + ro).to(dev)
            g = np.stack([np.stack([u.grads[j][k].view(torch.int16)[pt].cpu().numpy().view(np.uint16)
                                    for k in range(R)]) for j in range(M)])
            n_valid = int((pos < used).sum())
            acc = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard,
                                       len(pos), n_valid, g)
            delta = oracle.accumulation_error_bound(
                oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, len(pos),
                                     n_valid, oracle.abs_inputs(g)), M)
            for t in range(op.copies(b)):
                want_acc.append(acc[t])
                off = sum(len(samples[bb]) * op.copies(bb) for bb in range(b)) + t * len(pos)
                m0 = master0[off:off + len(pos)]
                z = np.zeros(len(pos), np.float32)
                p1, m1, v1, bits = oracle.adamw(acc[t], n_valid, M, c, hp, 1, m0, z, z)
                want_p.append(p1)
                want_m.append(m1)
                want_v.append(v1)
                want_bits.append(bits)
                for sign, dst in ((-1.0, (lo_p, lo_m, lo_v)), (1.0, (hi_p, hi_m, hi_v))):
                    r = oracle.adamw(acc[t] + sign * delta[t], n_valid, M, c, hp, 1, m0, z, z)
                    for d_, x in zip(dst, r[:3]):
                        d_.append(x)
        got_acc = u.acc[sidx].cpu().numpy()
        got_p = u.master[sidx].cpu().numpy()
        got_m = u.m[sidx].cpu().numpy()
        got_v = u.v[sidx].cpu().numpy()
        got_bits = u.params[sidx].cpu().numpy().view(np.uint16)
        assert_close(got_acc, np.concatenate(want_acc), f"workload {cid} acc")
        cat = np.concatenate
        assert_close_bracketed(got_p, cat(want_p), cat(lo_p), cat(hi_p), f"workload {cid} master")
        assert_close_bracketed(got_m, cat(want_m), cat(lo_m), cat(hi_m), f"workload {cid} m")
        assert_close_bracketed(got_v, cat(want_v), cat(lo_v), cat(hi_v), f"workload {cid} v")
        assert_bf16_cast(got_bits, got_p, np.concatenate(want_bits), np.concatenate(want_p),
                         f"workload {cid} params")
        pad = np.concatenate([np.repeat((samples[b] >= int(op.b_used[b]))[None], op.copies(b), 0).reshape(-1)
                              for b in range(op.n_buckets)])
        for arr in (got_acc, got_p, got_m, got_v, got_bits):
            assert np.all(arr[pad] == 0)
    finally:
        u.close()
        del u
        torch.cuda.empty_cache()
