"""Full-size parity: the four large workloads, one update from the seeded
state, in exactly the launch configuration bench.py times (bench.GpuUpdate:
grs_reduce_all per microbatch with the fused norm epilogue, grs_grad_norm_sq,
grs_clip_adamw_step).

Every element of each workload's update is compared with the oracle (the
67M plan in one piece, the larger ones bucket row by bucket row in chunks on
the host's cores), and so is every element of the measured variants (fp32
gradients, tensors without a gradient, frozen tensors, a trailing window).
The one tensor past 32-bit indices is checked at sampled elements: random
interior points, the first and last valid elements, tile edges and padding.
The host-buffer call the bench's end-to-end figure times is checked against
the device-resident path on the 3.2B plan, bit for bit.
"""
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_support import (assert_bf16_cast, assert_close, assert_close_bracketed,
                         assert_within_accumulation_bound)

RA = workloads.REPLICA_AVG

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


@pytest.fixture(autouse=True)
def _release_memory():
    """Each test here holds tens to hundreds of GB: hand the cached blocks
    back after it, so the next one sees the device's free memory."""
    yield
    import gc
    gc.collect()
    torch.cuda.empty_cache()


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


# The variants bench.py measures (--variant / --window), in the same launch
# configuration, every element: fp32 rank gradients, tensors without a
# gradient (masked reduction with its fused norm partials, masked update),
# frozen tensors, a trailing window of 3 of 4 microbatches.
@pytest.mark.parametrize("cid,variant,window", [(1, "fp32-grads", 0), (1, "unused", 0),
                                                (1, "frozen", 0), (3, "plain", 3)])
def test_full_size_variant_matches_oracle(cid, variant, window):
    _every_element(workloads.get(cid), variant, window)


def test_workload1_every_element_matches_oracle():
    """The 67M-parameter, world-16 workload (the benchmark's smallest large
    plan) with no sampling: one update in the bench's launch configuration,
    then every element of the accumulator, master, moments and bf16
    parameters against the oracle's whole update (all six buckets), the
    accumulator within the fp32 accumulation bound, padding exactly zero."""
    import bench
    from gpu_support import assert_bf16_cast as cast_check, padding_mask

    w = workloads.get(1)
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    u = bench.GpuUpdate(w, torch.device("cuda"))
    try:
        n = op.n_state_pad
        assert u.info["n_state_pad"] == n
        master0 = u.master[:n].cpu().numpy().copy()
        z = np.zeros(n, np.float32)
        u.step()
        torch.cuda.synchronize()
        assert u.grs.grs_check_device_errors(u.plan, u.stream) == 0
        M, R = w.n_micro, w.world

        def grads_of(b):
            ro, P = int(op.b_rank_off[b]), int(op.b_padded[b])
            return np.stack([np.stack([u.grads[j][k][ro:ro + P].view(torch.int16).cpu().numpy()
                                       for k in range(R)]) for j in range(M)]).view(np.uint16)

        a = w.adamw
        hp = (a.lr, a.beta1, a.beta2, a.eps, a.weight_decay)
        res = oracle.full_update(op, grads_of, M, hp, a.max_norm, 1, master0, z, z,
                                 threads=max(1, min(8, os.cpu_count() or 1)), bounds=True)
        what = "workload 1, every element"
        acc = u.acc[:n].cpu().numpy()
        assert_close(acc, res.acc, f"{what} acc")
        assert_within_accumulation_bound(acc, res.acc, res.delta, f"{what} acc")
        assert_close([float(u.norm.cpu()[0])], [res.norm_sq], f"{what} norm_sq")
        master = u.master[:n].cpu().numpy()
        mm = u.m[:n].cpu().numpy()
        vv = u.v[:n].cpu().numpy()
        for name, got, want, lo, hi in zip(("master", "m", "v"), (master, mm, vv), (res.master, res.m, res.v),
                                           res.lo, res.hi):
            assert_close_bracketed(got, want, lo, hi, f"{what} {name}")
        bits = u.params[:n].cpu().numpy().view(np.uint16)
        cast_check(bits, master, res.params_bf16, res.master, f"{what} params", lo_master=res.lo[0],
                   hi_master=res.hi[0])
        pad = padding_mask(op)  # (this plan's buckets need no padding: every size is a multiple of 64)
        for arr in (acc, master, mm, vv, bits):
            assert np.all(arr[pad] == 0)
    finally:
        u.close()
        del u
        torch.cuda.empty_cache()


@pytest.mark.parametrize("cid", [4, 3, 2])
def test_large_workload_every_element_matches_oracle(cid):
    """The 3.2B, MoE and 1.1B workloads with no sampling: one update in the
    bench's launch configuration, then every accumulator, master, moment and
    bf16 element against the oracle, bucket row by bucket row in chunks of
    at most 8M elements on the host's cores (the clip coefficient from the
    oracle's exact norm over every element, which must match the GPU's)."""
    _every_element(workloads.get(cid))


def _every_element(w, variant="plain", window=0, chunk=1 << 23):
    """One update of workload `w` (bench.GpuUpdate with the variant's plan
    flags, gradient type, window and mask), then every state element
    against the oracle, bucket row by bucket row in chunks on the host's
    cores.  Elements of tensors without a gradient this step (the unused
    variant) count zero in the norm and must keep master, bf16 copy and zero
    moments; their accumulator is unspecified."""
    import bench
    from gpu_support import assert_bf16_cast as cast_check

    fp32 = variant == "fp32-grads"
    flags = bench.frozen_pattern(len(w.numels)) if variant == "frozen" else None
    used_t = bench.unused_pattern(len(w.numels)) if variant == "unused" else None
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes, flags)
    M = window or w.n_micro
    need = (M * w.world * op.n_rank_pad * (4 if fp32 else 2) + op.n_state_pad * 24) / 1e9
    if _free_gb() < need * 1.05 + 4:
        pytest.skip(f"needs {need:.0f} GB of device memory")
    u = bench.GpuUpdate(w, torch.device("cuda"), variant, window)
    gview = torch.float32 if fp32 else torch.int16
    # per bucket: the per-rank elements that belong to a tensor with a gradient
    live = {}
    for b in range(op.n_buckets):
        mk = np.zeros(int(op.b_padded[b]), bool)
        for i in range(len(w.numels)):
            if int(op.t_bucket[i]) == b and (used_t is None or used_t[i]):
                o = int(op.t_offset[i])
                mk[o:o + op.per_rank(i)] = True
        live[b] = mk
    try:
        assert u.info["n_state_pad"] == op.n_state_pad and u.n_micro == M
        master0 = u.master.clone()
        params0 = u.params.clone()
        u.step()
        torch.cuda.synchronize()
        assert u.grs.grs_check_device_errors(u.plan, u.stream) == 0
        R = w.world
        a = w.adamw
        hp = (a.lr, a.beta1, a.beta2, a.eps, a.weight_decay)
        items = [(b, cs, min(chunk, int(op.b_padded[b]) - cs))
                 for b in range(op.n_buckets) for cs in range(0, int(op.b_padded[b]), chunk)]

        def reduce(item):
            b, cs, cl = item
            ro = int(op.b_rank_off[b]) + cs
            g = np.stack([np.stack([u.grads[j][k][ro:ro + cl].view(gview).cpu().numpy() for k in range(R)])
                          for j in range(M)])
            if not fp32:
                g = g.view(np.uint16)
            used = max(0, min(cl, int(op.b_used[b]) - cs))
            acc = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, cl, used, g)
            return g, used, acc

        def norm_part(item):
            acc = reduce(item)[2].copy()
            acc[:, ~live[item[0]][item[1]:item[1] + item[2]]] = 0.0  # no gradient: counts zero
            return oracle.norm_sq(acc, M)

        threads = max(1, min(16, os.cpu_count() or 1))
        with ThreadPoolExecutor(threads) as ex:
            parts = list(ex.map(norm_part, items))
        s_oracle = float(np.sum(np.array(parts, np.float64)))
        what0 = f"{w.name} {variant}" + (f" window {M}" if window else "")
        assert_close([float(u.norm.cpu()[0])], [s_oracle], f"{what0} norm_sq")
        c = oracle.clip_coef(s_oracle, a.max_norm)
        assert c < 1.0  # clipping is active on these workloads

        def compare(item):
            b, cs, cl = item
            g, used, acc = reduce(item)
            delta = oracle.accumulation_error_bound(
                oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, cl, used,
                                     oracle.abs_inputs(g)), M, oracle.group_terms(op, b))
            lv = live[b][cs:cs + cl]
            idle = ~lv.copy()
            idle[used:] = False  # padding is checked as padding
            for t in range(op.copies(b)):
                o = int(op.b_state_off[b]) + t * int(op.b_padded[b]) + cs
                sl = slice(o, o + cl)
                m0 = master0[sl].cpu().numpy()
                z = np.zeros(cl, np.float32)
                want = oracle.adamw(acc[t], used, M, c, hp, 1, m0, z, z)
                lo = oracle.adamw(acc[t] - delta[t], used, M, c, hp, 1, m0, z, z)
                hi = oracle.adamw(acc[t] + delta[t], used, M, c, hp, 1, m0, z, z)
                what = f"{what0} bucket {b} row {t} [{cs}, {cs + cl})"
                got_acc = u.acc[sl].cpu().numpy()
                got = [x[sl].cpu().numpy() for x in (u.master, u.m, u.v)]
                bits = u.params[sl].cpu().numpy().view(np.uint16)
                k = lv  # elements of tensors with a gradient (the masked update leaves the others)
                assert_close(got_acc[k], acc[t][k], f"{what} acc")
                assert_within_accumulation_bound(got_acc[k], acc[t][k], delta[t][k], f"{what} acc")
                for name, gv, wv, lw, hw in zip(("master", "m", "v"), got, want[:3], lo[:3], hi[:3]):
                    assert_close_bracketed(gv[k], wv[k], lw[k], hw[k], f"{what} {name}")
                cast_check(bits[k], got[0][k], want[3][k], want[0][k], f"{what} params", lo_master=lo[0][k],
                           hi_master=hi[0][k])
                if idle.any():  # no gradient this step: nothing read or written
                    assert np.array_equal(got[0][idle].view(np.uint32), m0[idle].view(np.uint32)), what
                    b0 = params0[sl].cpu().numpy().view(np.uint16)
                    assert np.array_equal(bits[idle], b0[idle]), what
                    assert np.all(got[1][idle] == 0) and np.all(got[2][idle] == 0), what
                for x in (got_acc, got[0], got[1], got[2], bits):
                    assert np.all(x[used:] == 0)
            return cl * op.copies(b), int(idle.sum()) * op.copies(b)

        with ThreadPoolExecutor(threads) as ex:
            done = list(ex.map(compare, items))
        assert sum(n for n, _ in done) == op.n_state_pad
        if used_t is not None:
            assert sum(i for _, i in done) > 0, "no element of a tensor without a gradient"
    finally:
        u.close()
        del u
        torch.cuda.empty_cache()


def test_single_tensor_beyond_32_bit_indices():
    """One REPLICA_AVG tensor of 2^31 + 4099 elements (world 1): every index
    of the reduction, norm, update and padding lies past the 32-bit range at
    the end of the tensor, where the samples include the last elements and
    the padding."""
    w = workloads.Workload(90, "single-2^31+4099", [workloads.Tensor("w", (2 ** 31 + 4099,), RA)],
                           tp=1, dp_replicate=1, dp_shard=1, n_micro=1, grad_std=1e-3)
    _full_size_w(w, "plain", 0)


def test_gather_and_layout_beyond_32_bit_indices():
    """The same 2^31 + 4099-element tensor through the gather to per-tensor
    storage, the state <-> logical conversions and the update that writes
    the tensor itself: for one tensor on one rank each is the identity on
    its elements, and the padding comes back as zeros."""
    from gradient_reduction_sharded_gb300 import grs
    n = 2 ** 31 + 4099
    if _free_gb() < 3 * n * 2 / 1e9 + 4 * n * 4 / 1e9 + 8:
        pytest.skip("needs about 56 GB of device memory")
    plan = grs.grs_plan_create([n], [RA], 1, 1, 1, 1, 25 << 20)
    try:
        info = grs.grs_plan_query(plan)
        nsp = info["n_state_pad"]
        assert nsp == (n + 7) // 8 * 8
        s = torch.cuda.current_stream().cuda_stream
        gen = torch.Generator(device="cuda").manual_seed(5)
        params = torch.randint(-32768, 32767, (nsp,), dtype=torch.int16, device="cuda", generator=gen)
        out = torch.empty(n, dtype=torch.int16, device="cuda")
        grs.grs_gather_params(plan, params.data_ptr(), [out.data_ptr()], s)
        torch.cuda.synchronize()
        assert torch.equal(out, params[:n])
        del out, params
        state = torch.randn(nsp, device="cuda", generator=gen)
        logical = torch.empty(n, device="cuda")
        grs.grs_state_to_logical(plan, state.data_ptr(), logical.data_ptr(), s)
        back = torch.full((nsp,), float("nan"), device="cuda")
        grs.grs_state_from_logical(plan, logical.data_ptr(), back.data_ptr(), s)
        torch.cuda.synchronize()
        assert grs.grs_check_device_errors(plan, s) == 0
        assert torch.equal(logical, state[:n])
        assert torch.equal(back[:n], state[:n]) and bool((back[n:] == 0).all())
        del logical, back
        # the update writing the tensor itself: every offset past 2^31 comes
        # from the per-tile records; the result equals the bucket-ordered
        # buffer the same update writes (the tensor is the buffer's first n)
        acc = state
        master = torch.randn(nsp, device="cuda", generator=gen)
        m = torch.zeros(nsp, device="cuda")
        v = torch.zeros(nsp, device="cuda")
        ref_params = torch.empty(nsp, dtype=torch.int16, device="cuda")
        out = torch.full((n,), -1, dtype=torch.int16, device="cuda")
        table = torch.tensor([out.data_ptr()], dtype=torch.int64, device="cuda")
        hp = grs.make_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 1, 1)
        grs.grs_clip_adamw_step_to_tensors(plan, hp, None, acc.data_ptr(), master.data_ptr(), m.data_ptr(),
                                           v.data_ptr(), ref_params.data_ptr(), table.data_ptr(), s)
        torch.cuda.synchronize()
        assert grs.grs_check_device_errors(plan, s) == 0
        assert torch.equal(out, ref_params[:n])
        assert bool((ref_params[n:] == 0).all())
    finally:
        grs.grs_plan_destroy(plan)
        torch.cuda.empty_cache()


def _full_size_w(w, variant, window):
    import bench  # the benchmark's own update object

    cid = w.name
    M = window or w.n_micro
    fp32 = variant == "fp32-grads"
    flags = bench.frozen_pattern(len(w.numels)) if variant == "frozen" else None
    used_t = bench.unused_pattern(len(w.numels)) if variant == "unused" else None
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes,
                     flags)
    need = (M * w.world * op.n_rank_pad * (4 if fp32 else 2) + op.n_state_pad * 18) / 1e9
    if _free_gb() < need * 1.05 + 4:
        pytest.skip(f"needs {need:.0f} GB of device memory")
    dev = torch.device("cuda")
    rng = np.random.default_rng(1000 + w.cid)
    u = bench.GpuUpdate(w, dev, variant, window)
    assert u.info["n_state_pad"] == op.n_state_pad and u.n_micro == M
    gview = torch.float32 if fp32 else torch.int16
    hdt = np.float32 if fp32 else np.uint16

    def host(t):
        x = t.view(gview).cpu().numpy()
        return x if fp32 else x.view(np.uint16)

    # per bucket: which per-rank elements belong to a tensor with a gradient
    counts = {}
    for b in range(op.n_buckets):
        mk = np.zeros(int(op.b_padded[b]), bool)
        for i in range(len(w.numels)):
            if int(op.t_bucket[i]) == b and (used_t is None or used_t[i]):
                o = int(op.t_offset[i])
                mk[o:o + op.per_rank(i)] = True
        counts[b] = mk
    try:
        R = w.world
        # samples and their initial state, before the update overwrites it
        samples = {}
        for b in range(op.n_buckets):
            P, used = int(op.b_padded[b]), int(op.b_used[b])
            samples[b] = sample_positions(rng, used, P)
        state_idx = np.concatenate([int(op.b_state_off[b]) + t * int(op.b_padded[b]) + samples[b]
                                    for b in range(op.n_buckets) for t in range(op.copies(b))])
        sidx = torch.from_numpy(state_idx).to(dev)
        master0 = u.master[sidx].cpu().numpy()
        bits0 = u.params[sidx].cpu().numpy().view(np.uint16)

        u.step()
        torch.cuda.synchronize()
        assert u.grs.grs_check_device_errors(u.plan, u.stream) == 0

        # ---- exact global norm: every element through the oracle, bucket by
        # bucket in chunks of at most CHUNK elements (bounded host memory);
        # elements of tensors without a gradient count zero
        CHUNK = 1 << 21
        items = [(b, cs, min(CHUNK, int(op.b_padded[b]) - cs))
                 for b in range(op.n_buckets) for cs in range(0, int(op.b_padded[b]), CHUNK)]
        pinned = threading.local()

        def host_buf():
            if not hasattr(pinned, "buf"):
                pinned.buf = torch.empty(M * R * CHUNK, dtype=gview).pin_memory()
            return pinned.buf

        def chunk_norm(item):
            b, cs, cl = item
            ro = int(op.b_rank_off[b]) + cs
            hb = host_buf()[:M * R * cl].view(M, R, cl)
            for j in range(M):
                for k in range(R):
                    hb[j, k].copy_(u.grads[j][k][ro:ro + cl].view(gview))
            g = hb.numpy() if fp32 else hb.numpy().view(np.uint16)
            used = max(0, min(cl, int(op.b_used[b]) - cs))
            acc = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, cl,
                                       used, g)
            acc[:, ~counts[b][cs:cs + cl]] = 0.0
            return oracle.norm_sq(acc, M)

        threads = max(1, min(8, os.cpu_count() or 1))
        with ThreadPoolExecutor(threads) as ex:
            parts = list(ex.map(chunk_norm, items))
        s_oracle = float(np.sum(np.array(parts, np.float64)))  # (bucket, chunk) order
        s_gpu = float(u.norm.cpu()[0])
        what = f"workload {cid} {variant}" + (f" window {M}" if window else "")
        assert_close([s_gpu], [s_oracle], f"{what} norm_sq")
        c = oracle.clip_coef(s_oracle, w.adamw.max_norm)
        assert c < 1.0  # clipping is active on these workloads

        # ---- sampled accumulator and update
        a = w.adamw
        hp = (a.lr, a.beta1, a.beta2, a.eps, a.weight_decay)
        want_acc, want_delta, want_p, want_m, want_v, want_bits = [], [], [], [], [], []
        lo_p, lo_m, lo_v, hi_p, hi_m, hi_v = [], [], [], [], [], []
        idle = []  # sampled state positions of tensors without a gradient
        for b in range(op.n_buckets):
            pos = samples[b]
            ro, used = int(op.b_rank_off[b]), int(op.b_used[b])
            pt = torch.from_numpy(pos + ro).to(dev)
            g = np.stack([np.stack([host(u.grads[j][k].view(gview)[pt]) for k in range(R)])
                          for j in range(M)]).astype(hdt)
            n_valid = int((pos < used).sum())
            acc = oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard,
                                       len(pos), n_valid, g)
            delta = oracle.accumulation_error_bound(
                oracle.reduce_bucket(int(op.b_tag[b]), op.tp, op.dp_replicate, op.dp_shard, len(pos),
                                     n_valid, oracle.abs_inputs(g)), M, oracle.group_terms(op, b))
            off_idle = (pos < used) & ~counts[b][pos]
            for t in range(op.copies(b)):
                want_acc.append(acc[t])
                want_delta.append(delta[t])
                off = sum(len(samples[bb]) * op.copies(bb) for bb in range(b)) + t * len(pos)
                m0 = master0[off:off + len(pos)]
                z = np.zeros(len(pos), np.float32)
                p1, m1, v1, bits = oracle.adamw(acc[t], n_valid, M, c, hp, 1, m0, z, z)
                rl = oracle.adamw(acc[t] - delta[t], n_valid, M, c, hp, 1, m0, z, z)
                rh = oracle.adamw(acc[t] + delta[t], n_valid, M, c, hp, 1, m0, z, z)
                # no gradient this step: master, moments and bf16 copy unchanged
                b0 = bits0[off:off + len(pos)]
                for arr, keep in ((p1, m0), (m1, z), (v1, z), (bits, b0), (rl[0], m0), (rl[1], z),
                                  (rl[2], z), (rh[0], m0), (rh[1], z), (rh[2], z)):
                    arr[off_idle] = keep[off_idle]
                idle.append(off_idle)
                want_p.append(p1)
                want_m.append(m1)
                want_v.append(v1)
                want_bits.append(bits)
                for d_, x in zip((lo_p, lo_m, lo_v), rl[:3]):
                    d_.append(x)
                for d_, x in zip((hi_p, hi_m, hi_v), rh[:3]):
                    d_.append(x)
        got_acc = u.acc[sidx].cpu().numpy()
        got_p = u.master[sidx].cpu().numpy()
        got_m = u.m[sidx].cpu().numpy()
        got_v = u.v[sidx].cpu().numpy()
        got_bits = u.params[sidx].cpu().numpy().view(np.uint16)
        cat = np.concatenate
        idle = cat(idle)
        # the masked reduction leaves the accumulator of tensors without a
        # gradient unspecified: only the others are compared
        assert_close(got_acc[~idle], cat(want_acc)[~idle], f"{what} acc")
        assert_within_accumulation_bound(got_acc[~idle], cat(want_acc)[~idle], cat(want_delta)[~idle],
                                         f"{what} acc")
        assert_close_bracketed(got_p, cat(want_p), cat(lo_p), cat(hi_p), f"{what} master")
        assert_close_bracketed(got_m, cat(want_m), cat(lo_m), cat(hi_m), f"{what} m")
        assert_close_bracketed(got_v, cat(want_v), cat(lo_v), cat(hi_v), f"{what} v")
        live = ~idle
        assert_bf16_cast(got_bits[live], got_p[live], cat(want_bits)[live], cat(want_p)[live],
                         f"{what} params", lo_master=cat(lo_p)[live], hi_master=cat(hi_p)[live])
        if used_t is not None:
            assert idle.any(), "the sample holds no element of a tensor without a gradient"
            # bit for bit: the masked update neither reads nor writes them
            assert np.array_equal(got_p[idle].view(np.uint32), master0[idle].view(np.uint32))
            assert np.array_equal(got_bits[idle], bits0[idle])
            assert np.all(got_m[idle] == 0) and np.all(got_v[idle] == 0)
        pad = np.concatenate([np.repeat((samples[b] >= int(op.b_used[b]))[None], op.copies(b), 0).reshape(-1)
                              for b in range(op.n_buckets)])
        for arr in (got_acc, got_p, got_m, got_v, got_bits):
            assert np.all(arr[pad] == 0)
    finally:
        u.close()
        del u
        torch.cuda.empty_cache()


def _host_available_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024 / 1e9
    except OSError:
        pass
    return 0.0


def test_step_from_host_full_size_equals_device_path():
    """grs_step_from_host on the 3.2B plan, as the bench's end-to-end leg
    calls it (pinned host gradients copied in bucket by bucket on the plan's
    copy stream, each bucket reduced when its copy lands; the bf16
    parameters and the norm read back to pinned host memory), two calls
    queued back to back (the second's copies overlap the first's update),
    against two steps of the device-resident path (bench.GpuUpdate: one
    grouped reduction, the finish, the update) on the same gradients and
    initial state: each call's host copies of the parameters and the norm
    equal that step's device values, and after the second call the
    accumulator, norm, master, m, v and bf16 parameters are equal bit for
    bit.  The device path itself is checked against the oracle element by
    element above."""
    import bench
    from gradient_reduction_sharded_gb300 import grs as g

    w = workloads.get(4)
    if _free_gb() < 190 or _host_available_gb() < 70:
        pytest.skip(f"needs ~170 GB of device and ~45 GB of host memory "
                    f"({_free_gb():.0f} GB, {_host_available_gb():.0f} GB available)")
    dev = torch.device("cuda")
    u = bench.GpuUpdate(w, dev)
    try:
        W, nrp, nsp = w.world, u.info["n_rank_pad"], u.info["n_state_pad"]
        # the host path's own state, from the same initial values
        acc = torch.empty(nsp, dtype=torch.float32, device=dev)
        master, m, v = u.master.clone(), u.m.clone(), u.v.clone()
        params = torch.empty(nsp, dtype=torch.int16, device=dev)
        ws = torch.zeros_like(u.ws)
        norm = torch.zeros(1, dtype=torch.float64, device=dev)
        host = [torch.empty(nrp, dtype=torch.int16, pin_memory=True) for _ in range(W)]
        for k in range(W):
            host[k].copy_(u.grads[0][k].view(torch.int16))
        stage = [torch.empty(nrp, dtype=torch.int16, device=dev) for _ in range(W)]
        stage_ptrs = [t.data_ptr() for t in stage] * 2  # one microbatch: one staging half
        out_params = [torch.empty(nsp, dtype=torch.int16, pin_memory=True) for _ in range(2)]
        out_norm = [torch.empty(1, dtype=torch.float64, pin_memory=True) for _ in range(2)]
        # the device path: step 1 (kept on the host), then step 2
        u.step()
        torch.cuda.synchronize()
        want1_params, want1_norm = u.params[:nsp].cpu(), float(u.norm.cpu()[0])
        u.step()
        torch.cuda.synchronize()
        # the host path: both calls queued without a synchronisation
        a = w.adamw
        for step in (1, 2):
            hp = g.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, step, 1)
            g.grs_step_from_host(u.plan, hp, [t.data_ptr() for t in host], stage_ptrs, acc.data_ptr(),
                                 master.data_ptr(), m.data_ptr(), v.data_ptr(), params.data_ptr(),
                                 ws.data_ptr(), norm.data_ptr(), out_params[step - 1].data_ptr(),
                                 out_norm[step - 1].data_ptr(), u.stream)
        torch.cuda.synchronize()
        assert g.grs_check_device_errors(u.plan, u.stream) == 0
        assert torch.equal(out_params[0], want1_params), "step 1 host params"
        assert float(out_norm[0][0]) == want1_norm, "step 1 host norm"
        for nm, got in (("acc", acc), ("norm", norm), ("master", master), ("m", m), ("v", v),
                        ("params", params)):
            assert torch.equal(got[:nsp], getattr(u, nm)[:nsp]), f"step 2 {nm}"
        assert torch.equal(out_params[1], u.params[:nsp].cpu()), "step 2 host params"
        assert float(out_norm[1][0]) == float(u.norm.cpu()[0]), "step 2 host norm"
    finally:
        u.close()


def test_update_to_tensors_full_size_matches_gather():
    """grs_clip_adamw_step_to_tensors on the 3.2B plan (254 tensors, 142
    buckets; the bench times it beside the plain update): from the same
    reduced gradient and state, master, m and v equal the plain update's
    bit for bit and every tensor written by the update equals
    oracle.gather_tensor of the plain update's bucket-ordered parameters,
    bit for bit; so does every tensor of the separate gather pass
    (grs_gather_params) from those parameters."""
    import bench
    from gradient_reduction_sharded_gb300 import grs as g

    w = workloads.get(4)
    if _free_gb() < 185 or _host_available_gb() < 30:
        pytest.skip(f"needs ~170 GB of device and ~15 GB of host memory "
                    f"({_free_gb():.0f} GB, {_host_available_gb():.0f} GB available)")
    dev = torch.device("cuda")
    op = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    u = bench.GpuUpdate(w, dev)
    try:
        nsp = u.info["n_state_pad"]
        assert nsp == op.n_state_pad
        u.reduce()
        u.norm_sq()
        saved = [u.master.clone(), u.m.clone(), u.v.clone()]
        u.adamw()  # the plain update, step 1
        torch.cuda.synchronize()
        plain = [u.master.clone(), u.m.clone(), u.v.clone()]
        params_ref = u.params[:nsp].cpu().numpy().view(np.uint16)
        # the separate gather pass from the same bucket-ordered parameters
        gathered = [torch.full((max(n, 1),), -1, dtype=torch.int16, device=dev) for n in w.numels]
        g.grs_gather_params(u.plan, u.params.data_ptr(), [t.data_ptr() for t in gathered], u.stream)
        for x, s0 in zip((u.master, u.m, u.v), saved):
            x.copy_(s0)
        del saved
        outs = [torch.full((max(n, 1),), -1, dtype=torch.int16, device=dev) for n in w.numels]
        table = torch.tensor([t.data_ptr() for t in outs], dtype=torch.int64, device=dev)
        a = w.adamw
        hp = g.make_adamw(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1, w.n_micro)
        g.grs_clip_adamw_step_to_tensors(u.plan, hp, u.norm.data_ptr(), u.acc.data_ptr(), u.master.data_ptr(),
                                         u.m.data_ptr(), u.v.data_ptr(), None, table.data_ptr(), u.stream)
        torch.cuda.synchronize()
        assert g.grs_check_device_errors(u.plan, u.stream) == 0
        for nm, x, y in zip(("master", "m", "v"), (u.master, u.m, u.v), plain):
            assert torch.equal(x, y), nm
        del plain
        for i, n in enumerate(w.numels):
            want = oracle.gather_tensor(op, i, params_ref)
            assert np.array_equal(outs[i][:n].cpu().numpy().view(np.uint16), want), (w.name, i)
            assert np.array_equal(gathered[i][:n].cpu().numpy().view(np.uint16), want), (w.name, i, "gather")
    finally:
        u.close()


def test_reshard_full_size_matches_oracle():
    """The bench's checkpoint row on the 67M plan: state written under the
    plan's geometry (tp 2, dp_replicate 2, dp_shard 4), moved to the
    canonical logical order (grs_state_to_logical) and into the reader's
    geometry (bench.reshard_geometry: dp_shard over all data ranks) with
    grs_state_from_logical; both results equal the oracle's own layout
    conversions element for element, bit for bit (padding zeros
    included)."""
    import bench
    from gradient_reduction_sharded_gb300 import grs as g

    w = workloads.get(1)
    tp, dr, ds = bench.reshard_geometry(w)
    assert (tp, dr, ds) != (w.tp, w.dp_replicate, w.dp_shard)
    ow = oracle.plan(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    orr = oracle.plan(w.numels, w.owners, w.world, tp, dr, ds, w.bucket_bytes)
    pw = g.grs_plan_create(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    pr = g.grs_plan_create(w.numels, w.owners, w.world, tp, dr, ds, w.bucket_bytes)
    try:
        iw, ir = g.grs_plan_query(pw), g.grs_plan_query(pr)
        assert iw["n_state_pad"] == ow.n_state_pad and ir["n_state_pad"] == orr.n_state_pad
        s = torch.cuda.current_stream().cuda_stream
        gen = torch.Generator(device="cuda").manual_seed(17)
        src = torch.randn(iw["n_state_pad"], generator=gen, device="cuda")
        lg = torch.empty(iw["n_unique"], device="cuda")
        dst = torch.full((ir["n_state_pad"],), float("nan"), device="cuda")
        g.grs_state_to_logical(pw, src.data_ptr(), lg.data_ptr(), s)
        g.grs_state_from_logical(pr, lg.data_ptr(), dst.data_ptr(), s)
        torch.cuda.synchronize()
        assert g.grs_check_device_errors(pw, s) == 0 and g.grs_check_device_errors(pr, s) == 0
        want_lg = oracle.to_logical(ow, src.cpu().numpy())
        assert np.array_equal(lg.cpu().numpy(), want_lg)
        assert np.array_equal(dst.cpu().numpy(), oracle.from_logical(orr, want_lg))
    finally:
        g.grs_plan_destroy(pw)
        g.grs_plan_destroy(pr)


def test_accumulate_full_size_matches_fp32_addition():
    """grs_accumulate over every bucket of the 3.2B plan (the entry point
    whose 142 launches the bench times): each accumulator element becomes
    the IEEE fp32 sum of its old value and the reduced microbatch's (numpy
    float32 addition, round to nearest even), padding exactly zero; bucket
    rows compared whole, one at a time."""
    from gradient_reduction_sharded_gb300 import grs as g

    w = workloads.get(4)
    plan = g.grs_plan_create(w.numels, w.owners, w.world, w.tp, w.dp_replicate, w.dp_shard, w.bucket_bytes)
    try:
        info = g.grs_plan_query(plan)
        nsp = info["n_state_pad"]
        if _free_gb() < 3 * nsp * 4 / 1e9 + 8:
            pytest.skip("needs about 47 GB of device memory")
        s = torch.cuda.current_stream().cuda_stream
        gen = torch.Generator(device="cuda").manual_seed(23)
        acc = torch.randn(nsp, generator=gen, device="cuda")
        mb = torch.randn(nsp, generator=gen, device="cuda")
        before = acc.clone()
        buckets = [g.grs_bucket_info(plan, b) for b in range(info["n_buckets"])]
        for b, d in enumerate(buckets):
            lo = int(d["state_offset"])
            g.grs_accumulate(plan, b, acc.data_ptr() + 4 * lo, mb.data_ptr() + 4 * lo, s)
        torch.cuda.synchronize()
        assert g.grs_check_device_errors(plan, s) == 0
        for d in buckets:
            lo, P, used = int(d["state_offset"]), int(d["padded"]), int(d["used"])
            for r in range(int(d["copies"])):
                a0 = lo + r * P
                x = before[a0:a0 + P].cpu().numpy()
                y = mb[a0:a0 + P].cpu().numpy()
                want = np.add(x, y, dtype=np.float32)
                want[used:] = 0.0
                assert np.array_equal(acc[a0:a0 + P].cpu().numpy(), want), (d, r)
    finally:
        g.grs_plan_destroy(plan)
