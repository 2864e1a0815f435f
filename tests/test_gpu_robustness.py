"""Robustness of the CUDA path: no writes outside the output buffers (guard
canaries), results independent of the reduction's grid size, and two host
threads driving separate plans on separate streams at once."""
import threading

import numpy as np
import pytest
import torch

from gpu_support import Case, Run, grs

pytestmark = pytest.mark.gpu

RA, PS, LS, AR = 0, 1, 2, 3
GUARD = 4096  # elements of canary on each side


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


def guarded(n, dtype, fill):
    """A buffer of n elements with GUARD canary elements on both sides."""
    full = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return full, full[GUARD:GUARD + n]


def canaries_intact(full, fill):
    lo, hi = full[:GUARD], full[-GUARD:]
    if full.dtype.is_floating_point and np.isnan(fill):
        return bool(torch.isnan(lo).all() and torch.isnan(hi).all())
    return bool((lo == fill).all() and (hi == fill).all())


def test_no_writes_outside_outputs():
    g = grs()
    c = Case([100003, 1024, 65536 * 2, 4099, 333, 70001, 8000], [RA, PS, LS, AR, PS, RA, LS], 16, 2, 2, 4,
             1 << 18, 2, 1e-3, 71)
    run = Run(c)
    try:
        nsp, s = run.nsp, run.stream()
        bufs = {}
        for name, dt, fill in (("acc", torch.float32, float("nan")), ("master", torch.float32, float("nan")),
                               ("m", torch.float32, float("nan")), ("v", torch.float32, float("nan")),
                               ("params", torch.int16, -12345)):
            full, view = guarded(nsp, dt, fill)
            src = getattr(run, name)[:nsp]
            view.copy_(src)
            bufs[name] = (full, view, fill)
        ws_full, ws = guarded(run.ws.numel(), torch.float32, float("nan"))
        ws.zero_()
        nrm_full, nrm = guarded(1, torch.float64, float("nan"))
        for j in range(c.n_micro):
            g.grs_reduce_all(run.plan, run.ptrs(j), bufs["acc"][1].data_ptr(), int(j > 0), int(j == c.n_micro - 1),
                             ws.data_ptr(), s)
        g.grs_grad_norm_sq(run.plan, bufs["acc"][1].data_ptr(), c.n_micro, ws.data_ptr(), 1, nrm.data_ptr(), s)
        hp = g.make_adamw(*c.hp, c.max_norm, 1, c.n_micro)
        g.grs_clip_adamw_step(run.plan, hp, nrm.data_ptr(), bufs["acc"][1].data_ptr(), bufs["master"][1].data_ptr(),
                              bufs["m"][1].data_ptr(), bufs["v"][1].data_ptr(), bufs["params"][1].data_ptr(), s)
        g.grs_grad_norm_sq(run.plan, bufs["acc"][1].data_ptr(), c.n_micro, ws.data_ptr(), 0, nrm.data_ptr(), s)
        outs = [guarded(n, torch.int16, 777) for n in c.numels]
        g.grs_gather_params(run.plan, bufs["params"][1].data_ptr(), [v.data_ptr() for _, v in outs], s)
        torch.cuda.synchronize()
        assert run.check_flags() == 0
        for name, (full, view, fill) in bufs.items():
            assert canaries_intact(full, fill), name
        assert canaries_intact(ws_full, float("nan"))
        assert canaries_intact(nrm_full, float("nan"))
        for full, _ in outs:
            assert canaries_intact(full, 777)
        assert torch.isfinite(bufs["master"][1]).all()
    finally:
        run.close()


def test_masked_and_layout_calls_write_inside_outputs():
    """The masked norm, the masked reduction with its fused norm partials and
    the masked update (tensors without a gradient, zero-size tensors among
    them) and the state layout conversions write nothing
    outside their outputs; the masked update leaves the state of tensors
    without a gradient untouched and the layout restore writes every
    padding element as zero."""
    g = grs()
    numels = [100003, 0, 1024, 65536 * 2, 4099, 333, 0, 70001, 8000]
    owners = [RA, RA, PS, LS, AR, PS, LS, RA, LS]
    c = Case(numels, owners, 16, 2, 2, 4, 1 << 18, 2, 1e-3, 72)
    run = Run(c)
    try:
        nsp, s = run.nsp, run.stream()
        n = len(numels)
        used = torch.tensor([1, 1, 0, 1, 1, 0, 0, 1, 0], dtype=torch.uint8, device="cuda")
        acc_full, acc = guarded(nsp, torch.float32, float("nan"))
        st = {}
        for name, dt, fill in (("master", torch.float32, float("nan")), ("m", torch.float32, float("nan")),
                               ("v", torch.float32, float("nan")), ("params", torch.int16, -12345)):
            full, view = guarded(nsp, dt, fill)
            view.copy_(getattr(run, name)[:nsp])
            st[name] = (full, view, fill)
        before = {k: v[1].clone() for k, v in st.items()}
        steps_full, steps = guarded(n, torch.int32, -7)
        steps.zero_()
        ws_full, ws = guarded(run.ws.numel(), torch.float32, float("nan"))
        ws.zero_()
        nrm_full, nrm = guarded(1, torch.float64, float("nan"))
        for j in range(c.n_micro):
            g.grs_reduce_all(run.plan, run.ptrs(j), acc.data_ptr(), int(j > 0), 0, ws.data_ptr(), s)
        g.grs_grad_norm_sq_masked(run.plan, acc.data_ptr(), c.n_micro, used.data_ptr(), ws.data_ptr(),
                                  nrm.data_ptr(), s)
        # the masked reduction with its fused norm partials, then the finish alone
        for j in range(c.n_micro):
            g.grs_reduce_all_masked(run.plan, run.ptrs(j), acc.data_ptr(), int(j > 0), int(j == c.n_micro - 1),
                                    used.data_ptr(), ws.data_ptr(), s)
        g.grs_grad_norm_sq(run.plan, acc.data_ptr(), c.n_micro, ws.data_ptr(), 1, nrm.data_ptr(), s)
        hp = g.make_adamw(*c.hp, c.max_norm, 1, c.n_micro)
        g.grs_clip_adamw_step_masked(run.plan, hp, nrm.data_ptr(), acc.data_ptr(), st["master"][1].data_ptr(),
                                     st["m"][1].data_ptr(), st["v"][1].data_ptr(), st["params"][1].data_ptr(),
                                     used.data_ptr(), steps.data_ptr(), ws.data_ptr(), s)
        nu = run.info["n_unique"]
        lg_full, lg = guarded(nu, torch.float32, float("nan"))
        g.grs_state_to_logical(run.plan, st["master"][1].data_ptr(), lg.data_ptr(), s)
        back_full, back = guarded(nsp, torch.float32, float("nan"))  # interior NaN too: padding must be written
        g.grs_state_from_logical(run.plan, lg.data_ptr(), back.data_ptr(), s)
        torch.cuda.synchronize()
        assert run.check_flags() == 0
        for full, fill in ((acc_full, float("nan")), (steps_full, -7), (ws_full, float("nan")),
                           (nrm_full, float("nan")), (lg_full, float("nan")), (back_full, float("nan"))):
            assert canaries_intact(full, fill)
        for name, (full, view, fill) in st.items():
            assert canaries_intact(full, fill), name
        assert steps.cpu().tolist() == [int(u) for u in used.cpu().tolist()]
        assert torch.equal(back, st["master"][1])  # padding included: exact zeros both sides
        # tensors without a gradient: state untouched, bit for bit
        op = run.op
        for i in range(n):
            if used[i].item():
                continue
            for lo, hi in op.tensor_rows(i):
                for name in ("master", "m", "v", "params"):
                    a, b = st[name][1][lo:hi], before[name][lo:hi]
                    assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                                       b.view(torch.int32) if b.dtype == torch.float32 else b), (i, name)
    finally:
        run.close()


def test_hundred_updates_are_deterministic():
    """Two independent runs of 100 updates (new gradients each step, two
    microbatches, every owner tag) end in bit-identical accumulator, norm,
    master, moments and bf16 parameters: nothing in the path depends on
    scheduling."""
    c = Case([100003, 1024, 65536 * 2, 4099, 333, 70001, 8000], [RA, PS, LS, AR, PS, RA, LS], 16, 2, 2, 4,
             1 << 18, 2, 1e-3, 73)
    finals = []
    for _ in range(2):
        run = Run(c)
        try:
            for step in range(1, 101):
                if step > 1 and step % 10 == 1:
                    run.fill_grads(step_seed=step)
                run.update()
            torch.cuda.synchronize()
            assert run.check_flags() == 0
            finals.append([t.clone() for t in (run.acc, run.norm, run.master, run.m, run.v, run.params)])
        finally:
            run.close()
    for a, b in zip(*finals):
        assert torch.equal(a, b)


def test_results_do_not_depend_on_the_grid():
    g = grs()
    c = Case([100003, 1024, 65536 * 2, 4099, 333], [RA, PS, LS, AR, PS], 16, 2, 2, 4, 1 << 18, 1, 1e-3, 72)
    run = Run(c)
    try:
        s = run.stream()
        ref_acc = ref_part = None
        for cap in (0, 1, 7, 152, 1000):
            run.acc.fill_(7.0)
            run.ws.zero_()
            for b in range(run.info["n_buckets"]):
                d = g.grs_bucket_info(run.plan, b)
                rp = [p + 2 * d["rank_offset"] for p in run.ptrs(0)]
                g.grs_reduce_bucket_ex(run.plan, b, rp, run.acc.data_ptr() + 4 * d["state_offset"], 0, 1,
                                       run.ws.data_ptr(), cap, None, s)
            torch.cuda.synchronize()
            part = run.ws[:run.info["n_reduce_tiles"]].clone()
            if ref_acc is None:
                ref_acc, ref_part = run.acc.clone(), part
            assert torch.equal(run.acc, ref_acc), cap
            assert torch.equal(part, ref_part), cap
    finally:
        run.close()


def test_two_threads_two_plans_two_streams():
    cases = [Case([50001, 512, 8192 * 2, 77], [RA, PS, LS, AR], 8, 2, 2, 2, 1 << 16, 2, 1e-3, 73 + i)
             for i in range(2)]
    refs = []
    for c in cases:  # sequential reference
        r = Run(c)
        r.update()
        torch.cuda.synchronize()
        refs.append([t.clone() for t in (r.acc, r.norm, r.master, r.m, r.v, r.params)])
        r.close()
    runs = [Run(c) for c in cases]
    torch.cuda.synchronize()  # buffers initialised before the threads' streams use them
    errors = []

    def work(run):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(1):
                    run.update()
                st.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(r,)) for r in runs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    try:
        assert not errors, errors
        for r, ref in zip(runs, refs):
            for x, y in zip((r.acc, r.norm, r.master, r.m, r.v, r.params), ref):
                assert torch.equal(x, y)
    finally:
        for r in runs:
            r.close()


@pytest.mark.parametrize("route", ["separate-masked-norm", "masked-reduction-partials"])
def test_step_captured_in_a_cuda_graph_matches_eager(route):
    """One update (grouped reduction, masked norm, masked AdamW with device
    step counters) captured once in a CUDA graph and replayed three times
    equals three eager updates: the path is stream-ordered, allocation-free
    and keeps its step counts on the device.  Two routes: the plain
    reduction and the separate masked norm pass, or the masked reduction
    with its fused partials and the finish alone (one tensor without a
    gradient)."""
    c = Case([50001, 512, 8192 * 2, 77], [RA, PS, LS, AR], 8, 2, 2, 2, 1 << 16, 2, 1e-3, 81)
    eager, graph_run = Run(c), Run(c)
    fused = route == "masked-reduction-partials"
    try:
        n = len(c.numels)
        used = torch.tensor([1, 0, 1, 1] if fused else [1] * n, dtype=torch.uint8, device="cuda")
        st_e = torch.zeros(n, dtype=torch.int32, device="cuda")
        st_g = torch.zeros(n, dtype=torch.int32, device="cuda")

        def step(run, st):
            if fused:
                run.masked_reduce(used)
            else:
                run.reduce(emit=False)
            run.masked_update(used, st, partials_ready=fused)

        for _ in range(3):
            step(eager, st_e)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            # the library needs no warm-up allocations: capture directly
            with torch.cuda.graph(graph, stream=side):
                step(graph_run, st_g)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        want_steps = [3 * int(u) for u in used.tolist()]
        assert st_g.tolist() == st_e.tolist() == want_steps
        for x, y in ((eager.norm, graph_run.norm), (eager.master, graph_run.master),
                     (eager.m, graph_run.m), (eager.v, graph_run.v), (eager.params, graph_run.params)):
            assert torch.equal(x, y)
        if not fused:  # with a mask the accumulator of the tensor without a gradient is unspecified
            assert torch.equal(eager.acc, graph_run.acc)
    finally:
        eager.close()
        graph_run.close()
