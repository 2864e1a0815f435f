"""grs_grad_norm_sq_noalloc: the global norm for callers that cannot allocate
device memory (a process whose caching allocator already holds the GPU's
memory, latency-critical code that cannot take an allocation's device
synchronisation, a host that only gets device pointers from another
runtime).  It keeps its scratch in a static device array instead of a
caller-provided workspace.

Checked through the C ABI against grs_grad_norm_sq (the workspace entry
point, with partials_ready = 0: the same pass and the same fixed-order fp64
finish, so the two agree bit for bit) and against the oracle's norm within
the suite's tolerance, on two calls in a row with different plans, so
contents left in the shared array by one call cannot leak into the next.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_support import RTOL, ATOL, Case, Run, case_from_workload, grs, oracle_update

pytestmark = pytest.mark.gpu

RA, PS, LS, AR = 0, 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.init()


def _norm_both(run: Run):
    g = grs()
    s = run.stream()
    run.reduce(emit=False)
    ref = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
    got = torch.full((1,), -2.0, dtype=torch.float64, device="cuda")
    g.grs_grad_norm_sq(run.plan, run.acc.data_ptr(), run.c.n_micro, run.ws.data_ptr(), 0,
                       ref.data_ptr(), s)
    g.grs_grad_norm_sq_noalloc(run.plan, run.acc.data_ptr(), run.c.n_micro, got.data_ptr(), s)
    torch.cuda.synchronize()
    return float(ref.cpu()[0]), float(got.cpu()[0])


def test_noalloc_norm_matches_workspace_entry_point_twice():
    cases = [
        Case([100003, 1024, 65536 * 2, 4099, 333, 70001, 8 * 1000], [RA, PS, LS, AR, PS, RA, LS],
             16, 2, 2, 4, 1 << 18, 2, 1e-3, 31),
        case_from_workload(0),
    ]
    seen = []
    for c in cases:
        run = Run(c)
        try:
            master0, m0, v0 = run.state_host()
            ref, got = _norm_both(run)
            assert ref > 0
            assert got == ref, (got, ref)  # bit for bit
            want = oracle_update(run, master0, m0, v0, step=1).norm_sq
            assert abs(got - want) <= ATOL + RTOL * abs(want), (got, want)
            seen.append(got)
        finally:
            run.close()
    assert seen[0] != seen[1]


def test_noalloc_rejects_plans_beyond_the_scratch_size():
    g = grs()
    # one 2^33-element tensor on one rank: 2^33 / 8192 > 10^6 reduction tiles
    plan = g.grs_plan_create([1 << 33], [RA], 1, 1, 1, 1, 1 << 40)
    try:
        acc = torch.zeros(16, dtype=torch.float32, device="cuda")
        out = torch.zeros(1, dtype=torch.float64, device="cuda")
        with pytest.raises(g.GrsError) as ei:
            g.grs_grad_norm_sq_noalloc(plan, acc.data_ptr(), 1, out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
        assert ei.value.status == g.GRS_ERR_SHAPE
        assert "scratch" in g.grs_last_error()
        assert float(out.cpu()[0]) == 0.0
    finally:
        g.grs_plan_destroy(plan)
