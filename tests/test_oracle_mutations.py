"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a temporary copy of oracle.c (CPU only),
builds it, points the oracle binding at it and runs the pins of
test_oracle_pins.py: at least one must fail.  The real oracle is restored
after every case.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = [
    ("rank order: replica and shard swapped", "return (r * dp_shard + s) * tp + t;",
     "return (s * dp_shard + r) * tp + t;"),
    ("REPLICA_AVG not averaged across TP", "tp_value = (tag == OR_REPLICA_AVG) ? tp_sum / tp : tp_sum;",
     "tp_value = tp_sum;"),
    ("PARTIAL_SUM averaged instead of summed", "tp_value = (tag == OR_REPLICA_AVG) ? tp_sum / tp : tp_sum;",
     "tp_value = tp_sum / tp;"),
    ("DP summed instead of averaged", "reduced = dp_sum / dp;", "reduced = dp_sum;"),
    ("LOCAL_SHARD reads tp index 0 for every row",
     "tp_value = value(grads, mb + (int64_t)oracle_rank(r, s, c, dp_shard, tp) * P + e);",
     "tp_value = value(grads, mb + (int64_t)oracle_rank(r, s, 0, dp_shard, tp) * P + e);"),
    ("ALREADY_REDUCED reads the last rank",
     "reduced = value(grads, mb + (int64_t)oracle_rank(0, 0, 0, dp_shard, tp) * P + e);",
     "reduced = value(grads, mb + (int64_t)(R - 1) * P + e);"),
    ("padding not zeroed", "acc[(int64_t)c * P + e] = 0.0;\n        continue;", "acc[(int64_t)c * P + e] = 0.0;"),
    ("norm ignores the microbatch mean", "double g = acc[e] / M;", "double g = acc[e];"),
    ("clip coefficient without the 1e-6", "c = max_norm / (sqrt(norm_sq) + 1e-6);", "c = max_norm / sqrt(norm_sq);"),
    ("clip coefficient not capped at 1", "return c < 1.0 ? c : 1.0;", "return c;"),
    ("AdamW without bias correction", "p = p - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps);",
     "p = p - lr * m / (sqrt(v) + eps);"),
    ("AdamW second moment of g, not g^2", "v = b2 * v + (1.0 - b2) * g * g;", "v = b2 * v + (1.0 - b2) * g;"),
    ("AdamW weight decay dropped", "p = p * (1.0 - lr * wd);", "p = p;"),
    ("bf16 ties rounded up, not to even", "w += 0x7fffu + ((w >> 16) & 1u);", "w += 0x8000u;"),
    ("padding quantum ignores dp_shard", "int64_t quantum = 8 * (int64_t)d[0];", "int64_t quantum = 8;"),
    ("greedy bucket test off by one", "2 * (used + per_rank) > bucket_bytes", "2 * (used + per_rank) >= bucket_bytes"),
    ("LOCAL_SHARD counted with its full numel per rank",
     "per_rank = (tag == OR_LOCAL_SHARD) ? numel[i] / tp : numel[i];", "per_rank = numel[i];"),
    ("bf16 gather: LOCAL_SHARD row t at t * chunk instead of t * padded",
     "params_full[bucket_state_off + (int64_t)t * bucket_padded + tensor_offset + i];",
     "params_full[bucket_state_off + (int64_t)t * chunk + tensor_offset + i];"),
    ("bf16 gather: offset inside the bucket dropped",
     "for (i = 0; i < numel; ++i) dst[i] = params_full[bucket_state_off + tensor_offset + i];",
     "for (i = 0; i < numel; ++i) dst[i] = params_full[bucket_state_off + i];"),
    ("bf16 gather: LOCAL_SHARD chunks in reverse tp order",
     "dst[t * chunk + i] =\n            params_full[",
     "dst[(tp - 1 - t) * chunk + i] =\n            params_full["),
    ("LOCAL_SHARD rows gathered in the wrong place",
     "dst[t * chunk + i] = state[bucket_state_off + (int64_t)t * bucket_padded + tensor_offset + i];",
     "dst[t * chunk + i] = state[bucket_state_off + tensor_offset + (int64_t)t * chunk + i];"),
]


# The pins of the fp32 accumulation error bound (Python side of the oracle).
BOUND_PINS = [
    ("bound_ranks", lambda: pins.test_accumulation_bound_absorption_across_ranks(None)),
    ("bound_micro", lambda: pins.test_accumulation_bound_absorption_across_microbatches(None)),
    ("bound_abs", lambda: pins.test_accumulation_bound_uses_absolute_values(None)),
    ("bound_random", lambda: pins.test_accumulation_bound_random_cancelling(None, 12, 3)),
    ("gamma", lambda: pins.test_gamma_closed_form(None)),
]


def run_pins():
    """Run the pins; return the names of those that fail."""
    failed = []
    calls = [
        ("hand_checked_single", lambda: pins.test_hand_checked_single_microbatch(None)),
        ("hand_checked_two", lambda: pins.test_hand_checked_two_microbatches(None)),
        ("hand_checked_fp32", lambda: pins.test_hand_checked_fp32_gradients(None)),
        ("dp_mesh", lambda: pins.test_dp_mesh_rank_order(None)),
        ("padding", lambda: pins.test_padding_ignored_and_zero(None)),
        ("identical", lambda: pins.test_identical_copies(None, 2, 2, 4)),
        ("already_reduced", lambda: pins.test_already_reduced_ignores_other_ranks(None)),
        ("local_shard", lambda: pins.test_local_shard_not_synchronised_across_tp(None)),
        ("norm", lambda: pins.test_norm_closed_form(None)),
        ("clip", lambda: pins.test_clip_special_cases(None)),
        ("adamw_step1", lambda: pins.test_adamw_step1_closed_form(None)),
        ("adamw_zero", lambda: pins.test_adamw_zero_gradient(None)),
        ("adamw_torch", lambda: pins.test_adamw_multistep_matches_torch(None, (1e-3, 0.9, 0.999, 1e-8, 0.01))),
        ("bf16", lambda: pins.test_bf16_rne_matches_torch(None)),
        ("logical", lambda: pins.test_logical_layout_hand_derived(None)),
        ("gather_bf16", lambda: pins.test_gather_tensor_bf16_hand_derived(None)),
    ] + BOUND_PINS + [(f"plan:{c['name']}", (lambda c=c: pins.test_plan_hand_derived(None, c)))
         for c in pins.PLAN_CASES["cases"]]
    for name, fn in calls:
        try:
            fn()
        except (AssertionError, oracle.OracleError):
            failed.append(name)
    return failed


def test_pins_pass_on_the_real_oracle():
    assert run_pins() == []


@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(what, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old}"
    mutant = src.replace(old, new)
    c_path = os.path.join(tmp_path, "oracle.c")
    with open(c_path, "w") as f:
        f.write(mutant)
    hdr = os.path.join(os.path.dirname(SRC), "oracle.h")
    so = os.path.join(tmp_path, "liboracle_mutant.so")
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                           "-I", os.path.dirname(hdr), "-o", so, c_path, "-lm"])
    real = oracle.lib()
    try:
        oracle._lib = oracle.load_library(so)
        failed = run_pins()
    finally:
        oracle._lib = real
    assert failed, f"no pin caught the mutant: {what}"


# Plausible slips in the bound that widens the master/moment checks: each
# replaces one function of the oracle's Python side, and a pin must fail.
U = 2.0 ** -24
BOUND_MUTANTS = [
    ("bound without the group's additions ((M + 2) u)", "accumulation_error_bound",
     lambda acc_abs, M, group: (M + 2) * U * acc_abs),
    ("bound without the microbatch term", "accumulation_error_bound",
     lambda acc_abs, M, group: oracle.gamma(group + 1) * acc_abs),
    ("bound four times too wide", "accumulation_error_bound",
     lambda acc_abs, M, group: 4 * oracle.gamma(group + M + 1) * acc_abs),
    ("bound from the signed inputs", "abs_inputs", lambda g: g),
    ("gamma without its denominator", "gamma", lambda k: k * U),
]


@pytest.mark.parametrize("what,name,fn", BOUND_MUTANTS, ids=[m[0] for m in BOUND_MUTANTS])
def test_bound_pins_catch_mutant(what, name, fn, monkeypatch):
    monkeypatch.setattr(oracle, name, fn)
    failed = []
    for nm, call in BOUND_PINS:
        try:
            call()
        except AssertionError:
            failed.append(nm)
    assert failed, f"no pin caught the mutant: {what}"
