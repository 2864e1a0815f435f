"""Synthetic workloads and seeded input generators.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests.  It holds *only* workload descriptions (tensor shapes, owner tags,
parallel degrees, hyper-parameters) and seeded random generators.  It holds
none of the method's arithmetic: no routing, no reduction, no bucketing, no
norm, no optimizer step.

The workloads follow the shapes described for the ownership-aware
reduction problem ("refactor(distributed): establish shared native TP
replica ownership", section *Why this needs separate work*: replica /
partial / local-shard / already-reduced gradients) and the HSDP geometry of
"Cosmos 3 training framework / distributed parallelism" (section 1, the
four axes: dp_replicate x dp_shard = world).  No public dataset is involved:
every value is drawn from a seeded normal distribution.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np

# Owner tags, in the numbering the C boundary uses.
REPLICA_AVG = 0
PARTIAL_SUM = 1
LOCAL_SHARD = 2
ALREADY_REDUCED = 3
OWNER_NAMES = ("REPLICA_AVG", "PARTIAL_SUM", "LOCAL_SHARD", "ALREADY_REDUCED")

MIB = 1 << 20
DEFAULT_BUCKET_BYTES = 25 * MIB  # "25 MB buckets", read as 25 MiB


@dataclass
class Tensor:
    name: str
    shape: Tuple[int, ...]
    owner: int

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= int(s)
        return n


@dataclass
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_norm: float = 1.0  # <= 0 turns clipping off


@dataclass
class Workload:
    cid: int
    name: str
    tensors: List[Tensor]
    tp: int
    dp_replicate: int
    dp_shard: int
    n_micro: int
    grad_std: float
    master_std: float = 0.02
    bucket_bytes: int = DEFAULT_BUCKET_BYTES
    adamw: AdamW = field(default_factory=AdamW)

    @property
    def world(self) -> int:
        return self.tp * self.dp_replicate * self.dp_shard

    @property
    def numels(self) -> List[int]:
        return [t.numel for t in self.tensors]

    @property
    def owners(self) -> List[int]:
        return [t.owner for t in self.tensors]

    @property
    def n_unique(self) -> int:
        return sum(self.numels)

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "params": self.n_unique,
            "tensors": len(self.tensors),
            "tp": self.tp,
            "dp_replicate": self.dp_replicate,
            "dp_shard": self.dp_shard,
            "world": self.world,
            "microbatches": self.n_micro,
            "bucket_bytes": self.bucket_bytes,
        }


# ---------------------------------------------------------------------------
# Workload 0: the tiny hand-sized plan (world 4: tp 2, dp_shard 2).
# ---------------------------------------------------------------------------
def _tiny() -> Workload:
    ts = [
        Tensor("W_a", (64, 64), REPLICA_AVG),
        Tensor("qnorm", (32,), PARTIAL_SUM),
        Tensor("W_tp", (128, 64), LOCAL_SHARD),
        Tensor("b", (64,), ALREADY_REDUCED),
        Tensor("W_b", (256, 64), REPLICA_AVG),
        Tensor("W_c", (64, 128), LOCAL_SHARD),
    ]
    return Workload(0, "tiny-6-tensor-world4", ts, tp=2, dp_replicate=1, dp_shard=2,
                    n_micro=1, grad_std=1e-2,
                    adamw=AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0))


# ---------------------------------------------------------------------------
# Workload 1: the synthetic 2^26-parameter model (world 16).
# 16 blocks x 4 [1024,1024] matrices: 3 REPLICA_AVG + 1 LOCAL_SHARD each,
# plus 16 PARTIAL_SUM norm vectors [1024].
# ---------------------------------------------------------------------------
def _synthetic67m(blocks: int = 16) -> Workload:
    ts = []
    for i in range(blocks):
        ts.append(Tensor(f"blk{i}.norm", (1024,), PARTIAL_SUM))
        ts.append(Tensor(f"blk{i}.w0", (1024, 1024), REPLICA_AVG))
        ts.append(Tensor(f"blk{i}.w1", (1024, 1024), REPLICA_AVG))
        ts.append(Tensor(f"blk{i}.w2", (1024, 1024), REPLICA_AVG))
        ts.append(Tensor(f"blk{i}.w_tp", (1024, 1024), LOCAL_SHARD))
    name = "synthetic-67M-world16" if blocks == 16 else f"synthetic-{blocks}blk-world16"
    return Workload(1, name, ts, tp=2, dp_replicate=2, dp_shard=4,
                    n_micro=1, grad_std=1e-3,
                    adamw=AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0))


def _llama(d, layers, n_heads, n_kv, ffn, vocab, tied, owner=REPLICA_AVG):
    hd = d // n_heads
    ts = [Tensor("embed", (vocab, d), owner)]
    for i in range(layers):
        p = f"layers.{i}."
        ts += [
            Tensor(p + "input_norm", (d,), owner),
            Tensor(p + "q_proj", (n_heads * hd, d), owner),
            Tensor(p + "k_proj", (n_kv * hd, d), owner),
            Tensor(p + "v_proj", (n_kv * hd, d), owner),
            Tensor(p + "o_proj", (d, n_heads * hd), owner),
            Tensor(p + "post_norm", (d,), owner),
            Tensor(p + "gate_proj", (ffn, d), owner),
            Tensor(p + "up_proj", (ffn, d), owner),
            Tensor(p + "down_proj", (d, ffn), owner),
        ]
    ts.append(Tensor("final_norm", (d,), owner))
    if not tied:
        ts.append(Tensor("lm_head", (vocab, d), owner))
    return ts


# ---------------------------------------------------------------------------
# Workload 2: Llama-shaped 1.1B decoder, HSDP 2 x 4, tp 1, 8 microbatches.
# 32 query heads with 4 KV heads (head_dim 64), untied lm_head: exactly
# 1,100,048,384 parameters.
# ---------------------------------------------------------------------------
# Profiling slices of workloads 2-4 (`layers` > 0): the same geometry, owner
# tags and per-layer shapes with `layers` decoder layers, a SLICE_VOCAB-row
# embedding (and lm_head) and, for the MoE, SLICE_EXPERTS experts: a few GB
# on the device, inputs still larger than L2, so that ncu captures stay small
# while every kernel sees the full workload's per-element traffic.
SLICE_VOCAB = 8192
SLICE_EXPERTS = 8


def _llama1b(layers: int = 0) -> Workload:
    n, vocab = (layers, SLICE_VOCAB) if layers else (22, 32000)
    ts = _llama(2048, n, 32, 4, 5632, vocab, tied=False)
    name = "llama-1.1B-hsdp2x4-8mb" + (f"-slice{layers}L" if layers else "")
    return Workload(2, name, ts, tp=1, dp_replicate=2, dp_shard=4,
                    n_micro=8, grad_std=1e-3,
                    adamw=AdamW(3e-4, 0.9, 0.999, 1e-8, 0.1, 1.0))


# ---------------------------------------------------------------------------
# Workload 3: Qwen3-style MoE, 8 layers, d 2048, 16 heads x 128, tp 2
# (head-sharded), dp_shard 4, 4 microbatches.  Attention projections are
# LOCAL_SHARD, Q/K RMSNorm [128] PARTIAL_SUM, 32 experts stacked as three
# [32, ., .] tensors per layer (expert-owned LOCAL_SHARD, 16 experts per
# tp/ep index), router / norms / embeddings REPLICA_AVG.
# ---------------------------------------------------------------------------
def _qwen3_moe(layers: int = 0) -> Workload:
    d, hd, nh, ne, fe, vocab = 2048, 128, 16, 32, 768, 151936
    n_layers = 8
    if layers:
        n_layers, ne, vocab = layers, SLICE_EXPERTS, SLICE_VOCAB
    ts = [Tensor("embed", (vocab, d), REPLICA_AVG)]
    for i in range(n_layers):
        p = f"layers.{i}."
        ts += [
            Tensor(p + "input_norm", (d,), REPLICA_AVG),
            Tensor(p + "q_proj", (nh * hd, d), LOCAL_SHARD),
            Tensor(p + "k_proj", (nh * hd, d), LOCAL_SHARD),
            Tensor(p + "v_proj", (nh * hd, d), LOCAL_SHARD),
            Tensor(p + "o_proj", (d, nh * hd), LOCAL_SHARD),
            Tensor(p + "q_norm", (hd,), PARTIAL_SUM),
            Tensor(p + "k_norm", (hd,), PARTIAL_SUM),
            Tensor(p + "post_norm", (d,), REPLICA_AVG),
            Tensor(p + "router", (d, ne), REPLICA_AVG),
            Tensor(p + "experts.gate", (ne, fe, d), LOCAL_SHARD),
            Tensor(p + "experts.up", (ne, fe, d), LOCAL_SHARD),
            Tensor(p + "experts.down", (ne, d, fe), LOCAL_SHARD),
        ]
    ts.append(Tensor("final_norm", (d,), REPLICA_AVG))
    ts.append(Tensor("lm_head", (vocab, d), REPLICA_AVG))
    name = "qwen3-moe-8L-tp2-ds4-4mb" + (f"-slice{layers}L" if layers else "")
    return Workload(3, name, ts, tp=2, dp_replicate=1, dp_shard=4,
                    n_micro=4, grad_std=1e-3,
                    adamw=AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0))


# ---------------------------------------------------------------------------
# Workload 4: Llama-3.2-3B-shaped decoder, tied embedding, HSDP 2 x 2.
# ---------------------------------------------------------------------------
def _llama3b(layers: int = 0) -> Workload:
    n, vocab = (layers, SLICE_VOCAB) if layers else (28, 128256)
    ts = _llama(3072, n, 24, 8, 8192, vocab, tied=True)
    name = "llama3.2-3B-hsdp2x2" + (f"-slice{layers}L" if layers else "")
    return Workload(4, name, ts, tp=1, dp_replicate=2, dp_shard=2,
                    n_micro=1, grad_std=1e-3,
                    adamw=AdamW(3e-4, 0.9, 0.999, 1e-8, 0.1, 1.0))


def get(cid: int, blocks: int = 0, layers: int = 0) -> Workload:
    """Workload `cid`.  `blocks` > 0 shrinks workload 1 to that many blocks
    (same tensor shapes and geometry; used for small profiling cases);
    `layers` > 0 gives the profiling slice of workload 2, 3 or 4."""
    if cid == 1 and blocks > 0:
        return _synthetic67m(blocks)
    if layers > 0:
        if cid not in (2, 3, 4):
            raise ValueError("profiling slices exist for workloads 2, 3 and 4")
        return {2: _llama1b, 3: _qwen3_moe, 4: _llama3b}[cid](layers)
    return {0: _tiny, 1: _synthetic67m, 2: _llama1b, 3: _qwen3_moe, 4: _llama3b}[cid]()


ALL_IDS = (0, 1, 2, 3, 4)


# ---------------------------------------------------------------------------
# Seeded generators.  Seeds: grads 1_000_003*cid + 10_007*j + k for
# microbatch j and rank k; master 7_919 + cid.  Values are fp32 normals,
# rounded to bf16 by torch's cast where bf16 is wanted.
# ---------------------------------------------------------------------------
def grad_seed(cid: int, j: int, k: int) -> int:
    return 1_000_003 * cid + 10_007 * j + k


def master_seed(cid: int) -> int:
    return 7_919 + cid


def _torch():
    import torch
    return torch


def normal_bf16(n: int, std: float, seed: int, device="cpu", out=None, chunk=1 << 28):
    """n bf16 values ~ N(0, std), drawn as fp32 from a seeded torch generator.

    When `out` is given (a bf16 tensor of n elements) it is filled in place,
    `chunk` elements at a time, so that the fp32 temporary stays bounded.
    """
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        tmp = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        tmp.mul_(std)
        out[s:e].copy_(tmp)
        del tmp
    return out


def normal_f32(n: int, std: float, seed: int, device="cpu", out=None, chunk=1 << 28):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e].normal_(0.0, std, generator=g)
    return out


def bf16_bits(t) -> np.ndarray:
    """Raw uint16 bit patterns of a CPU bf16 tensor, as a numpy array."""
    torch = _torch()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
