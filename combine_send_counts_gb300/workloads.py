"""Seeded synthetic inputs for MoE top-k dispatch / combine.

This module only draws inputs: hidden rows, router choices (``topk_idx``),
router weights (``topk_weights``) and stand-in expert outputs.  It holds none
of the dispatch / combine arithmetic, so both the CUDA path and the CPU oracle
consume the same arrays without sharing any of the method's code.

Every tensor comes from its own PCG64 substream (``SeedSequence.spawn``), so a
tensor's values do not depend on which other tensors were drawn.  Hidden rows
and expert outputs are N(0,1) drawn in float32 and rounded to bfloat16 by
torch's CPU conversion.

Workloads (the five shapes on which the method is exercised):

========== ======= ===== ===== == == ================================== ======================
name       T       H     E     K  P  routing                            weights
========== ======= ===== ===== == == ================================== ======================
tiny       128     256   16    2  4  K distinct, uniform                softmax of K N(0,1)
mid        4096    2048  64    6  8  K distinct, uniform; 5% slots -1   softmax over routed
large      16384   7168  256   8  8  K distinct, Zipf(1.2) popularity   sigmoid, normalised
batched    8192    4096  128   8  4  K distinct, uniform; rank 1, M=4096 softmax
chunk_fp8  32768   7168  256   8  16 K distinct, Zipf(1.0); 4 chunks    softmax
========== ======= ===== ===== == == ================================== ======================

Zipf routing draws K experts without replacement with probability
proportional to ``(e+1)**-s`` (expert id = popularity rank, so expert 0 and
therefore rank 0 is hot).  Sequential sampling without replacement is drawn
with the Gumbel-top-k construction.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

# substream indices; never reorder (it would change every workload)
_S_X, _S_ROUTE, _S_LOGIT, _S_DROP, _S_Y = range(5)
_N_STREAMS = 8


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # hidden size (bf16 elements per row)
    E: int            # experts
    K: int            # top-k slots per token
    P: int            # logical destination ranks (partitions of one HBM)
    routing: str      # "uniform" | "zipf"
    zipf_s: float = 0.0
    unrouted_frac: float = 0.0
    weights: str = "softmax"      # "softmax" | "sigmoid_norm"
    rank: int = 0                 # local rank for the expert-batched layout
    max_num_tokens: int = 0       # M for the expert-batched layout
    chunks: int = 1
    fp8: bool = False
    seed: int = 0

    @property
    def E_local(self) -> int:
        return self.E // self.P

    def scaled(self, T: int, name: Optional[str] = None) -> "Workload":
        """Same recipe with another token count (for oracle-sized parity cases)."""
        return dataclasses.replace(self, T=T, name=name or f"{self.name}_T{T}")

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["E_local"] = self.E_local
        return d


WORKLOADS = {
    "tiny": Workload("tiny", T=128, H=256, E=16, K=2, P=4, routing="uniform"),
    "mid": Workload("mid", T=4096, H=2048, E=64, K=6, P=8, routing="uniform",
                    unrouted_frac=0.05),
    "large": Workload("large", T=16384, H=7168, E=256, K=8, P=8, routing="zipf",
                      zipf_s=1.2, weights="sigmoid_norm"),
    "batched": Workload("batched", T=8192, H=4096, E=128, K=8, P=4, routing="uniform",
                        rank=1, max_num_tokens=4096),
    "chunk_fp8": Workload("chunk_fp8", T=32768, H=7168, E=256, K=8, P=16, routing="zipf",
                          zipf_s=1.0, chunks=4, fp8=True),
}


def _streams(seed: int):
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(_N_STREAMS)]


def _to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def hidden(w: Workload) -> torch.Tensor:
    """x [T,H] bf16, N(0,1)."""
    g = _streams(w.seed)[_S_X]
    return _to_bf16(g.standard_normal((w.T, w.H), dtype=np.float32))


def routing(w: Workload):
    """(topk_idx [T,K] int64 with -1 = unrouted, topk_weights [T,K] float32).

    Weights are 0 on unrouted slots; over the routed slots they are a softmax of
    N(0,1) logits, or sigmoid(logit) normalised to sum 1.
    """
    st = _streams(w.seed)
    T, E, K = w.T, w.E, w.K
    g = st[_S_ROUTE]
    if w.routing == "uniform":
        keys = g.random((T, E))
    elif w.routing == "zipf":
        log_p = -w.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        u = g.random((T, E))
        keys = log_p[None, :] - np.log(-np.log(u))   # Gumbel-top-k
    else:
        raise ValueError(w.routing)
    idx = np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int64)

    routed = np.ones((T, K), dtype=bool)
    if w.unrouted_frac > 0:
        n_drop = int(np.floor(w.unrouted_frac * T * K))
        drop = st[_S_DROP].choice(T * K, size=n_drop, replace=False)
        routed.reshape(-1)[drop] = False
        idx[~routed] = -1

    logits = st[_S_LOGIT].standard_normal((T, K), dtype=np.float32)
    if w.weights == "softmax":
        z = np.where(routed, logits, np.float32(-np.inf))
        z = z - np.max(np.where(routed, z, np.float32(-1e30)), axis=1, keepdims=True)
        e = np.where(routed, np.exp(z), np.float32(0))
    elif w.weights == "sigmoid_norm":
        e = np.where(routed, np.float32(1) / (np.float32(1) + np.exp(-logits)), np.float32(0))
    else:
        raise ValueError(w.weights)
    s = e.sum(axis=1, keepdims=True, dtype=np.float32)
    wts = np.where(s > 0, e / np.where(s > 0, s, np.float32(1)), np.float32(0)).astype(np.float32)
    return torch.from_numpy(idx), torch.from_numpy(np.ascontiguousarray(wts))


def expert_outputs(w: Workload, n_rows: int) -> torch.Tensor:
    """Stand-in expert outputs Y [n_rows, H] bf16, N(0,1).

    The row count comes from the caller (each side counts its own received
    rows); the first r rows are the same whatever n_rows >= r is asked for.
    """
    g = _streams(w.seed)[_S_Y]
    return _to_bf16(g.standard_normal((int(n_rows), w.H), dtype=np.float32))


def batched_expert_outputs(w: Workload, tokens_per_expert) -> torch.Tensor:
    """Stand-in expert outputs in the expert-batched layout [E_local, M, H] bf16.

    Rows below ``tokens_per_expert[e]`` hold N(0,1) values (taken in expert
    order from one stream); padding rows hold NaN so that a combine that reads
    padding shows it.
    """
    tpe = np.asarray(tokens_per_expert, dtype=np.int64)
    M = w.max_num_tokens
    pool = expert_outputs(w, int(tpe.sum()))
    y = torch.full((w.E_local, M, w.H), float("nan"), dtype=torch.bfloat16)
    off = 0
    for e in range(w.E_local):
        c = int(tpe[e])
        y[e, :c] = pool[off:off + c]
        off += c
    return y


def make(w: Workload):
    """x, topk_idx, topk_weights for a workload (all CPU tensors)."""
    idx, wts = routing(w)
    return hidden(w), idx, wts
