"""Slots of the expert-batched layout (vLLM BatchedPrepareAndFinalize.prepare:
per local expert, the tokens naming it get slots 0, 1, ... in token order;
tokens_per_expert counts them) on both sides of the size at which the library
switches from its one-cluster slot kernel to the grid-wide cooperative one
(16 CTAs x 2 rounds of 1024 tokens = 32 768 tokens where the device runs
clusters of 16, else half that), against the oracle.

The cases cover CTAs of the cluster that own no token, a second round of
tokens in a CTA, exactly the cluster's maximum, the first size past it, more
than 32 local experts (the second ballot word), generic K (no unrolled form),
repeated expert ids, capacity drops and invalid ids."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle

from _paths import assert_equal, bits16, np_, randn_bf16, routing_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # T, K, E, E_local, rank, dup
    (1, 8, 64, 32, 1, False),
    (33, 8, 128, 32, 1, False),          # CTAs 2..15 of the cluster own no token
    (16385, 8, 128, 32, 1, False),       # a second round of 32 tokens in every CTA
    (20000, 3, 96, 48, 1, False),        # generic K, 48 local experts (second ballot word)
    (5000, 1, 64, 64, 0, False),         # K = 1, 64 local experts
    (9000, 32, 256, 64, 3, False),       # K = 32
    (12000, 8, 64, 16, 2, True),         # repeated expert ids
    (16384, 8, 128, 32, 1, False),       # the largest problem of a cluster of 8
    (32768, 8, 128, 32, 1, False),       # the largest problem of a cluster of 16
    (32769, 8, 128, 32, 1, False),       # one token more: the cooperative kernel
    (70000, 3, 96, 32, 2, False),        # cooperative, generic K
]


@pytest.mark.parametrize("T,K,E,El,rank,dup", CASES)
def test_batched_slots_match_oracle(T, K, E, El, rank, dup):
    H = 8
    idx, _ = routing_inputs(T, K, E, seed=T + K, frac_unrouted=0.1, dup=dup)
    x = randn_bf16(T, H, seed=T)
    M = T                                                     # room for every token
    o = oracle.batched_prepare(x, idx, E, El, rank, M)
    err = ep.error_word()
    r = ep.batched_prepare(x.cuda(), idx.cuda(), E, El, rank, M, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and o["err"] == 0
    tpe = o["tokens_per_expert"]
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), tpe)
    assert_equal("slot", np_(r["slot"]), o["slot"])
    bx = bits16(r["b_x"])
    for e in range(El):
        assert_equal(f"b_x[{e}]", bx[e, :tpe[e]], o["b_x"][e, :tpe[e]])


@pytest.mark.parametrize("T", [3000, 70000])
def test_batched_slots_capacity_drops(T):
    # a capacity below the experts' loads: later tokens are dropped (slot -1)
    # and counted, in both slot kernels
    K, E, El, rank, H = 8, 64, 32, 1, 8
    idx, _ = routing_inputs(T, K, E, seed=5 + T, frac_unrouted=0.05)
    x = randn_bf16(T, H, seed=6)
    M = T
    C = max(1, int(T * K / E * 0.6))
    o = oracle.batched_prepare_ex(x, idx, E, El, rank, M, C, 1)
    err = ep.error_word()
    r = ep.batched_prepare_ex(x.cuda(), idx.cuda(), E, El, rank, M, capacity=C, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(o["dropped"].sum()) > 0
    assert_equal("slot", np_(r["slot"]), o["slot"])
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o["tokens_per_expert"])
    assert_equal("dropped", np_(r["dropped"]), o["dropped"])


@pytest.mark.parametrize("T", [500, 40000])
def test_batched_slots_invalid_ids_are_flagged_and_skipped(T):
    K, E, El, rank, H = 4, 32, 8, 1, 8
    idx, _ = routing_inputs(T, K, E, seed=9, frac_unrouted=0.1)
    bad = idx.clone()
    bad[7, 1] = -5
    bad[T // 2, 3] = E + 3
    x = randn_bf16(T, H, seed=10)
    clean = bad.clone()
    clean[7, 1] = -1
    clean[T // 2, 3] = -1
    o = oracle.batched_prepare(x, clean, E, El, rank, T)
    err = ep.error_word()
    r = ep.batched_prepare(x.cuda(), bad.cuda(), E, El, rank, T, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERR_INVALID_EXPERT
    assert_equal("slot", np_(r["slot"]), o["slot"])
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o["tokens_per_expert"])
