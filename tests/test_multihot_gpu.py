"""GPU parity of the top-k -> multihot conversion (NeMo token_dispatcher
_DeepepManager / _HybridEPManager._indices_to_multihot) with the oracle, bit
for bit: the routing map and the dense fp32 probabilities."""
import json
import os

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl
from _paths import assert_equal, np_, routing_inputs

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "multihot.json")))


def _check(idx, p, E, err_want=0):
    o = oracle.indices_to_multihot(idx, p, E)
    err = ep.error_word()
    rm, pr = ep.indices_to_multihot(idx.cuda(), p.cuda(), E, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == err_want == o["err"]
    assert_equal("routing_map", np_(rm).astype(np.uint8), o["routing_map"])
    assert_equal("probs (bits)", np_(pr).view(np.uint32), o["probs"].view(np.uint32))


def test_hand_worked():
    idx = torch.tensor(GOLDEN["topk_idx"], dtype=torch.int64)
    p = torch.tensor(GOLDEN["topk_probs"], dtype=torch.float32)
    rm, pr = ep.indices_to_multihot(idx.cuda(), p.cuda(), GOLDEN["E"])
    torch.cuda.synchronize()
    assert np_(rm).astype(int).tolist() == GOLDEN["routing_map"]
    assert np_(pr).tolist() == GOLDEN["probs"]


@pytest.mark.parametrize("name", ["tiny", "mid", "large"])
def test_workloads(name):
    w = wl.WORKLOADS[name]
    idx, p = wl.routing(w)
    _check(idx, p, w.E)


@pytest.mark.parametrize("T,K,E,dup", [(1, 1, 1, False), (333, 3, 5, True), (1000, 8, 13, False),
                                       (777, 32, 64, True), (4096, 6, 8, True), (50, 4, 8192, False)])
def test_shapes_and_duplicates(T, K, E, dup):
    idx, p = routing_inputs(T, K, E, T + E, 0.2, dup=dup)
    _check(idx, p, E)


def test_invalid_ids_are_flagged_and_ignored():
    idx, p = routing_inputs(400, 6, 32, 3, 0.1)
    idx[5, 2] = 32
    idx[9, 0] = -7
    _check(idx, p, 32, ep.EP_ERR_INVALID_EXPERT)


def test_map_only_probs_only_unaligned_and_empty():
    T, K, E = 300, 4, 16
    idx, p = routing_inputs(T, K, E, 4, 0.1)
    o = oracle.indices_to_multihot(idx, p, E)
    dev = "cuda"
    err = ep.error_word()
    rm = torch.empty((T, E), dtype=torch.uint8, device=dev)
    ep.ep_indices_to_multihot(idx.cuda(), None, T, K, E, rm, None, err)
    # probs into a buffer offset by 4 bytes: not 16-byte aligned (element-wise stores)
    buf = torch.empty(T * E + 1, dtype=torch.float32, device=dev)
    pr = buf[1:]
    ep.ep_indices_to_multihot(idx.cuda(), p.cuda(), T, K, E, None, pr, err)
    ep.ep_indices_to_multihot(idx[:0].cuda(), p[:0].cuda(), 0, K, E, rm, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_equal("map only", np_(rm), o["routing_map"])
    assert_equal("probs only, unaligned", np_(pr).reshape(T, E).view(np.uint32), o["probs"].view(np.uint32))
