"""Pins of the oracle's top-k -> multihot conversion (NeMo token_dispatcher
_DeepepManager / _HybridEPManager._indices_to_multihot): a hand-worked case,
numpy's scatter-add over the same slots, and invariants."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "multihot.json")))


def test_hand_worked():
    r = oracle.indices_to_multihot(np.array(GOLDEN["topk_idx"]), np.array(GOLDEN["topk_probs"], np.float32),
                                   GOLDEN["E"])
    assert r["err"] == 0
    assert r["routing_map"].tolist() == GOLDEN["routing_map"]
    assert r["probs"].tolist() == GOLDEN["probs"]


@pytest.mark.parametrize("dup", [False, True])
def test_matches_numpy_scatter_add(dup):
    rng = np.random.Generator(np.random.PCG64(7 + dup))
    T, K, E = 500, 8, 64
    idx = (rng.integers(0, E, size=(T, K)) if dup else np.argsort(rng.random((T, E)), 1)[:, :K]).astype(np.int64)
    idx[rng.random((T, K)) < 0.2] = -1
    p = rng.random((T, K)).astype(np.float32)
    r = oracle.indices_to_multihot(idx, p, E)
    want_p = np.zeros((T, E), np.float32)
    want_m = np.zeros((T, E), np.uint8)
    t, k = np.nonzero(idx >= 0)
    np.add.at(want_p, (t, idx[t, k]), p[t, k])       # processes (t, k) in row-major order: ascending k
    want_m[t, idx[t, k]] = 1
    assert np.array_equal(r["routing_map"], want_m)
    assert np.array_equal(r["probs"].view(np.uint32), want_p.view(np.uint32))


def test_invariants_and_invalid_ids():
    rng = np.random.Generator(np.random.PCG64(9))
    T, K, E = 300, 6, 40
    idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)
    p = rng.random((T, K)).astype(np.float32)
    r = oracle.indices_to_multihot(idx, p, E)
    assert r["err"] == 0
    distinct = np.array([len(set(row[row >= 0].tolist())) for row in idx])
    assert np.array_equal(r["routing_map"].sum(1), distinct)
    assert np.all(r["probs"][r["routing_map"] == 0] == 0)
    assert np.allclose(r["probs"].sum(1, dtype=np.float64), np.where(idx >= 0, p, 0).sum(1, dtype=np.float64),
                       rtol=1e-5)
    bad = idx.copy()
    bad[3, 2] = E
    bad[7, 0] = -5
    rb = oracle.indices_to_multihot(bad, p, E)
    assert rb["err"] == oracle.ERR_INVALID_EXPERT
    keep = np.ones_like(bad, bool)
    keep[3, 2] = keep[7, 0] = False
    ok = oracle.indices_to_multihot(np.where(keep, bad, -1), p, E)
    assert np.array_equal(rb["routing_map"], ok["routing_map"]) and np.array_equal(rb["probs"], ok["probs"])
