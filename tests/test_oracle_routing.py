"""Pins for the oracle's routing metadata: compute_send_counts and
build_send_layout (axolotl integrations.expert_parallel.torch_dispatch), and
chunk_bounds.  Checked against a hand-worked example, brute force over every
tiny routing, library sorts for the special cases, and the invariants the
pages state."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from combine_send_counts_gb300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_hand_worked_send_layout():
    g = _gold("send_layout_T4.json")
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array(g["topk_weights"], np.float32)
    c = oracle.compute_send_counts(idx, g["P"], g["E_local"])
    assert c["err"] == 0
    assert c["dest"].tolist() == g["dest"]
    assert c["is_in_rank"].tolist() == g["is_in_rank"]
    assert c["send_counts"].tolist() == g["send_counts"]
    assert c["tokens_per_expert"].tolist() == g["tokens_per_expert"]
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], g["E_local"])
    assert lay["n"] == sum(g["send_counts"])
    for key in ("send_token_idx", "send_rank", "send_idx", "token_pos"):
        assert lay[key].tolist() == g[key], key
    assert lay["send_w"].tolist() == g["send_w"]
    # +0.0 (not -0.0) on slots owned elsewhere
    assert not np.any(np.signbit(lay["send_w"][lay["send_idx"] < 0]))


def _set_based_layout(idx, P, E_local):
    """The layout as the sorted list of (rank, token) pairs: a token goes once
    to every rank owning one of its experts, ordered rank-major, token-ascending."""
    pairs = set()
    for t, row in enumerate(idx.tolist()):
        for e in row:
            if e >= 0:
                pairs.add((e // E_local, t))
    return sorted(pairs)


@pytest.mark.parametrize("P,E_local", [(1, 4), (2, 2), (4, 1)])
def test_brute_force_all_tiny_routings(P, E_local):
    E = P * E_local
    ids = list(range(-1, E))
    for T, K in ((1, 1), (2, 2), (3, 1), (1, 2)):
        for flat in itertools.product(ids, repeat=T * K):
            idx = np.array(flat, np.int64).reshape(T, K)
            w = (np.arange(T * K, dtype=np.float32).reshape(T, K) + 1) / 8
            c = oracle.compute_send_counts(idx, P, E_local)
            lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], E_local)
            want = _set_based_layout(idx, P, E_local)
            got = list(zip(lay["send_rank"].tolist(), lay["send_token_idx"].tolist()))
            assert got == want, (idx.tolist(), got, want)
            assert c["send_counts"].tolist() == [sum(1 for p, _ in want if p == r) for r in range(P)]
            for n, (p, t) in enumerate(want):
                for k in range(K):
                    e = int(idx[t, k])
                    owned = e >= 0 and e // E_local == p
                    assert lay["send_idx"][n, k] == (e - p * E_local if owned else -1)
                    assert lay["send_w"][n, k] == (w[t, k] if owned else 0.0)
            tpe = [len({t for t in range(T) if e in idx[t].tolist()}) for e in range(E)]
            assert c["tokens_per_expert"].tolist() == tpe


def _random_routing(T, K, E, seed, frac_unrouted=0.1, allow_dup=False):
    g = np.random.Generator(np.random.PCG64(seed))
    if allow_dup:
        idx = g.integers(0, E, size=(T, K))
    else:
        idx = np.argsort(g.random((T, E)), axis=1)[:, :K]
    idx = idx.astype(np.int64)
    idx[g.random((T, K)) < frac_unrouted] = -1
    w = g.random((T, K)).astype(np.float32)
    return idx, w


@pytest.mark.parametrize("T,K,P,E_local,dup", [(1000, 8, 8, 4, False), (777, 3, 5, 3, True),
                                               (513, 1, 16, 2, False), (300, 6, 1, 7, True)])
def test_layout_invariants(T, K, P, E_local, dup):
    idx, w = _random_routing(T, K, P * E_local, seed=T, allow_dup=dup)
    c = oracle.compute_send_counts(idx, P, E_local)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], E_local)
    N = lay["n"]
    sti, sr, si, sw, tp = (lay[k] for k in ("send_token_idx", "send_rank", "send_idx", "send_w", "token_pos"))
    # num_send == is_in_rank.sum() == sum(send_counts)
    assert N == int(c["is_in_rank"].sum()) == int(c["send_counts"].sum())
    # rank-major, token-ascending
    assert np.all(np.diff(sr) >= 0)
    same = sr[1:] == sr[:-1]
    assert np.all(np.diff(sti)[same] > 0)
    # each (t, p) with is_in_rank appears exactly once; token_pos is the inverse map
    assert np.array_equal(tp[sti, sr], np.arange(N))
    assert int((tp >= 0).sum()) == N
    assert np.array_equal(tp >= 0, c["is_in_rank"].astype(bool))
    # owned slots carry the local id and the weight; others -1 and +0.0
    owned = si >= 0
    assert np.array_equal(si[owned] + (sr[:, None] * E_local).repeat(K, 1)[owned], idx[sti][owned])
    assert np.array_equal(sw[owned], w[sti][owned])
    assert np.all(sw[~owned] == 0) and not np.any(np.signbit(sw[~owned]))
    assert np.array_equal(owned, (idx[sti] >= 0) & (idx[sti] // E_local == sr[:, None]))


def test_k1_is_stable_counting_sort():
    idx, w = _random_routing(5000, 1, 32, seed=7, frac_unrouted=0.2)
    P, E_local = 8, 4
    c = oracle.compute_send_counts(idx, P, E_local)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], E_local)
    rank = np.where(idx[:, 0] >= 0, idx[:, 0] // E_local, -1)
    routed = np.nonzero(rank >= 0)[0]
    order = routed[np.argsort(rank[routed], kind="stable")]
    assert np.array_equal(lay["send_token_idx"], order)


def test_p1_is_routed_tokens_in_order():
    idx, w = _random_routing(4000, 4, 16, seed=9, frac_unrouted=0.6)
    c = oracle.compute_send_counts(idx, 1, 16)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], 16)
    assert np.array_equal(lay["send_token_idx"], np.nonzero((idx >= 0).any(1))[0])


def test_layout_is_lexsort_of_rank_token_pairs():
    idx, w = _random_routing(3000, 8, 64, seed=11, frac_unrouted=0.05)
    P, E_local = 8, 8
    c = oracle.compute_send_counts(idx, P, E_local)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], E_local)
    t, p = np.nonzero(c["is_in_rank"])
    order = np.lexsort((t, p))
    assert np.array_equal(lay["send_token_idx"], t[order])
    assert np.array_equal(lay["send_rank"], p[order])


def test_tokens_per_expert_counts_tokens_once():
    idx, _ = _random_routing(2000, 6, 12, seed=3, allow_dup=True)
    c = oracle.compute_send_counts(idx, 3, 4)
    pairs = {(t, int(e)) for t in range(idx.shape[0]) for e in idx[t] if e >= 0}
    want = np.bincount(np.array([e for _, e in pairs]), minlength=12)
    assert np.array_equal(c["tokens_per_expert"], want)


def test_invalid_expert_ids_flagged_and_treated_unrouted():
    idx = np.array([[0, 5], [-2, 1], [3, -1]], np.int64)   # E = 4: 5 and -2 invalid
    c = oracle.compute_send_counts(idx, 2, 2)
    assert c["err"] & oracle.ERR_INVALID_EXPERT
    assert c["dest"].tolist() == [[0, -1], [-1, 0], [1, -1]]
    assert c["send_counts"].tolist() == [2, 1]


def test_chunk_bounds_remainder_rule():
    for case in _gold("chunk_bounds.json")["cases"]:
        assert oracle.chunk_bounds(case["T"], case["C"]).tolist() == case["bounds"]


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_workload_recipe_counts(name):
    w = wl.WORKLOADS[name]
    idx, wts = wl.routing(w)
    assert idx.shape == (w.T, w.K) and wts.dtype.is_floating_point
    i = idx.numpy()
    routed = i >= 0
    # K distinct experts per token among routed slots
    for row, r in zip(i[:200], routed[:200]):
        assert len(set(row[r].tolist())) == int(r.sum())
    if w.unrouted_frac:
        assert int((~routed).sum()) == int(np.floor(w.unrouted_frac * w.T * w.K))
    ws = wts.numpy()
    assert np.all(ws[~routed] == 0)
    s = ws.sum(1)
    assert np.allclose(s[routed.any(1)], 1.0, atol=1e-5)
