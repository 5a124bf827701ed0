"""Pins of the oracle's per-expert capacity, receive alignment and send-layout
rank alignment (NeMo token_dispatcher TokenDispatcherConfig capacity factor
and pad multiple; NeMo uccl_ep.buffer Buffer.dispatch expert_alignment):
hand-worked cases, the unconstrained case reducing to the pinned prepare,
and invariants over random routing."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "capacity_align.json")))


def _rows(T, H, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return oracle.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)


def _routing(T, K, E, seed, frac=0.1):
    rng = np.random.Generator(np.random.PCG64(seed))
    idx = np.argsort(rng.random((T, E)), 1)[:, :K].astype(np.int64)
    idx[rng.random((T, K)) < frac] = -1
    return idx


def test_batched_capacity_alignment_hand_worked():
    g = GOLDEN["batched"]
    T, H = g["T"], 8
    x = np.repeat(np.arange(1, T + 1, dtype=np.uint16)[:, None], H, 1)       # row t holds the bits t+1
    idx = np.array(g["topk_idx"], np.int64)
    r = oracle.batched_prepare_ex(x, idx, g["E"], g["E_local"], g["rank"], g["M"], g["capacity"], g["alignment"],
                                  rows_init=np.full((g["E_local"], g["M"], H), 0xBEEF, np.uint16))
    assert r["err"] == 0
    assert r["slot"].tolist() == g["slot"]
    assert r["tokens_per_expert"].tolist() == g["tokens_per_expert"]
    assert r["dropped"].tolist() == g["dropped"]
    for e, toks in enumerate(g["rows_of_expert"]):
        for s, t in enumerate(toks):
            assert np.all(r["b_rows"][e, s] == t + 1)
        assert np.all(r["b_rows"][e, len(toks):g["tokens_per_expert"][e]] == 0)       # the alignment rows
        assert np.all(r["b_rows"][e, g["tokens_per_expert"][e]:] == 0xBEEF)           # untouched without zero_pad


def test_capacity_formula_hand_worked():
    g = GOLDEN["capacity_factor"]
    got = [oracle.expert_capacity(g["T"], g["K"], g["E"], f) for f in g["factors"]]
    assert got == g["capacity"]


def test_send_layout_alignment_hand_worked():
    g = GOLDEN["send_layout"]
    idx = np.array(g["topk_idx"], np.int64)
    w = np.where(idx >= 0, np.float32(0.5), np.float32(0.0)).astype(np.float32)
    c = oracle.compute_send_counts(idx, g["P"], g["E_local"])
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], g["E_local"])
    a = oracle.align_send_layout(lay, c["send_counts"], g["alignment"])
    assert a["rank_offsets"].tolist() == g["rank_offsets"]
    assert a["send_token_idx"].tolist() == g["send_token_idx"]
    assert a["send_rank"].tolist() == g["send_rank"]
    assert a["send_idx"].tolist() == g["send_idx"]
    assert a["token_pos"].tolist() == g["token_pos"]
    assert np.all(a["send_w"][np.array(g["send_token_idx"]) < 0] == 0)


@pytest.mark.parametrize("fmt", [None, 0, 1, 2])
def test_unconstrained_reduces_to_the_pinned_prepare(fmt):
    T, H, K, E, El, rank, M = 70, 512, 4, 16, 4, 2, 80
    x = _rows(T, H, 1)
    idx = _routing(T, K, E, 2)
    rs = fmt == 2
    r = oracle.batched_prepare_ex(x, idx, E, El, rank, M, None, 1, fmt, rs, zero_pad=True)
    if fmt is None:
        o = oracle.batched_prepare(x, idx, E, El, rank, M, zero_pad=True)
        assert np.array_equal(r["b_rows"], o["b_x"])
    else:
        o = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, rs, zero_pad=True)
        assert np.array_equal(r["b_rows"], o["b_q"])
        assert np.array_equal(r["b_scale"].view(np.uint32), o["b_scale"].view(np.uint32))
    assert np.array_equal(r["slot"], o["slot"])
    assert np.array_equal(r["tokens_per_expert"], o["tokens_per_expert"])
    assert np.all(r["dropped"] == 0)


@pytest.mark.parametrize("C,A", [(1, 1), (7, 1), (7, 8), (20, 16), (64, 3)])
def test_capacity_and_alignment_invariants(C, A):
    T, H, K, E, El, rank, M = 200, 128, 6, 24, 8, 1, 64
    x = _rows(T, H, 3)
    idx = _routing(T, K, E, 4, 0.2)
    r = oracle.batched_prepare_ex(x, idx, E, El, rank, M, C, A, zero_pad=False,
                                  rows_init=np.full((El, M, H), 0x7777, np.uint16))
    assert r["err"] == 0
    for el in range(El):
        e = rank * El + el
        hits = [t for t in range(T) if (idx[t] == e).any()]          # tokens naming e, ascending
        kept = hits[:C]
        assert r["dropped"][el] == len(hits) - len(kept)
        aligned = min(-(-len(kept) // A) * A, M)
        assert r["tokens_per_expert"][el] == aligned
        for s, t in enumerate(kept):
            assert np.array_equal(r["b_rows"][el, s], x[t])
            assert set(r["slot"][t][idx[t] == e].tolist()) == {s}
        for t in hits[C:]:
            assert np.all(r["slot"][t][idx[t] == e] == -1)
        assert np.all(r["b_rows"][el, len(kept):aligned] == 0)
        assert np.all(r["b_rows"][el, aligned:] == 0x7777)


@pytest.mark.parametrize("A", [1, 2, 5, 16])
def test_send_layout_alignment_invariants(A):
    T, K, P, El = 300, 4, 8, 4
    idx = _routing(T, K, P * El, 5, 0.1)
    w = np.random.Generator(np.random.PCG64(6)).random((T, K)).astype(np.float32)
    w[idx < 0] = 0
    c = oracle.compute_send_counts(idx, P, El)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], El)
    a = oracle.align_send_layout(lay, c["send_counts"], A)
    ro = a["rank_offsets"]
    assert np.all(ro % A == 0)
    assert np.all(np.diff(ro) == -(-c["send_counts"] // A) * A)
    real = a["send_token_idx"] >= 0
    assert np.array_equal(a["send_token_idx"][real], lay["send_token_idx"])      # pad rows removed
    assert np.array_equal(a["send_idx"][real], lay["send_idx"])
    assert np.array_equal(a["send_w"][real].view(np.uint32), lay["send_w"].view(np.uint32))
    assert np.all(a["send_idx"][~real] == -1) and np.all(a["send_w"][~real] == 0)
    for p in range(P):
        assert np.all(a["send_rank"][ro[p]:ro[p + 1]] == p)
    t, p = np.nonzero(a["token_pos"] >= 0)
    n = a["token_pos"][t, p]
    assert np.array_equal(a["send_token_idx"][n], t) and np.array_equal(a["send_rank"][n], p)
    assert np.array_equal(a["token_pos"] >= 0, lay["token_pos"] >= 0)
