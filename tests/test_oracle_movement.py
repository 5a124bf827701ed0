"""Pins for the oracle's data movement and reductions: dispatch, combine
(send layout), expert-batched prepare / combine, the fp8 group quantisation
and the synthetic fp8 expert.  Checked against hand-worked fixtures, closed
forms (identity experts), exact fp64 sums within the fp32-accumulation error
bound, library routines (numpy indexing / nonzero) and a cross-check between
the two layouts, which reach the same weighted sum along different routes."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0**-24          # unit roundoff of fp32


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def _f(bits):
    return oracle.bf16_bits_to_f32(bits)


def _routing(T, K, E, seed, frac_unrouted=0.1, dup=False):
    g = np.random.Generator(np.random.PCG64(seed))
    idx = (g.integers(0, E, size=(T, K)) if dup else np.argsort(g.random((T, E)), 1)[:, :K]).astype(np.int64)
    idx[g.random((T, K)) < frac_unrouted] = -1
    w = g.random((T, K)).astype(np.float32)
    w[idx < 0] = 0
    return idx, w


def _randn_bf16(shape, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return _bf16(g.standard_normal(shape, dtype=np.float32))


# ------------------------------------------------------------- send layout --
def test_hand_worked_dispatch_combine():
    g = _gold("send_layout_T4.json")
    x = _bf16(g["x"])
    recv = oracle.dispatch(x, np.array(g["send_token_idx"], np.int32))
    assert _f(recv).tolist() == g["recv_x"]
    out = oracle.combine(_bf16(g["y"]), np.array(g["token_pos"], np.int32))
    assert _f(out).tolist() == g["combined"]
    assert oracle.combine(_bf16(g["y"]), np.array(g["token_pos"], np.int32), out_f32=True).tolist() == g["combined"]


def test_dispatch_is_row_gather():
    x = _randn_bf16((300, 64), 1)
    idx, w = _routing(300, 4, 16, 2)
    r = oracle.send_path(x, idx, w, None, 4, 4)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["recv_x"], xb[r["layout"]["send_token_idx"]])


def test_combine_identity_expert_returns_input():
    # P = 1: each routed token has exactly one row; with the identity expert
    # (Y = recv_x) combine returns x on routed tokens and +0 elsewhere.
    x = _randn_bf16((500, 96), 3)
    idx, w = _routing(500, 3, 8, 4, frac_unrouted=0.5)
    r = oracle.send_path(x, idx, w, None, 1, 8)
    out = oracle.combine(r["recv_x"], r["layout"]["token_pos"])
    xb = x.view(torch.int16).numpy().view(np.uint16)
    routed = (idx >= 0).any(1)
    assert np.array_equal(out[routed], xb[routed])
    assert np.all(out[~routed] == 0)


@pytest.mark.parametrize("P", [2, 8, 16])
def test_combine_within_fp32_bound_of_exact_sum(P):
    T, H, K, E_local = 400, 128, 8, 4
    idx, w = _routing(T, K, P * E_local, 5 + P)
    c = oracle.compute_send_counts(idx, P, E_local)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], E_local)
    y = _randn_bf16((lay["n"], H), 6)
    yf = y.float().numpy().astype(np.float64)
    tp = lay["token_pos"]
    exact = np.zeros((T, H))
    absum = np.zeros((T, H))
    nterms = (tp >= 0).sum(1)
    for t in range(T):
        rows = tp[t][tp[t] >= 0]
        exact[t] = yf[rows].sum(0)
        absum[t] = np.abs(yf[rows]).sum(0)
    out32 = oracle.combine(y, tp, out_f32=True).astype(np.float64)
    bound = (np.maximum(nterms - 1, 0)[:, None] * U32 * absum) * (1 + 1e-6)
    assert np.all(np.abs(out32 - exact) <= bound)
    out16 = _f(oracle.combine(y, tp)).astype(np.float64)
    assert np.all(np.abs(out16 - exact) <= bound + 2.0**-8 * np.abs(exact) * (1 + 1e-6) + 1e-30)


def test_chunked_equals_unchunked():
    T, H, K, P, E_local, C = 1000, 64, 4, 4, 4, 3
    x = _randn_bf16((T, H), 7)
    idx, w = _routing(T, K, P * E_local, 8)
    full = oracle.send_path(x, idx, w, None, P, E_local)
    y_full = oracle.dispatch(x, full["layout"]["send_token_idx"])   # identity expert
    out_full = oracle.combine(y_full, full["layout"]["token_pos"])
    b = oracle.chunk_bounds(T, C)
    parts = []
    for i in range(C):
        s, e = int(b[i]), int(b[i + 1])
        r = oracle.send_path(x[s:e], idx[s:e], w[s:e], None, P, E_local)
        parts.append(oracle.combine(r["recv_x"], r["layout"]["token_pos"]))
    assert np.array_equal(np.concatenate(parts), out_full)


# ------------------------------------------------------------ batched layout --
def test_hand_worked_batched():
    g = _gold("batched_T4.json")
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array(g["topk_weights"], np.float32)
    x = _bf16(g["x"])
    r = oracle.batched_prepare(x, idx, g["E"], g["E_local"], g["rank"], g["M"])
    assert r["err"] == 0
    assert r["tokens_per_expert"].tolist() == g["tokens_per_expert"]
    assert r["slot"].tolist() == g["slot"]
    for e, rows in g["b_x_valid"].items():
        assert _f(r["b_x"][int(e), :len(rows)]).tolist() == rows
    y = _bf16(np.array(g["y"], dtype=np.float32))
    out = oracle.batched_combine(y, idx, w, r["slot"], g["E_local"], g["rank"])
    assert _f(out).tolist() == g["combined"]


def test_batched_prepare_matches_nonzero_listing():
    T, H, K, E, P, rank = 700, 32, 6, 24, 3, 2
    E_local = E // P
    x = _randn_bf16((T, H), 9)
    idx, _ = _routing(T, K, E, 10, dup=True)
    M = 400
    r = oracle.batched_prepare(x, idx, E, E_local, rank, M, zero_pad=True)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for el in range(E_local):
        e = rank * E_local + el
        toks = np.nonzero((idx == e).any(1))[0]          # ascending token order
        c = len(toks)
        assert r["tokens_per_expert"][el] == c
        assert np.array_equal(r["b_x"][el, :c], xb[toks])
        assert np.all(r["b_x"][el, c:] == 0)              # zero_pad
        for s, t in enumerate(toks):
            ks = np.nonzero(idx[t] == e)[0]
            assert np.all(r["slot"][t, ks] == s)
    local = (idx >= rank * E_local) & (idx < (rank + 1) * E_local)
    assert np.all(r["slot"][~local] == -1) and np.all(r["slot"][local] >= 0)


def test_batched_capacity_overflow_drops_and_flags():
    T, K, E = 50, 2, 4
    idx = np.tile(np.array([[0, 1]], np.int64), (T, 1))
    x = _randn_bf16((T, 8), 11)
    r = oracle.batched_prepare(x, idx, E, 2, 0, M=20)
    assert r["err"] & oracle.ERR_CAPACITY
    assert r["tokens_per_expert"].tolist() == [20, 20]
    assert np.all(r["slot"][:20] == np.arange(20)[:, None]) and np.all(r["slot"][20:] == -1)


def test_batched_combine_within_bound_and_skips_padding():
    T, H, K, E, rank, E_local, M = 300, 64, 8, 32, 1, 8, 200
    x = _randn_bf16((T, H), 12)
    idx, w = _routing(T, K, E, 13, frac_unrouted=0.0)
    r = oracle.batched_prepare(x, idx, E, E_local, rank, M)
    g = np.random.Generator(np.random.PCG64(14))
    y = np.full((E_local, M, H), np.nan, np.float32)
    for el, c in enumerate(r["tokens_per_expert"]):
        y[el, :c] = g.standard_normal((c, H), dtype=np.float32)
    yb = _bf16(y)
    out = _f(oracle.batched_combine(yb, idx, w, r["slot"], E_local, rank)).astype(np.float64)
    assert np.all(np.isfinite(out))          # padding (NaN) never read
    yf = yb.float().numpy().astype(np.float64)
    exact = np.zeros((T, H))
    absum = np.zeros((T, H))
    n = np.zeros(T)
    for t in range(T):
        for k in range(K):
            el = idx[t, k] - rank * E_local
            if 0 <= el < E_local:
                term = np.float64(w[t, k]) * yf[el, r["slot"][t, k]]
                exact[t] += term
                absum[t] += np.abs(term)
                n[t] += 1
    bound = (2 * n[:, None] * U32 * absum + 2.0**-8 * np.abs(exact)) * (1 + 1e-6) + 1e-30
    assert np.all(np.abs(out - exact) <= bound)


def test_send_and_batched_layouts_agree_for_one_rank():
    # With P = 1 and rank 0, both routes compute sum_k w_k * f_{e_k}(x) with
    # fp32 fma in ascending k: via the send layout (local kernel per row, then
    # combine of one row) and via the expert-batched layout.  Expert e is
    # f_e(x) = bf16(x * (1 + e/64)).
    T, H, K, E = 256, 32, 4, 8
    x = _randn_bf16((T, H), 15)
    idx, w = _routing(T, K, E, 16, frac_unrouted=0.2)
    xf = x.float().numpy()
    scale = (1.0 + np.arange(E, dtype=np.float32) / np.float32(64.0)).astype(np.float32)

    def f(e, rows):
        return _bf16(rows * scale[e]).float().numpy()

    # send layout, P = 1
    r = oracle.send_path(x, idx, w, None, 1, E)
    lay = r["layout"]
    # the local kernel's fma, emulated exactly: the product of two fp32 values
    # is exact in fp64, and so is its sum with an fp32 accumulator of this
    # magnitude, so one rounding to fp32 gives fma's result
    local = np.zeros((lay["n"], H), np.float32)
    for n in range(lay["n"]):
        acc = np.zeros(H, np.float32)
        for k in range(K):
            l = lay["send_idx"][n, k]
            if l >= 0:
                prod = np.float64(lay["send_w"][n, k]) * f(l, _f(r["recv_x"][n])).astype(np.float64)
                acc = (prod + acc.astype(np.float64)).astype(np.float32)
        local[n] = acc
    out_send = oracle.combine(_bf16(local), lay["token_pos"])

    # expert-batched layout, rank 0 of 1
    M = T
    b = oracle.batched_prepare(x, idx, E, E, 0, M)
    yb = np.zeros((E, M, H), np.float32)
    for e in range(E):
        c = b["tokens_per_expert"][e]
        yb[e, :c] = f(e, _f(b["b_x"][e, :c]))
    out_b = oracle.batched_combine(_bf16(yb), idx, w, b["slot"], E, 0)
    # both routes take the same roundings in the same order: bit for bit equal
    assert np.array_equal(out_send, out_b)


# ---------------------------------------------------------------------- fp8 --
def test_hand_worked_fp8_group_and_expert():
    g = _gold("fp8_group.json")
    H = g["H"]
    x = np.zeros((1, H), np.float32)
    head = g["x_group0_head"]
    x[0, :len(head)] = head
    q, s = oracle.quantize_fp8_rows(_bf16(x))
    assert q[0, :len(head)].tolist() == g["q_group0_head"]
    assert np.all(q[0, len(head):] == 0)
    assert s[0, 0] == np.float32(g["scale_group0"])
    assert s[0, 1] == np.float32(np.float32(1e-4) / np.float32(448.0))
    ex = g["expert"]
    out = oracle.local_expert_fp8(q, s, np.array([ex["send_idx"]], np.int64),
                                  np.array([ex["send_w"]], np.float32))
    assert _f(out[0, :2]).tolist() == ex["out_head"]


def test_fp8_group_invariants_and_error_bound():
    g = np.random.Generator(np.random.PCG64(17))
    x = g.standard_normal((64, 1024), dtype=np.float32) * np.exp(g.uniform(-8, 8, (64, 1))).astype(np.float32)
    xb = _bf16(x)
    q, s = oracle.quantize_fp8_rows(xb)
    xf = xb.float().numpy()
    d = oracle.e4m3_to_f32(q).reshape(q.shape)
    for gi in range(1024 // 128):
        cols = slice(gi * 128, (gi + 1) * 128)
        amax = np.abs(xf[:, cols]).max(1)
        # the largest element of each group lands on the largest code, 448
        assert np.all(np.abs(d[:, cols]).max(1) == 448.0)
        assert np.array_equal(s[:, gi], (np.maximum(amax, np.float32(1e-4)) / np.float32(448.0)).astype(np.float32))
        deq = d[:, cols].astype(np.float64) * s[:, gi:gi + 1]
        err = np.abs(deq - xf[:, cols])
        # 3 mantissa bits: relative error <= 2^-4 in the normal range, plus
        # half a subnormal step (2^-10 * scale) below it, plus fp32 roundings
        bound = (2.0**-4 + 1e-6) * np.abs(xf[:, cols]) + 2.0**-10 * s[:, gi:gi + 1] * 1.0001
        assert np.all(err <= bound)


def test_fp8_dispatch_rows_identical_per_token():
    x = _randn_bf16((100, 256), 18)
    idx, w = _routing(100, 4, 16, 19)
    r = oracle.send_path(x, idx, w, None, 4, 4)
    q, s = oracle.dispatch_fp8(x, r["layout"]["send_token_idx"])
    qt, st = oracle.quantize_fp8_rows(x)
    sti = r["layout"]["send_token_idx"]
    assert np.array_equal(q, qt[sti]) and np.array_equal(s, st[sti])


def test_fp8_expert_closed_form():
    # out[n] ~= sum_k w_k * x * (1 + l_k/64) within the fp8 + bf16 error bounds
    T, H, K, P, E_local = 200, 256, 8, 4, 8
    x = _randn_bf16((T, H), 20)
    idx, w = _routing(T, K, P * E_local, 21, frac_unrouted=0.0)
    r = oracle.send_path(x, idx, w, None, P, E_local)
    lay = r["layout"]
    q, s = oracle.dispatch_fp8(x, lay["send_token_idx"])
    out = _f(oracle.local_expert_fp8(q, s, lay["send_idx"], lay["send_w"])).astype(np.float64)
    xf = x.float().numpy().astype(np.float64)[lay["send_token_idx"]]
    si, sw = lay["send_idx"], lay["send_w"].astype(np.float64)
    fac = np.where(si >= 0, 1.0 + si / 64.0, 0.0)
    gain = (sw * fac).sum(1)
    want = xf * gain[:, None]
    bound = (2.0**-4 + 2.0**-7) * np.abs(want) + 2.0**-10 * np.repeat(s, 128, 1) * gain[:, None] * 1.1 + 1e-7
    assert np.all(np.abs(out - want) <= bound)
