"""GPU parity of the expert-batched prepare with a per-expert capacity and a
receive alignment (NeMo token_dispatcher TokenDispatcherConfig capacity
factor and pad multiple; NeMo uccl_ep.buffer Buffer.dispatch
expert_alignment) against the oracle, bit for bit, including the rows the
call must leave untouched."""
import json
import os

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl
from _paths import assert_combine_parity, assert_equal, bits16, np_, randn_bf16, routing_inputs

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "capacity_align.json")))


def _run(x, idx, E, El, rank, M, C, A, fmt, rs, zero_pad):
    """Both sides on buffers pre-filled with the same pattern."""
    T, H = x.shape
    K = idx.shape[1]
    dev = "cuda"
    fp8 = fmt is not None
    row_dt = np.uint8 if fp8 else np.uint16
    rows0 = np.full((El, M, H), 0xA5 if fp8 else 0x7E57, row_dt)
    s0 = None
    if fp8:
        shape, dt = oracle.batched_scale_shape(El, M, H, fmt)
        s0 = np.full(shape, 0x7F7F7F7F if dt == np.int32 else np.nan, dt)
    # capacity 0 is the library's "max_num_tokens, overflow reported"
    o = oracle.batched_prepare_ex(x, idx, E, El, rank, M, C if C > 0 else M, A, fmt, rs, zero_pad, rows0, s0)
    g_rows = torch.from_numpy(rows0.view(np.int16) if not fp8 else rows0).to(dev)
    g_s = torch.from_numpy(s0).to(dev) if fp8 else None
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    dropped = torch.empty(El, dtype=torch.int32, device=dev)
    err = ep.error_word()
    ep.ep_batched_prepare_ex(x.to(dev), idx.to(dev), T, K, H, E, El, rank, M, C, A, g_rows, g_s,
                             -1 if not fp8 else fmt, int(rs), tpe, slot, dropped, int(zero_pad),
                             ep.workspace(T, K, E // El, El), err)
    torch.cuda.synchronize()
    return o, dict(b_rows=g_rows, b_scale=g_s, tokens_per_expert=tpe, slot=slot, dropped=dropped, err=err)


def _compare(o, g, fp8):
    assert_equal("tokens_per_expert", np_(g["tokens_per_expert"]), o["tokens_per_expert"])
    assert_equal("dropped", np_(g["dropped"]), o["dropped"])
    assert_equal("slot", np_(g["slot"]), o["slot"])
    rows = np_(g["b_rows"])
    assert_equal("rows", rows if fp8 else rows.view(np.uint16), o["b_rows"])
    if fp8:
        assert_equal("scales (bits)", np_(g["b_scale"]).view(np.uint32), o["b_scale"].view(np.uint32))


CASES = [
    # capacity, alignment, scale layout (None: bf16), round_scale, zero_pad
    (0, 1, None, False, False),
    (37, 1, None, False, False),
    (37, 16, None, False, False),
    (100, 8, None, False, True),
    (1, 4, None, False, False),
    (50, 8, 1, False, False),
    (50, 32, 2, True, True),
    (64, 5, 0, True, False),
]


@pytest.mark.parametrize("C,A,fmt,rs,zero_pad", CASES)
def test_capacity_alignment_matches_oracle(C, A, fmt, rs, zero_pad):
    T, H, K, E, El, rank, M = 1200, 512, 6, 40, 10, 3, 160
    idx, _ = routing_inputs(T, K, E, 41 + C + A, 0.1)
    x = randn_bf16(T, H, 42)
    o, g = _run(x, idx, E, El, rank, M, C, A, fmt, rs, zero_pad)
    assert o["err"] == 0
    overflow = C == 0 and int(o["dropped"].sum()) > 0          # reported only without a capacity
    assert int(g["err"].item()) == (ep.EP_ERR_CAPACITY if overflow else 0)
    _compare(o, g, fmt is not None)


def test_capacity_hand_worked():
    gd = GOLDEN["batched"]
    T, H = gd["T"], 64
    x = torch.from_numpy(np.repeat(np.arange(1, T + 1, dtype=np.int16)[:, None], H, 1)).view(torch.bfloat16)
    idx = torch.tensor(gd["topk_idx"], dtype=torch.int64)
    o, g = _run(x, idx, gd["E"], gd["E_local"], gd["rank"], gd["M"], gd["capacity"], gd["alignment"], None, False,
                False)
    assert np_(g["slot"]).tolist() == gd["slot"]
    assert np_(g["tokens_per_expert"]).tolist() == gd["tokens_per_expert"]
    assert np_(g["dropped"]).tolist() == gd["dropped"]
    _compare(o, g, False)


def test_capacity_factor_on_the_batched_workload_then_combine():
    w = wl.WORKLOADS["batched"]
    x, idx, wts = wl.make(w)
    C = ep.expert_capacity(w.T, w.K, w.E, 1.0)
    assert C == oracle.expert_capacity(w.T, w.K, w.E, 1.0) == -(-w.T * w.K // w.E)
    r = ep.batched_prepare_ex(x.cuda(), idx.cuda(), w.E, w.E_local, w.rank, w.max_num_tokens, capacity=C,
                              alignment=128)
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    o = oracle.batched_prepare_ex(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, C, 128)
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o["tokens_per_expert"])
    assert_equal("dropped", np_(r["dropped"]), o["dropped"])
    assert int(o["dropped"].sum()) > 0                     # the factor does drop tokens here
    assert_equal("slot", np_(r["slot"]), o["slot"])
    rows = bits16(r["b_rows"])
    for e in range(w.E_local):
        n = int(o["tokens_per_expert"][e])
        assert_equal(f"rows e={e}", rows[e, :n], o["b_rows"][e, :n])
    # the dropped slots are -1, so the weighted combine leaves those experts out
    y = wl.batched_expert_outputs(w, o["tokens_per_expert"])
    want = oracle.batched_combine(y, idx, wts, o["slot"], w.E_local, w.rank)
    got = ep.batched_combine(y.cuda(), idx.cuda(), wts.cuda(), r["slot"], w.rank)
    torch.cuda.synchronize()
    assert_combine_parity("combine after drops", bits16(got), want)


def test_capacity_host_checks():
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    for kw in (dict(capacity=9), dict(capacity=-1), dict(alignment=0)):
        with pytest.raises(ep.EPError):
            ep.batched_prepare_ex(x, idx, 4, 4, 0, 8, **kw)
    with pytest.raises(ep.EPError):
        ep.expert_capacity(8, 2, 4, 0.0)


# ------------------------------------------------ aligned send layout (route) --
# 1M tokens cannot be resident in one cooperative grid, so that case runs the
# two-launch fallback (count_kernel + layout_write_kernel).
@pytest.mark.parametrize("T,K,P,El,A", [(1500, 8, 8, 4, 16), (777, 6, 16, 2, 3), (300, 32, 64, 1, 8),
                                        (5000, 8, 8, 4, 1), (1000000, 2, 4, 8, 128)])
def test_route_aligned_matches_oracle(T, K, P, El, A):
    idx, w = routing_inputs(T, K, P * El, 50 + A, 0.1)
    H = 64
    x = randn_bf16(T, H, 51)
    r = ep.route_nosync(idx.cuda(), w.cuda(), P, El, alignment=A)
    W = r["num_worst_rows"]
    recv = ep.dispatch_rows(x.cuda(), r["token_pos"], W, err=r["err"])
    out = ep.combine_rows(recv, r["token_pos"], err=r["err"])
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    c = oracle.compute_send_counts(idx, P, El)
    lay = oracle.build_send_layout(idx, w, c["dest"], c["is_in_rank"], El)
    a = oracle.align_send_layout(lay, c["send_counts"], A)
    n = a["n"]
    assert_equal("dest", np_(r["dest"]), c["dest"])
    assert_equal("is_in_rank", np_(r["is_in_rank"]), c["is_in_rank"])
    assert_equal("send_counts", np_(r["send_counts"]), c["send_counts"])
    assert_equal("rank_offsets", np_(r["rank_offsets"]), a["rank_offsets"])
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), -(-c["tokens_per_expert"] // A) * A)
    for k in ("send_token_idx", "send_rank", "send_idx"):
        assert_equal(k, np_(r[k])[:n], a[k])
    assert_equal("send_w (bits)", np_(r["send_w"])[:n].view(np.uint32), a["send_w"].view(np.uint32))
    assert_equal("token_pos", np_(r["token_pos"]), a["token_pos"])
    real = a["send_token_idx"] >= 0
    assert_equal("recv_x (real rows)", bits16(recv)[:n][real], oracle.dispatch(x, lay["send_token_idx"]))
    assert_combine_parity("combine", bits16(out), oracle.combine(oracle.dispatch(x, lay["send_token_idx"]),
                                                                 lay["token_pos"]))


def test_route_aligned_capacity_is_flagged():
    T, K, P, El, A = 900, 8, 8, 4, 64
    idx, w = routing_inputs(T, K, P * El, 52, 0.0)
    c = oracle.compute_send_counts(idx, P, El)
    need = int(sum(-(-int(v) // A) * A for v in c["send_counts"]))
    r = ep.route_nosync(idx.cuda(), w.cuda(), P, El, alignment=A, num_worst_rows=need - A)
    torch.cuda.synchronize()
    assert int(r["err"].item()) & ep.EP_ERR_CAPACITY
    assert int(r["rank_offsets"][P].item()) == need
    assert int(r["token_pos"].max().item()) < need - A


@pytest.mark.parametrize("fmt,rs,C,A", [(None, False, 0, 1), (1, False, 0, 1), (2, True, 30, 8), (None, False, 25, 4)])
def test_repeated_expert_ids_write_one_row(fmt, rs, C, A):
    # tokens naming one local expert in several slots: one row per (expert,
    # token), every such slot gets the same slot value; several tokens per
    # block (short rows), so the row-list dedup spans a block's tokens
    T, H, K, E, El, rank, M = 700, 512, 6, 12, 4, 1, 300
    idx, _ = routing_inputs(T, K, E, 61, 0.1, dup=True)
    x = randn_bf16(T, H, 62)
    o, g = _run(x, idx, E, El, rank, M, C, A, fmt, rs, True)
    assert o["err"] == 0
    overflow = C == 0 and int(o["dropped"].sum()) > 0
    assert int(g["err"].item()) == (ep.EP_ERR_CAPACITY if overflow else 0)
    _compare(o, g, fmt is not None)
