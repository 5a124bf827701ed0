"""Row movement past 2^32 bytes: a receive buffer and an expert-batched buffer
of about 5 GB each, so that the rows at their ends sit at byte offsets no
32-bit index reaches.  Counts, layouts and slots are compared with the oracle
in full (integer work, cheap on the host); rows and combined outputs on
sampled tokens, always including the tokens whose rows lie at the highest
offsets.  Each token's moved rows and combined output depend only on its own
row, routing and weights, so a sampled token is checked against the oracle on
the one-token problem."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_combine_parity, assert_equal, bits16, np_, randn_bf16, routing_inputs

pytestmark = pytest.mark.gpu

GIB4 = 1 << 32


def _sample(T, last, n=64, seed=5):
    g = np.random.Generator(np.random.PCG64(seed))
    s = set(g.choice(T, size=n, replace=False).tolist()) | set(last)
    return sorted(s)


def test_send_path_rows_past_4_gib():
    T, H, K, P, El = 65536, 8192, 8, 8, 8
    idx, wts = routing_inputs(T, K, P * El, 4242, 0.05)
    x = randn_bf16(T, H, 4243)
    oc = oracle.compute_send_counts(idx, P, El, with_tokens_per_expert=False)
    ol = oracle.build_send_layout(idx, wts, oc["dest"], oc["is_in_rank"], El)
    N = int(ol["n"])
    assert N * H * 2 > GIB4 + (64 << 20), "the receive buffer must reach past 4 GiB"
    dev = "cuda"
    xd, idd, wd = x.to(dev), idx.to(dev), wts.to(dev)
    err = ep.error_word()
    c = ep.compute_send_counts(idd, P, El, err=err, with_tokens_per_expert=False)
    lay = ep.build_send_layout(idd, wd, c["dest"], c["is_in_rank"], N, El, err=err)
    recv = ep.dispatch_rows(xd, lay["token_pos"], N, err=err)
    out = ep.combine_rows(recv, lay["token_pos"], err=err)   # identity expert
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
    assert_equal("send_counts", np_(c["send_counts"]).reshape(-1), oc["send_counts"])
    assert_equal("token_pos", np_(lay["token_pos"]), ol["token_pos"])
    assert_equal("send_token_idx", np_(lay["send_token_idx"]), ol["send_token_idx"])
    # the last tokens of every rank segment sit at its highest rows
    tp = ol["token_pos"]
    last = []
    for p in range(P):
        ts = np.nonzero(tp[:, p] >= 0)[0]
        last += ts[-3:].tolist()
    sample = _sample(T, last)
    rows_hi = [int(tp[t, p]) for t in last for p in range(P) if tp[t, p] >= 0]
    assert max(rows_hi) * H * 2 > GIB4
    outb = bits16(out)
    for t in sample:
        r = oracle.send_path(x[t:t + 1], idx[t:t + 1], wts[t:t + 1], None, P, El)
        rows = [int(v) for v in tp[t] if v >= 0]
        got = bits16(recv[torch.tensor(rows, device=dev)]) if rows else np.zeros((0, H), np.uint16)
        assert_equal(f"recv rows of token {t}", got, r["recv_x"])
        want = oracle.combine(r["recv_x"], r["layout"]["token_pos"])
        assert_combine_parity(f"combine of token {t}", outb[t:t + 1], want)


def test_batched_rows_past_4_gib():
    T, H, K, E, El, rank, M = 16384, 4096, 8, 128, 32, 1, 20000
    assert El * M * H * 2 > GIB4 + (256 << 20)
    idx, wts = routing_inputs(T, K, E, 777, 0.05)
    x = randn_bf16(T, H, 778)
    # slots and counts from the oracle on 8-column rows (they do not depend on H)
    o8 = oracle.batched_prepare(torch.zeros((T, 8), dtype=torch.bfloat16), idx, E, El, rank, M)
    dev = "cuda"
    xd, idd, wd = x.to(dev), idx.to(dev), wts.to(dev)
    err = ep.error_word()
    r = ep.batched_prepare(xd, idd, E, El, rank, M, err=err)
    out = ep.batched_combine(r["b_x"], idd, wd, r["slot"], rank, err=err)   # identity expert
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o8["tokens_per_expert"])
    assert_equal("slot", np_(r["slot"]), o8["slot"])
    slot = o8["slot"]
    # tokens holding the highest slots of the last local experts: their rows
    # sit past 4 GiB in the batched buffer
    e0 = rank * El
    last = []
    for el in range(El - 3, El):
        hit = np.nonzero((idx.numpy() == e0 + el).any(1))[0]
        last += hit[-3:].tolist()
    sample = _sample(T, last, seed=6)
    hi = max((int(idx[t, k]) - e0) * M + int(slot[t, k]) for t in last for k in range(K)
             if 0 <= int(idx[t, k]) - e0 < El)
    assert hi * H * 2 > GIB4
    outb = bits16(out)
    b_x = r["b_x"]
    for t in sample:
        it, wt = idx[t:t + 1], wts[t:t + 1]
        one = oracle.batched_prepare(x[t:t + 1], it, E, El, rank, 1)
        for k in range(K):
            el = int(it[0, k]) - e0
            if 0 <= el < El:
                s = int(slot[t, k])
                assert_equal(f"b_x row of token {t}, expert {el}", bits16(b_x[el, s:s + 1]), one["b_x"][el, :1])
        want = oracle.batched_combine(one["b_x"], it, wt, one["slot"], El, rank)
        assert_combine_parity(f"batched combine of token {t}", outb[t:t + 1], want)
