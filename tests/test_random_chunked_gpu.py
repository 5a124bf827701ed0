"""Seeded random shapes through the chunked drivers (axolotl torch_dispatch,
chunk_bounds and dispatch_chunked_forward: one count pass for all chunks, then
per chunk layout -> dispatch -> local kernel -> combine), host-sync and
without host sync (one and two row sets), against the oracle run chunk by
chunk.  Cases include more chunks than tokens (empty leading chunks), one
chunk, bf16 rows with an identity expert and fp8 rows with the synthetic fp8
expert; every output element bit for bit."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_combine_parity, assert_equal, bits16, randn_bf16, routing_inputs

pytestmark = pytest.mark.gpu

N_CASES = 64


def _draw(i):
    g = np.random.Generator(np.random.PCG64(8000 + i))
    while True:
        P = int(g.choice([1, 2, 4, 8, 16, 32]))
        El = int(g.choice([1, 4, 8, 32, 64]))
        if P * El > 4096:
            continue
        dup = bool(g.random() < 0.25)
        K = int(g.integers(1, min(16, P * El if not dup else 16) + 1))
        fp8 = bool(g.random() < 0.5)
        H = int(g.integers(1, 17)) * 128 if fp8 else int(g.integers(1, 257)) * 8
        chunks = int(g.integers(1, 9))
        T = int(np.exp(g.uniform(0, np.log(5000))))
        T = max(1, min(T, 30_000_000 // (H * min(K, P))))
        return dict(P=P, El=El, K=K, H=H, T=T, chunks=chunks, dup=dup, fp8=fp8,
                    frac=float(g.choice([0.0, 0.1, 0.5])), seed=8000 + i)


CASES = [_draw(i) for i in range(N_CASES)]


def _oracle_chunked(x, idx, w, P, El, chunks, fp8):
    b = oracle.chunk_bounds(x.shape[0], chunks)
    H = x.shape[1]
    outs = []
    for i in range(chunks):
        s, e = int(b[i]), int(b[i + 1])
        if e == s:
            continue
        r = oracle.send_path(x[s:e], idx[s:e], w[s:e], None, P, El)
        lay = r["layout"]
        if fp8:
            q, sc = oracle.dispatch_fp8(x[s:e], lay["send_token_idx"])
            local = oracle.local_expert_fp8(q, sc, lay["send_idx"], lay["send_w"])
        else:
            local = r["recv_x"]                       # identity expert
        outs.append(oracle.combine(local, lay["token_pos"]))
    return np.concatenate(outs) if outs else np.zeros((0, H), np.uint16)


def _id(c):
    return "T{T}-C{chunks}-H{H}-K{K}-P{P}-El{El}{d}{f}".format(d="-dup" if c["dup"] else "",
                                                                f="-fp8" if c["fp8"] else "", **c)


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_random_chunked_drivers_match_oracle(c):
    P, El, K, H, T, C = c["P"], c["El"], c["K"], c["H"], c["T"], c["chunks"]
    idx, w = routing_inputs(T, K, P * El, c["seed"], c["frac"], dup=c["dup"])
    x = randn_bf16(T, H, c["seed"] + 1)
    want = _oracle_chunked(x, idx, w, P, El, C, c["fp8"])
    xd, idd, wd = x.cuda(), idx.cuda(), w.cuda()
    err = ep.error_word()

    def identity(chunk, recv_x, recv_scale, send_idx, send_w, local_out, *n_rows):
        local_out.copy_(recv_x)

    lk = None if c["fp8"] else identity
    out = ep.dispatch_chunked_forward(xd, idd, wd, num_local_experts=El, num_ranks=P, chunks=C, fp8=c["fp8"],
                                      local_kernel=lk, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_combine_parity("host-sync driver", bits16(out), want)
    for n_sets in (1, 2):
        out2 = ep.dispatch_chunked_forward_nosync(xd, idd, wd, num_local_experts=El, num_ranks=P, chunks=C,
                                                  fp8=c["fp8"], local_kernel=lk, n_sets=n_sets, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_equal(f"no-sync driver, {n_sets} row set(s)", bits16(out2), bits16(out))
