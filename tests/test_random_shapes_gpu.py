"""Seeded random shapes through every entry point, against the oracle: counts,
send layout, dispatch and combine (axolotl torch_dispatch; the host-sync and
no-sync call orders, bf16 and fp8 payloads of NeMo uccl_ep.buffer
Buffer.dispatch), the expert-batched prepare and weighted combine (vLLM
BatchedPrepareAndFinalize, bf16 and every fp8 scale layout), and the multihot
map (NeMo token_dispatcher _indices_to_multihot), with capacity drops and
receive alignment on both layouts (NeMo token_dispatcher capacity factor and
pad multiple, uccl_ep.buffer expert_alignment).

Each case draws P, E_local, K, T, H, the share of unrouted slots and
whether ids repeat within a token, so that the kernels' template forms
(unrolled and generic K, row geometries, one- or two-word expert masks,
cluster or grid-wide slot kernels) meet shapes the named workloads do not.
Every output is compared element by element, bit for bit."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import (assert_combine_parity, assert_equal, bits16, compare_send_path, gpu_send_path, np_,
                    randn_bf16, routing_inputs)

pytestmark = pytest.mark.gpu

N_CASES = 120
CAP = 100_000_000   # elements of the largest buffer a case may need (oracle time and host memory)


def _draw(i):
    g = np.random.Generator(np.random.PCG64(7000 + i))
    while True:
        P = int(g.choice([1, 2, 3, 4, 6, 8, 13, 16, 32, 64]))
        El = int(g.choice([1, 2, 5, 8, 16, 32, 48, 64, 96, 128]))
        E = P * El
        if E > 8192:
            continue
        dup = bool(g.random() < 0.25)
        K = int(g.integers(1, min(32, E if not dup else 32) + 1))
        fp8 = bool(g.random() < 0.5)
        H = int(g.integers(1, 33)) * 128 if fp8 else int(g.integers(1, 376)) * 8
        T = int(np.exp(g.uniform(0, np.log(20000))))
        T = max(1, min(T, CAP // max(1, H * min(K, P)), CAP // max(1, El * H)))
        frac = float(g.choice([0.0, 0.05, 0.3, 0.9]))
        rank = int(g.integers(0, P))
        return dict(P=P, El=El, E=E, K=K, H=H, T=T, dup=dup, fp8=fp8, frac=frac, rank=rank, seed=7000 + i)


def _draw_large(i):
    # many tokens (past one thread-block cluster's 32 768 for some), moderate rows
    g = np.random.Generator(np.random.PCG64(9000 + i))
    P = int(g.choice([2, 4, 8, 16]))
    El = int(g.choice([4, 8, 16, 32]))
    dup = bool(g.random() < 0.25)
    K = int(g.integers(1, min(8, P * El) + 1))
    fp8 = bool(g.random() < 0.5)
    H = int(g.choice([128, 256, 512, 1024])) if fp8 else int(g.integers(1, 129)) * 8
    T = int(g.integers(8000, 60001))
    T = max(1, min(T, CAP // max(1, H * min(K, P)), CAP // max(1, El * H)))
    return dict(P=P, El=El, E=P * El, K=K, H=H, T=T, dup=dup, fp8=fp8, frac=float(g.choice([0.0, 0.05, 0.3])),
                rank=int(g.integers(0, P)), seed=9000 + i)


CASES = [_draw(i) for i in range(N_CASES)] + [_draw_large(i) for i in range(16)] + [
    # past the one-cluster slot kernel's 32 768 tokens (the grid-wide slot kernels)
    dict(P=4, El=8, E=32, K=4, H=128, T=50000, dup=False, fp8=True, frac=0.05, rank=1, seed=9100),
    dict(P=8, El=16, E=128, K=6, H=96, T=45000, dup=True, fp8=False, frac=0.3, rank=5, seed=9101),
]


def _id(c):
    return "T{T}-H{H}-K{K}-P{P}-El{El}{d}{f}-u{frac}".format(d="-dup" if c["dup"] else "", f="-fp8" if c["fp8"] else "",
                                                             **c)


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_random_shape_matches_oracle(c):
    P, El, E, K, H, T, rank = c["P"], c["El"], c["E"], c["K"], c["H"], c["T"], c["rank"]
    idx, w = routing_inputs(T, K, E, c["seed"], c["frac"], dup=c["dup"])
    x = randn_bf16(T, H, c["seed"] + 1)
    dev = "cuda"

    # send layout, host-sync order
    o = oracle.send_path(x, idx, w, None, P, El)
    N = int(o["layout"]["n"])
    y = randn_bf16(N, H, c["seed"] + 2)
    o["out"] = oracle.combine(y, o["layout"]["token_pos"])
    g = gpu_send_path(x, idx, w, y, P, El)
    compare_send_path(x, idx, w, y, P, El, g, o)

    # no-sync route, dispatch (bf16 or fp8) and combine
    r = ep.route_nosync(idx.to(dev), w.to(dev), P, El)
    W = r["num_worst_rows"]
    assert_equal("token_pos (no-sync)", np_(r["token_pos"]), o["layout"]["token_pos"])
    for k in ("send_token_idx", "send_rank", "send_idx"):
        assert_equal(k + " (no-sync)", np_(r[k])[:N], o["layout"][k])
    if c["fp8"]:
        q, s = ep.dispatch_rows(x.to(dev), r["token_pos"], W, fp8=True, err=r["err"])
        oq, os_ = oracle.dispatch_fp8(x, o["layout"]["send_token_idx"])
        torch.cuda.synchronize()
        assert_equal("fp8 codes", np_(q)[:N], oq)
        assert_equal("fp8 scales (bits)", np_(s)[:N].view(np.uint32), os_.view(np.uint32))
    y_pad = torch.zeros((W, H), dtype=torch.bfloat16, device=dev)
    y_pad[:N] = y.to(dev)
    out = ep.combine_rows(y_pad, r["token_pos"], err=r["err"])
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    assert_combine_parity("combine (no-sync)", bits16(out), o["out"])

    # expert-batched prepare and weighted combine for one rank
    M = max(1, int(o["counts"]["tokens_per_expert"].reshape(P, El)[rank].max()) + int(c["seed"] % 5))
    zero_pad = bool(c["seed"] % 2)
    ob = oracle.batched_prepare(x, idx, E, El, rank, M, zero_pad=zero_pad)
    rb = ep.batched_prepare(x.to(dev), idx.to(dev), E, El, rank, M, zero_pad=zero_pad)
    yb = randn_bf16(El * M, H, c["seed"] + 3).reshape(El, M, H)
    ocb = oracle.batched_combine(yb, idx, w, ob["slot"], El, rank)
    outb = ep.batched_combine(yb.to(dev), idx.to(dev), w.to(dev), rb["slot"], rank, err=rb["err"])
    torch.cuda.synchronize()
    assert int(rb["err"].item()) == 0 and ob["err"] == 0
    assert_equal("tokens_per_expert (batched)", np_(rb["tokens_per_expert"]), ob["tokens_per_expert"])
    assert_equal("slot", np_(rb["slot"]), ob["slot"])
    bx = bits16(rb["b_x"])
    if zero_pad:
        assert_equal("b_x", bx, ob["b_x"])
    else:
        for e in range(El):
            n = int(ob["tokens_per_expert"][e])
            assert_equal(f"b_x[{e}]", bx[e, :n], ob["b_x"][e, :n])
    assert_combine_parity("batched combine", bits16(outb), ocb)

    # fp8 on the expert-batched layout, one scale layout per case
    if c["fp8"]:
        forms = [(ep.EP_SCALE_ROW_F32, False), (ep.EP_SCALE_COL_F32, True)]
        if H % 512 == 0:
            forms.append((ep.EP_SCALE_COL_UE8M0, True))
        fmt, rs = forms[c["seed"] % len(forms)]
        o8 = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, rs, zero_pad=True)
        r8 = ep.batched_prepare_fp8(x.to(dev), idx.to(dev), E, El, rank, M, fmt, rs, zero_pad=True)
        torch.cuda.synchronize()
        assert int(r8["err"].item()) == 0
        assert_equal("fp8 batched slot", np_(r8["slot"]), o8["slot"])
        assert_equal("fp8 batched codes", np_(r8["b_q"]), o8["b_q"])
        assert_equal("fp8 batched scales (bits)", np_(r8["b_scale"]).view(np.uint32), o8["b_scale"].view(np.uint32))

    # capacity drops and receive alignment on the batched layout (bf16 or fp8 rows)
    C = 1 + (c["seed"] * 7919) % M
    A = [1, 4, 16, 128][c["seed"] % 4]
    fx = ep.EP_SCALE_COL_F32 if c["fp8"] else None
    ox = oracle.batched_prepare_ex(x, idx, E, El, rank, M, C, A, fmt=fx, zero_pad=True)
    rx = ep.batched_prepare_ex(x.to(dev), idx.to(dev), E, El, rank, M, capacity=C, alignment=A, scale_fmt=fx,
                               zero_pad=True)
    torch.cuda.synchronize()
    assert int(rx["err"].item()) == 0 and ox["err"] == 0
    for k in ("slot", "tokens_per_expert", "dropped"):
        assert_equal(k + " (capacity)", np_(rx[k]), ox[k])
    rows = np_(rx["b_rows"]) if c["fp8"] else bits16(rx["b_rows"])
    assert_equal("rows (capacity)", rows, ox["b_rows"])
    if c["fp8"]:
        assert_equal("scales (capacity, bits)", np_(rx["b_scale"]).view(np.uint32), ox["b_scale"].view(np.uint32))

    # send layout with every rank segment aligned
    Ar = [2, 4, 16, 128][(c["seed"] // 4) % 4]
    ra = ep.route_nosync(idx.to(dev), w.to(dev), P, El, alignment=Ar)
    torch.cuda.synchronize()
    al = oracle.align_send_layout(o["layout"], o["counts"]["send_counts"], Ar)
    n = al["n"]
    assert int(ra["err"].item()) == 0
    assert_equal("rank_offsets (aligned)", np_(ra["rank_offsets"]), al["rank_offsets"])
    assert_equal("tokens_per_expert (aligned)", np_(ra["tokens_per_expert"]),
                 -(-o["counts"]["tokens_per_expert"] // Ar) * Ar)
    for k in ("send_token_idx", "send_rank", "send_idx"):
        assert_equal(k + " (aligned)", np_(ra[k])[:n], al[k])
    assert_equal("send_w (aligned, bits)", np_(ra["send_w"])[:n].view(np.uint32), al["send_w"].view(np.uint32))
    assert_equal("token_pos (aligned)", np_(ra["token_pos"]), al["token_pos"])

    # multihot map and dense probabilities
    if T * E <= CAP:
        om = oracle.indices_to_multihot(idx, w, E)
        rm, pr = ep.indices_to_multihot(idx.to(dev), w.to(dev), E)
        torch.cuda.synchronize()
        assert_equal("routing_map", np_(rm).astype(np.uint8), om["routing_map"])
        assert_equal("probs (bits)", np_(pr).view(np.uint32), om["probs"].view(np.uint32))
