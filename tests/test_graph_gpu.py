"""CUDA graph capture of the no-sync calls: one captured launch sequence,
replayed on new routing each time, must recompute every output from the
current inputs (parity with the oracle after every replay).  The
single-launch routing kernels synchronise their blocks through tagged flags
in the workspace; a replay repeats the host's arguments, so these tests are
what shows that a replay never passes the barrier on an earlier replay's
flags."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_combine_parity, assert_equal, bits16, np_, randn_bf16, routing_inputs

pytestmark = pytest.mark.gpu

# (seed, share of masked slots) of the inputs copied in before each replay
REPLAYS = [(101, 0.1), (202, 0.0), (303, 0.6), (404, 1.0), (505, 0.05)]


def _capture(fn, stream):
    """Run fn once on `stream` (first-call set-up), then capture it."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("with_tpe", [True, False])
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("T,H,K,P,El", [(5000, 256, 8, 8, 4), (1537, 136, 6, 16, 2)])
def test_route_dispatch_combine_graph_replays_new_routing(T, H, K, P, El, fused, with_tpe):
    dev = "cuda"
    W = T * min(K, P)
    idx = torch.empty((T, K), dtype=torch.int64, device=dev)
    wts = torch.empty((T, K), dtype=torch.float32, device=dev)
    x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    o_dest = torch.empty((T, K), dtype=torch.int32, device=dev)
    o_iir = torch.empty((T, P), dtype=torch.uint8, device=dev)
    o_sc = torch.empty(P, dtype=torch.int32, device=dev)
    o_ro = torch.empty(P + 1, dtype=torch.int32, device=dev)
    o_tpe = torch.empty(P * El, dtype=torch.int32, device=dev) if with_tpe else None
    o_sti = torch.empty(W, dtype=torch.int32, device=dev)
    o_sr = torch.empty(W, dtype=torch.int32, device=dev)
    o_si = torch.empty((W, K), dtype=torch.int64, device=dev)
    o_sw = torch.empty((W, K), dtype=torch.float32, device=dev)
    o_tp = torch.empty((T, P), dtype=torch.int32, device=dev)
    recv = torch.empty((W, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = ep.workspace(T, K, P, El)
    cws = ep.combine_ws()
    err = ep.error_word()

    def step():
        s = torch.cuda.current_stream()
        if fused:   # route, then the dispatch as its programmatic dependent
            ep.ep_dispatch_nosync(x, idx, wts, T, K, H, P, El, W, 0, o_dest, o_iir, o_sc, o_ro, o_tpe, o_sti, o_sr,
                                  o_si, o_sw, o_tp, recv, None, ws, err, s)
        else:
            ep.ep_route_nosync(idx, wts, T, K, P, El, W, o_dest, o_iir, o_sc, o_ro, o_tpe, o_sti, o_sr, o_si, o_sw,
                               o_tp, ws, err, s)
            ep.ep_dispatch(x, T, H, o_tp, P, W, recv, None, 0, err, s)
        # combine the received rows themselves: out[t] = (ranks of t) * x[t]
        ep.ep_combine(recv, T, H, o_tp, P, W, out, 0, cws, err, s)

    i0, w0 = routing_inputs(T, K, P * El, 99, 0.2)
    idx.copy_(i0)
    wts.copy_(w0)
    x.copy_(randn_bf16(T, H, 98))
    g = _capture(step, torch.cuda.Stream())
    for seed, fu in REPLAYS:
        hi, hw = routing_inputs(T, K, P * El, seed, fu)
        hx = randn_bf16(T, H, seed + 1)
        idx.copy_(hi)
        wts.copy_(hw)
        x.copy_(hx)
        err.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
        o = oracle.send_path(hx, hi, hw, None, P, El)
        oc, ol = o["counts"], o["layout"]
        N = ol["n"]
        assert_equal(f"dest/{seed}", np_(o_dest), oc["dest"])
        assert_equal(f"is_in_rank/{seed}", np_(o_iir), oc["is_in_rank"])
        assert_equal(f"send_counts/{seed}", np_(o_sc), oc["send_counts"])
        if with_tpe:
            assert_equal(f"tokens_per_expert/{seed}", np_(o_tpe), oc["tokens_per_expert"])
        assert int(o_ro[P].item()) == N
        for k, t in (("send_token_idx", o_sti), ("send_rank", o_sr), ("send_idx", o_si)):
            assert_equal(f"{k}/{seed}", np_(t)[:N], ol[k])
        assert_equal(f"send_w/{seed}", np_(o_sw)[:N].view(np.uint32), ol["send_w"].view(np.uint32))
        assert_equal(f"token_pos/{seed}", np_(o_tp), ol["token_pos"])
        assert_equal(f"recv_x/{seed}", bits16(recv)[:N], o["recv_x"])
        assert_combine_parity(f"combine/{seed}", bits16(out), oracle.combine(o["recv_x"], ol["token_pos"]))


@pytest.mark.parametrize("T,H,K,E,El,rank,M", [(4000, 128, 8, 64, 16, 2, 4000), (999, 64, 4, 32, 32, 0, 700)])
def test_batched_prepare_combine_graph_replays_new_routing(T, H, K, E, El, rank, M):
    dev = "cuda"
    idx = torch.empty((T, K), dtype=torch.int64, device=dev)
    wts = torch.empty((T, K), dtype=torch.float32, device=dev)
    x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    b_x = torch.empty((El, M, H), dtype=torch.bfloat16, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = ep.workspace(T, K, E // El, El, 1)
    cws = ep.combine_ws()
    err = ep.error_word()

    def step():
        s = torch.cuda.current_stream()
        ep.ep_batched_prepare(x, idx, T, K, H, E, El, rank, M, b_x, tpe, slot, 1, ws, err, s)
        # the expert is the identity: out[t] = sum_k w[t,k] x[t] over local k
        ep.ep_batched_combine(b_x, idx, wts, slot, T, K, H, El, rank, M, out, cws, err, s)

    i0, w0 = routing_inputs(T, K, E, 77, 0.1)
    idx.copy_(i0)
    wts.copy_(w0)
    x.copy_(randn_bf16(T, H, 78))
    g = _capture(step, torch.cuda.Stream())
    for seed, fu in REPLAYS:
        hi, hw = routing_inputs(T, K, E, seed, fu)
        hx = randn_bf16(T, H, seed + 2)
        idx.copy_(hi)
        wts.copy_(hw)
        x.copy_(hx)
        err.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
        o = oracle.batched_prepare(hx, hi, E, El, rank, M, zero_pad=True)
        assert_equal(f"tokens_per_expert/{seed}", np_(tpe), o["tokens_per_expert"])
        assert_equal(f"slot/{seed}", np_(slot), o["slot"])
        assert_equal(f"b_x/{seed}", bits16(b_x), o["b_x"])
        o_out = oracle.batched_combine(o["b_x"], hi, hw, o["slot"], El, rank)
        assert_combine_parity(f"batched combine/{seed}", bits16(out), o_out)


@pytest.mark.parametrize("fmt,rs", [(ep.EP_SCALE_COL_F32, 0), (ep.EP_SCALE_COL_UE8M0, 1)])
@pytest.mark.parametrize("T,H,K,E,El,rank,M", [(6000, 512, 8, 64, 16, 2, 3000), (999, 512, 4, 32, 32, 0, 700)])
def test_batched_prepare_fp8_graph_replays_new_routing(T, H, K, E, El, rank, M, fmt, rs):
    # slot kernel + fp8 row scatter (its programmatic dependent) + zero fill,
    # replayed on new routing: every output is recomputed by each replay
    dev = "cuda"
    idx = torch.empty((T, K), dtype=torch.int64, device=dev)
    x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    shape, dt = ep.batched_scale_storage(El, M, H, fmt)
    b_q = torch.empty((El, M, H), dtype=torch.uint8, device=dev)
    b_s = torch.empty(shape, dtype=dt, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws = ep.workspace(T, K, E // El, El, 1)
    err = ep.error_word()

    def step():
        s = torch.cuda.current_stream()
        ep.ep_batched_prepare_fp8(x, idx, T, K, H, E, El, rank, M, b_q, b_s, fmt, rs, tpe, slot, 1, ws, err, s)

    i0, _ = routing_inputs(T, K, E, 71, 0.1)
    idx.copy_(i0)
    x.copy_(randn_bf16(T, H, 72))
    g = _capture(step, torch.cuda.Stream())
    for seed, fu in REPLAYS:
        hi, _ = routing_inputs(T, K, E, seed, fu)
        hx = randn_bf16(T, H, seed + 3)
        idx.copy_(hi)
        x.copy_(hx)
        err.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
        o = oracle.batched_prepare_fp8(hx, hi, E, El, rank, M, fmt, bool(rs), zero_pad=True)
        assert_equal(f"tokens_per_expert/{seed}", np_(tpe), o["tokens_per_expert"])
        assert_equal(f"slot/{seed}", np_(slot), o["slot"])
        assert_equal(f"codes/{seed}", np_(b_q), o["b_q"])
        assert_equal(f"scales/{seed}", np_(b_s).view(np.uint32), o["b_scale"].view(np.uint32))
