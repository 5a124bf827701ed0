"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.  Counts, layouts, indices and moved bytes are
compared bit for bit; combine outputs too (both sides accumulate in fp32 in
the same order with the same roundings, which is stricter than the 1 bf16 ulp
target).  Full-size workloads run at the sizes the benchmark times."""
import dataclasses

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl

from _paths import (assert_combine_parity, assert_equal, bits16, compare_send_path, gpu_send_path, np_)
from _paths import randn_bf16 as _randn
from _paths import routing_inputs as _routing

pytestmark = pytest.mark.gpu


def _send_inputs(w: wl.Workload):
    x, idx, wts = wl.make(w)
    return x, idx, wts


@pytest.mark.parametrize("name", ["tiny", "mid", "large"])
def test_send_path_workload(name):
    w = wl.WORKLOADS[name]
    x, idx, wts = _send_inputs(w)
    o = oracle.send_path(x, idx, wts, None, w.P, w.E_local)
    y = wl.expert_outputs(w, o["layout"]["n"])
    o["out"] = oracle.combine(y, o["layout"]["token_pos"])
    g = gpu_send_path(x, idx, wts, y, w.P, w.E_local)
    compare_send_path(x, idx, wts, y, w.P, w.E_local, g, o)


def test_send_path_fp32_combine():
    w = wl.WORKLOADS["mid"]
    x, idx, wts = _send_inputs(w)
    o = oracle.send_path(x, idx, wts, None, w.P, w.E_local)
    y = wl.expert_outputs(w, o["layout"]["n"])
    want = oracle.combine(y, o["layout"]["token_pos"], out_f32=True)
    g = gpu_send_path(x, idx, wts, y, w.P, w.E_local, out_f32=True)
    assert_equal("combine fp32 (bits)", np_(g["out"]).view(np.uint32), want.view(np.uint32))


def _batched(w: wl.Workload, zero_pad=False):
    x, idx, wts = wl.make(w)
    o = oracle.batched_prepare(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, zero_pad=zero_pad)
    dev = "cuda"
    r = ep.batched_prepare(x.to(dev), idx.to(dev), w.E, w.E_local, w.rank, w.max_num_tokens, zero_pad=zero_pad)
    y = wl.batched_expert_outputs(w, o["tokens_per_expert"])
    o_out = oracle.batched_combine(y, idx, wts, o["slot"], w.E_local, w.rank)
    g_out = ep.batched_combine(y.to(dev), idx.to(dev), wts.to(dev), r["slot"], w.rank, err=r["err"])
    torch.cuda.synchronize()
    return x, idx, wts, o, r, o_out, g_out


def test_batched_workload():
    w = wl.WORKLOADS["batched"]
    x, idx, wts, o, r, o_out, g_out = _batched(w)
    assert int(r["err"].item()) == 0
    tpe = o["tokens_per_expert"]
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), tpe)
    assert_equal("slot", np_(r["slot"]), o["slot"])
    bx = bits16(r["b_x"])
    for e in range(w.E_local):
        assert_equal(f"b_x[{e}] valid rows", bx[e, :tpe[e]], o["b_x"][e, :tpe[e]])
    out_bits = bits16(g_out)
    assert not np.any(np.isnan(g_out.float().cpu().numpy())), "combine read a NaN padding row"
    assert_combine_parity("batched combine", out_bits, o_out)


def test_batched_zero_pad_small():
    w = dataclasses.replace(wl.WORKLOADS["batched"].scaled(T=1000), max_num_tokens=300, H=264)
    x, idx, wts, o, r, o_out, g_out = _batched(w, zero_pad=True)
    assert int(r["err"].item()) == 0
    assert_equal("b_x (zero padded)", bits16(r["b_x"]), o["b_x"])
    assert_combine_parity("batched combine", bits16(g_out), o_out)


def _chunked_fp8(w: wl.Workload):
    """One count launch for all chunks, one D2H of the counts, then per chunk
    layout -> fp8 dispatch -> synthetic expert -> combine on the GPU."""
    dev = "cuda"
    x, idx, wts = wl.make(w)
    bounds = ep.chunk_bounds(w.T, w.chunks)
    xd, idd, wd = x.to(dev), idx.to(dev), wts.to(dev)
    err = ep.error_word()
    c = ep.compute_send_counts(idd, w.P, w.E_local, chunk_bounds=bounds, err=err)
    counts = c["send_counts"].cpu()                       # the one device-to-host copy
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    per_chunk = []
    for i in range(w.chunks):
        s, e = bounds[i], bounds[i + 1]
        N = int(counts[i].sum())
        lay = ep.build_send_layout(idd[s:e], wd[s:e], c["dest"][s:e], c["is_in_rank"][s:e], N, w.E_local, err=err)
        q, sc = ep.dispatch_rows(xd[s:e], lay["token_pos"], N, fp8=True, err=err)
        local = ep.local_expert_fp8(q, sc, lay["send_idx"], lay["send_w"], err=err)
        out[s:e] = ep.combine_rows(local, lay["token_pos"], err=err)
        per_chunk.append(dict(layout=lay, q=q, scale=sc, local=local, N=N))
    torch.cuda.synchronize()
    return x, idx, wts, bounds, c, per_chunk, out, int(err.item())


def test_chunked_fp8_reduced_full_compare():
    w = wl.WORKLOADS["chunk_fp8"].scaled(T=2048 + 37)    # 4 ragged chunks
    x, idx, wts, bounds, c, per_chunk, out, err = _chunked_fp8(w)
    assert err == 0
    assert bounds == oracle.chunk_bounds(w.T, w.chunks).tolist()
    ob = oracle.chunk_bounds(w.T, w.chunks)
    for i in range(w.chunks):
        s, e = int(ob[i]), int(ob[i + 1])
        oc = oracle.compute_send_counts(idx[s:e], w.P, w.E_local)
        assert_equal(f"chunk {i} send_counts", np_(c["send_counts"][i]), oc["send_counts"])
        ol = oracle.build_send_layout(idx[s:e], wts[s:e], oc["dest"], oc["is_in_rank"], w.E_local)
        g = per_chunk[i]
        for k in ("send_token_idx", "send_rank", "send_idx", "token_pos"):
            assert_equal(f"chunk {i} {k}", np_(g["layout"][k]), ol[k])
        q, sc = oracle.dispatch_fp8(x[s:e], ol["send_token_idx"])
        assert_equal(f"chunk {i} fp8 codes", np_(g["q"]), q)
        assert_equal(f"chunk {i} fp8 scales (bits)", np_(g["scale"]).view(np.uint32), sc.view(np.uint32))
        local = oracle.local_expert_fp8(q, sc, ol["send_idx"], ol["send_w"])
        assert_equal(f"chunk {i} local expert", bits16(g["local"]), local)
        o_out = oracle.combine(local, ol["token_pos"])
        assert_combine_parity(f"chunk {i} combine", bits16(out[s:e]), o_out)
    # tokens_per_expert over all chunks from the same single count launch
    assert_equal("tokens_per_expert", np_(c["tokens_per_expert"]),
                 oracle.compute_send_counts(idx, w.P, w.E_local)["tokens_per_expert"])


def test_chunked_fp8_full_size_sampled():
    w = wl.WORKLOADS["chunk_fp8"]
    x, idx, wts, bounds, c, per_chunk, out, err = _chunked_fp8(w)
    assert err == 0
    # counts of every chunk, exactly (integer work, cheap on the host)
    for i in range(w.chunks):
        s, e = bounds[i], bounds[i + 1]
        oc = oracle.compute_send_counts(idx[s:e], w.P, w.E_local, with_tokens_per_expert=False)
        assert_equal(f"chunk {i} send_counts", np_(c["send_counts"][i]), oc["send_counts"])
    # sampled tokens: the whole pipeline for one token is the pipeline on the
    # one-token problem (each token's result depends only on its own row,
    # routing and weights)
    g = np.random.Generator(np.random.PCG64(123))
    sample = np.sort(g.choice(w.T, size=96, replace=False))
    outb = bits16(out)
    for t in sample.tolist():
        xi, ii, wi = x[t:t + 1], idx[t:t + 1], wts[t:t + 1]
        r = oracle.send_path(xi, ii, wi, None, w.P, w.E_local)
        lay = r["layout"]
        q, sc = oracle.dispatch_fp8(xi, lay["send_token_idx"])
        local = oracle.local_expert_fp8(q, sc, lay["send_idx"], lay["send_w"])
        want = oracle.combine(local, lay["token_pos"])
        assert_combine_parity(f"token {t}", outb[t:t + 1], want)


def test_fp8_codes_for_every_bf16_input():
    # Groups whose max is exactly 448 have inv = 448/448 = 1, so the codes are
    # the plain e4m3 conversion of every finite bf16 value with |x| <= 448.
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_bits_to_f32(allb)
    vals = allb[np.isfinite(f) & (np.abs(f) <= 448.0)]
    per = 127
    ngroups = -(-vals.size // per)
    H = 128 * 16
    rows = -(-ngroups // 16)
    buf = np.zeros((rows * 16, 128), np.uint16)
    buf[:, 0] = 0x43E0                                    # 448.0 in bf16
    flat = np.zeros(rows * 16 * per, np.uint16)
    flat[:vals.size] = vals
    buf[:, 1:] = flat.reshape(rows * 16, per)
    x = torch.from_numpy(buf.reshape(rows, H).view(np.int16)).view(torch.bfloat16)
    T = rows
    token_pos = torch.arange(T, dtype=torch.int32).view(T, 1)
    err = ep.error_word()
    q, s = ep.dispatch_rows(x.cuda(), token_pos.cuda(), T, fp8=True, err=err)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize_fp8_rows(x)
    assert int(err.item()) == 0
    assert_equal("codes", np_(q), oq)
    assert np.all(np_(s) == np.float32(1.0))
    assert_equal("scales", np_(s), os_)


# ------------------------------------------------------------------ edges --
EDGE = [
    # T, H, K, P, E_local, frac_unrouted, dup
    (1, 64, 2, 4, 2, 0.0, False),
    (1000, 136, 4, 8, 4, 0.1, False),        # ragged tokens and a ragged vector count
    (257, 8, 3, 2, 3, 0.3, True),            # smallest row, duplicate experts
    (600, 256, 8, 1, 16, 0.2, False),        # P = 1
    (300, 128, 32, 64, 1, 0.05, False),      # K = 32, P = 64
    (777, 512, 1, 16, 4, 0.25, False),       # K = 1: counting sort
    (513, 1024, 6, 8, 8, 1.0, False),        # nothing routed
    (300, 16384, 4, 4, 4, 0.0, False),       # a row longer than one pass of the block
    (1000, 64, 8, 64, 128, 0.1, False),      # E = P * E_local = 8192, the largest expert count
]


@pytest.mark.parametrize("T,H,K,P,E_local,fu,dup", EDGE)
def test_send_path_edges(T, H, K, P, E_local, fu, dup):
    idx, wts = _routing(T, K, P * E_local, seed=T + H, frac_unrouted=fu, dup=dup)
    x = _randn(T, H, T)
    o = oracle.send_path(x, idx, wts, None, P, E_local)
    y = _randn(max(o["layout"]["n"], 1), H, T + 1)[:o["layout"]["n"]]
    o["out"] = oracle.combine(y, o["layout"]["token_pos"])
    g = gpu_send_path(x, idx, wts, y, P, E_local)
    compare_send_path(x, idx, wts, y, P, E_local, g, o)


def test_empty_inputs():
    dev = "cuda"
    idx = torch.empty((0, 4), dtype=torch.int64, device=dev)
    c = ep.compute_send_counts(idx, 4, 2)
    torch.cuda.synchronize()
    assert np_(c["send_counts"]).tolist() == [[0, 0, 0, 0]]
    assert np_(c["rank_offsets"]).tolist() == [[0, 0, 0, 0, 0]]
    assert np_(c["tokens_per_expert"]).tolist() == [0] * 8
    lay = ep.build_send_layout(idx, torch.empty((0, 4), device=dev), c["dest"], c["is_in_rank"], 0, 2)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    assert ep.dispatch_rows(x, lay["token_pos"], 0).shape == (0, 64)
    assert ep.combine_rows(torch.empty((0, 64), dtype=torch.bfloat16, device=dev), lay["token_pos"]).shape == (0, 64)
    r = ep.batched_prepare(x, idx, 8, 2, 1, 16)
    torch.cuda.synchronize()
    assert np_(r["tokens_per_expert"]).tolist() == [0, 0]
    with pytest.raises(ep.EPError):
        ep.build_send_layout(idx, torch.empty((0, 4), device=dev), c["dest"], c["is_in_rank"], 3, 2)


def test_invalid_expert_ids_are_flagged_and_skipped():
    idx = torch.tensor([[0, 99], [-7, 3], [5, -1], [2, 1]], dtype=torch.int64)
    wts = torch.full((4, 2), 0.5)
    x = _randn(4, 64, 5)
    o = oracle.send_path(x, idx, wts, None, 4, 2)
    assert o["counts"]["err"] & oracle.ERR_INVALID_EXPERT
    y = _randn(o["layout"]["n"], 64, 6)
    o["out"] = oracle.combine(y, o["layout"]["token_pos"])
    g = gpu_send_path(x, idx, wts, y, 4, 2)
    assert g["err"] & ep.EP_ERR_INVALID_EXPERT
    g["err"] = 0
    compare_send_path(x, idx, wts, y, 4, 2, g, o)


def test_num_send_mismatch_is_flagged_and_writes_stay_in_bounds():
    T, H, K, P, El = 500, 64, 4, 4, 4
    idx, wts = _routing(T, K, P * El, 3)
    dev = "cuda"
    c = ep.compute_send_counts(idx.to(dev), P, El)
    N = int(c["send_counts"].sum().item())
    short = N - 7
    guard = 16
    err = ep.error_word()
    sti = torch.full((short + guard,), -12345, dtype=torch.int32, device=dev)
    sr = torch.full_like(sti, -12345)
    si = torch.full(((short + guard), K), -12345, dtype=torch.int64, device=dev)
    sw = torch.full(((short + guard), K), 7.0, dtype=torch.float32, device=dev)
    tp = torch.empty((T, P), dtype=torch.int32, device=dev)
    ws = ep.workspace(T, K, P, El)
    ep.ep_build_send_layout(idx.to(dev), wts.to(dev), c["dest"], c["is_in_rank"], T, K, P, El, short,
                            sti, sr, si, sw, tp, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERR_COUNT_MISMATCH
    assert np.all(np_(sti[short:]) == -12345) and np.all(np_(si[short:]) == -12345)
    assert np.all(np_(sw[short:]) == 7.0)
    assert int(tp.max().item()) < short
    # dispatch with the clipped handle writes only rows < short
    x = _randn(T, H, 4).to(dev)
    recv = torch.full((short + guard, H), 3.0, dtype=torch.bfloat16, device=dev)
    ep.ep_dispatch(x, T, H, tp, P, short, recv, None, 0, err)
    torch.cuda.synchronize()
    assert torch.all(recv[short:] == 3.0)


def test_batched_capacity_overflow():
    T, H, K, E, El, rank, M = 400, 64, 4, 8, 4, 0, 50
    idx, wts = _routing(T, K, E, 8, frac_unrouted=0.0)
    x = _randn(T, H, 9)
    o = oracle.batched_prepare(x, idx, E, El, rank, M)
    assert o["err"] & oracle.ERR_CAPACITY
    dev = "cuda"
    guard = torch.full((El * M + 8, H), 5.0, dtype=torch.bfloat16, device=dev)
    b_x = guard[:El * M].view(El, M, H)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    err = ep.error_word()
    ws = ep.workspace(T, K, E // El, El)
    ep.ep_batched_prepare(x.to(dev), idx.to(dev), T, K, H, E, El, rank, M, b_x, tpe, slot, 0, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERR_CAPACITY
    assert_equal("tokens_per_expert (clipped)", np_(tpe), o["tokens_per_expert"])
    assert_equal("slot", np_(slot), o["slot"])
    assert torch.all(guard[El * M:] == 5.0)
    bx = bits16(b_x)
    for e in range(El):
        assert_equal(f"b_x[{e}]", bx[e, :o["tokens_per_expert"][e]], o["b_x"][e, :o["tokens_per_expert"][e]])


def test_batched_duplicate_experts_small():
    T, H, K, E, El, rank, M = 333, 128, 6, 12, 4, 2, 400
    idx, wts = _routing(T, K, E, 10, dup=True)
    x = _randn(T, H, 11)
    o = oracle.batched_prepare(x, idx, E, El, rank, M)
    dev = "cuda"
    r = ep.batched_prepare(x.to(dev), idx.to(dev), E, El, rank, M)
    w = wl.Workload("dup", T=T, H=H, E=E, K=K, P=E // El, routing="uniform", rank=rank, max_num_tokens=M)
    y = wl.batched_expert_outputs(w, o["tokens_per_expert"])
    o_out = oracle.batched_combine(y, idx, wts, o["slot"], El, rank)
    g_out = ep.batched_combine(y.to(dev), idx.to(dev), wts.to(dev), r["slot"], rank, err=r["err"])
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    assert_equal("slot", np_(r["slot"]), o["slot"])
    assert_combine_parity("batched combine", bits16(g_out), o_out)


# --------------------------------------------------- no-sync (worst-case) path --
# with_tpe: tokens_per_expert asked for, or not (no expert partials)
@pytest.mark.parametrize("with_tpe", [True, False])
@pytest.mark.parametrize("name", ["tiny", "mid", "large"])
def test_route_nosync_matches_oracle(name, with_tpe):
    w = wl.WORKLOADS[name]
    x, idx, wts = wl.make(w)
    o = oracle.send_path(x, idx, wts, None, w.P, w.E_local)
    N = o["layout"]["n"]
    y = wl.expert_outputs(w, N)
    want_out = oracle.combine(y, o["layout"]["token_pos"])
    dev = "cuda"
    r = ep.route_nosync(idx.to(dev), wts.to(dev), w.P, w.E_local, with_tokens_per_expert=with_tpe)
    W = r["num_worst_rows"]
    recv = ep.dispatch_rows(x.to(dev), r["token_pos"], W, err=r["err"])
    y_pad = torch.zeros((W, w.H), dtype=torch.bfloat16, device=dev)
    y_pad[:N] = y.to(dev)
    out = ep.combine_rows(y_pad, r["token_pos"], err=r["err"])
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    oc, ol = o["counts"], o["layout"]
    assert_equal("dest", np_(r["dest"]), oc["dest"])
    assert_equal("is_in_rank", np_(r["is_in_rank"]), oc["is_in_rank"])
    assert_equal("send_counts", np_(r["send_counts"]), oc["send_counts"])
    assert_equal("rank_offsets", np_(r["rank_offsets"]), np.concatenate([[0], np.cumsum(oc["send_counts"])]))
    if with_tpe:
        assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), oc["tokens_per_expert"])
    for k in ("send_token_idx", "send_rank", "send_idx"):
        assert_equal(k, np_(r[k])[:N], ol[k])
    assert_equal("send_w(bits)", np_(r["send_w"])[:N].view(np.uint32), ol["send_w"].view(np.uint32))
    assert_equal("token_pos", np_(r["token_pos"]), ol["token_pos"])
    assert_equal("recv_x", bits16(recv)[:N], o["recv_x"])
    assert_combine_parity("combine", bits16(out), want_out)


def test_route_nosync_capacity_is_flagged_and_bounded():
    T, K, P, El = 700, 4, 4, 4
    idx, wts = _routing(T, K, P * El, 21)
    o = oracle.send_path(_randn(T, 8, 1), idx, wts, None, P, El)
    N = o["layout"]["n"]
    cap = N - 11
    dev = "cuda"
    guard = 8
    r = ep.route_nosync(idx.to(dev), wts.to(dev), P, El, num_worst_rows=N + guard)   # enough rows
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    assert int(r["rank_offsets"][P].item()) == N
    # now with too few rows: flagged, nothing past the capacity written
    sti = torch.full((cap + guard,), -5, dtype=torch.int32, device=dev)
    sr = torch.full_like(sti, -5)
    si = torch.full((cap + guard, K), -5, dtype=torch.int64, device=dev)
    sw = torch.full((cap + guard, K), 9.0, device=dev)
    outs = dict(dest=torch.empty((T, K), dtype=torch.int32, device=dev),
                iir=torch.empty((T, P), dtype=torch.uint8, device=dev),
                sc=torch.empty(P, dtype=torch.int32, device=dev), ro=torch.empty(P + 1, dtype=torch.int32, device=dev),
                tp=torch.empty((T, P), dtype=torch.int32, device=dev))
    err = ep.error_word()
    ep.ep_route_nosync(idx.to(dev), wts.to(dev), T, K, P, El, cap, outs["dest"], outs["iir"], outs["sc"], outs["ro"],
                       None, sti, sr, si, sw, outs["tp"], ep.workspace(T, K, P, El), err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERR_CAPACITY
    assert int(outs["ro"][P].item()) == N
    assert torch.all(sti[cap:] == -5) and torch.all(si[cap:] == -5) and torch.all(sw[cap:] == 9.0)
    assert int(outs["tp"].max().item()) < cap
    ol = o["layout"]
    assert_equal("rows below capacity", np_(sti[:cap]), ol["send_token_idx"][:cap])


@pytest.mark.parametrize("with_tpe", [True, False])
@pytest.mark.parametrize("T,H,K,P,E_local,fu,dup", EDGE)
def test_route_nosync_edges(T, H, K, P, E_local, fu, dup, with_tpe):
    idx, wts = _routing(T, K, P * E_local, seed=T + H + 1, frac_unrouted=fu, dup=dup)
    o = oracle.send_path(_randn(T, 8, 2), idx, wts, None, P, E_local)
    N = o["layout"]["n"]
    dev = "cuda"
    r = ep.route_nosync(idx.to(dev), wts.to(dev), P, E_local, with_tokens_per_expert=with_tpe)
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    oc, ol = o["counts"], o["layout"]
    assert_equal("dest", np_(r["dest"]), oc["dest"])
    assert_equal("is_in_rank", np_(r["is_in_rank"]), oc["is_in_rank"])
    assert_equal("send_counts", np_(r["send_counts"]), oc["send_counts"])
    if with_tpe:
        assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), oc["tokens_per_expert"])
    assert int(r["rank_offsets"][P].item()) == N
    for k in ("send_token_idx", "send_rank", "send_idx"):
        assert_equal(k, np_(r[k])[:N], ol[k])
    assert_equal("send_w(bits)", np_(r["send_w"])[:N].view(np.uint32), ol["send_w"].view(np.uint32))
    assert_equal("token_pos", np_(r["token_pos"]), ol["token_pos"])


@pytest.mark.parametrize("T,K,P,El", [(16385, 8, 8, 4), (32768, 6, 16, 4), (32769, 8, 8, 4), (30000, 3, 40, 2)])
def test_route_nosync_larger_problems(T, K, P, El):
    # the no-sync route without expert counts on larger problems (more than
    # 32 ranks with a generic K among them), and ep_dispatch_nosync on the same
    # inputs: both give the oracle's layout
    idx, wts = _routing(T, K, P * El, seed=T + 5, frac_unrouted=0.1)
    x = _randn(T, 16, 3)
    o = oracle.send_path(x, idx, wts, None, P, El)
    oc, ol = o["counts"], o["layout"]
    N = ol["n"]
    dev = "cuda"
    r = ep.route_nosync(idx.to(dev), wts.to(dev), P, El, with_tokens_per_expert=False)
    W = r["num_worst_rows"]
    outs = {k: torch.full_like(r[k], -9) for k in ("dest", "is_in_rank", "send_counts", "rank_offsets",
                                                    "send_token_idx", "send_rank", "send_idx", "send_w", "token_pos")}
    recv = torch.empty((W, 16), dtype=torch.bfloat16, device=dev)
    err = ep.error_word()
    ep.ep_dispatch_nosync(x.to(dev), idx.to(dev), wts.to(dev), T, K, 16, P, El, W, 0, outs["dest"],
                          outs["is_in_rank"], outs["send_counts"], outs["rank_offsets"], None, outs["send_token_idx"],
                          outs["send_rank"], outs["send_idx"], outs["send_w"], outs["token_pos"], recv, None,
                          ep.workspace(T, K, P, El), err)
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0 and int(err.item()) == 0
    for g in (r, outs):
        assert_equal("dest", np_(g["dest"]), oc["dest"])
        assert_equal("is_in_rank", np_(g["is_in_rank"]), oc["is_in_rank"])
        assert_equal("send_counts", np_(g["send_counts"]), oc["send_counts"])
        assert int(g["rank_offsets"][P].item()) == N
        for k in ("send_token_idx", "send_rank", "send_idx"):
            assert_equal(k, np_(g[k])[:N], ol[k])
        assert_equal("send_w(bits)", np_(g["send_w"])[:N].view(np.uint32), ol["send_w"].view(np.uint32))
        assert_equal("token_pos", np_(g["token_pos"]), ol["token_pos"])
    assert_equal("recv_x", bits16(recv)[:N], o["recv_x"])


def test_route_nosync_repeated_calls_reuse_workspace():
    # back-to-back calls on one workspace: each call's arrival flags carry a
    # new tag, so the previous call's flags never satisfy the barrier
    w = wl.WORKLOADS["mid"]
    idx, wts = wl.routing(w)
    dev = "cuda"
    ws = ep.workspace(w.T, w.K, w.P, w.E_local)
    first = ep.route_nosync(idx.to(dev), wts.to(dev), w.P, w.E_local, ws=ws)
    idx2 = idx.clone()
    idx2[:, 0] = -1
    second = ep.route_nosync(idx2.to(dev), wts.to(dev), w.P, w.E_local, ws=ws)
    third = ep.route_nosync(idx.to(dev), wts.to(dev), w.P, w.E_local, ws=ws)
    torch.cuda.synchronize()
    o2 = oracle.compute_send_counts(idx2, w.P, w.E_local)
    assert_equal("second send_counts", np_(second["send_counts"]), o2["send_counts"])
    N = int(first["rank_offsets"][w.P].item())
    for k in ("send_counts", "rank_offsets", "token_pos"):
        assert torch.equal(first[k], third[k]), k
    for k in ("send_token_idx", "send_rank", "send_idx", "send_w"):   # rows past N are not written
        assert torch.equal(first[k][:N], third[k][:N]), k
    assert int(first["err"].item()) == int(second["err"].item()) == int(third["err"].item()) == 0


@pytest.mark.parametrize("name", ["mid", "large"])
def test_combine_static_and_shared_work_split_agree(name):
    # The combine deals (token, chunk) items to the SMs either round-robin (no
    # scratch) or from a shared counter (with scratch); the results are the
    # same bits and equal the oracle.
    w = wl.WORKLOADS[name]
    idx, wts = wl.routing(w)
    o = oracle.compute_send_counts(idx, w.P, w.E_local, with_tokens_per_expert=False)
    ol = oracle.build_send_layout(idx, wts, o["dest"], o["is_in_rank"], w.E_local)
    y = wl.expert_outputs(w, ol["n"])
    want = oracle.combine(y, ol["token_pos"])
    yd, tp = y.cuda(), torch.from_numpy(ol["token_pos"]).cuda()
    a = ep.combine_rows(yd, tp, ws=None)
    b = ep.combine_rows(yd, tp)
    c = ep.combine_rows(yd, tp, ws=ep.combine_ws())
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(b, c)
    assert_combine_parity("combine", bits16(b), want)


# --------------------------------------------------------- native chunk driver --
def _oracle_chunked(x, idx, wts, P, E_local, chunks, fp8):
    b = oracle.chunk_bounds(x.shape[0], chunks)
    outs = []
    for i in range(chunks):
        s, e = int(b[i]), int(b[i + 1])
        r = oracle.send_path(x[s:e], idx[s:e], wts[s:e], None, P, E_local)
        lay = r["layout"]
        if fp8:
            q, sc = oracle.dispatch_fp8(x[s:e], lay["send_token_idx"])
            local = oracle.local_expert_fp8(q, sc, lay["send_idx"], lay["send_w"])
        else:
            local = r["recv_x"]                       # identity expert
        outs.append(oracle.combine(local, lay["token_pos"]))
    return np.concatenate(outs)


def test_chunked_driver_fp8_matches_oracle():
    w = wl.WORKLOADS["chunk_fp8"].scaled(T=2048 + 37)
    x, idx, wts = wl.make(w)
    out = ep.dispatch_chunked_forward(x.cuda(), idx.cuda(), wts.cuda(), num_local_experts=w.E_local, num_ranks=w.P,
                                      chunks=w.chunks, fp8=True)
    torch.cuda.synchronize()
    assert_combine_parity("chunked fp8", bits16(out), _oracle_chunked(x, idx, wts, w.P, w.E_local, w.chunks, True))


def test_chunked_driver_bf16_python_local_kernel():
    w = dataclasses.replace(wl.WORKLOADS["mid"].scaled(T=1500), chunks=5)
    x, idx, wts = wl.make(w)
    seen = []

    def identity(chunk, recv_x, recv_scale, send_idx, send_w, local_out):
        seen.append((chunk, recv_x.shape[0]))
        local_out.copy_(recv_x)

    out = ep.dispatch_chunked_forward(x.cuda(), idx.cuda(), wts.cuda(), num_local_experts=w.E_local, num_ranks=w.P,
                                      chunks=w.chunks, local_kernel=identity)
    torch.cuda.synchronize()
    assert [c for c, _ in seen] == list(range(w.chunks))
    assert_combine_parity("chunked bf16", bits16(out), _oracle_chunked(x, idx, wts, w.P, w.E_local, w.chunks, False))


def test_chunked_driver_fp8_full_size_sampled():
    w = wl.WORKLOADS["chunk_fp8"]
    x, idx, wts = wl.make(w)
    out = ep.dispatch_chunked_forward(x.cuda(), idx.cuda(), wts.cuda(), num_local_experts=w.E_local, num_ranks=w.P,
                                      chunks=w.chunks, fp8=True)
    torch.cuda.synchronize()
    outb = bits16(out)
    g = np.random.Generator(np.random.PCG64(321))
    for t in np.sort(g.choice(w.T, size=64, replace=False)).tolist():
        r = oracle.send_path(x[t:t + 1], idx[t:t + 1], wts[t:t + 1], None, w.P, w.E_local)
        lay = r["layout"]
        q, sc = oracle.dispatch_fp8(x[t:t + 1], lay["send_token_idx"])
        want = oracle.combine(oracle.local_expert_fp8(q, sc, lay["send_idx"], lay["send_w"]), lay["token_pos"])
        assert_combine_parity(f"token {t}", outb[t:t + 1], want)


# ------------------------------------------- chunked forward without host sync --
@pytest.mark.parametrize("n_sets", [1, 2])
def test_chunked_nosync_fp8_matches_oracle_and_sync_driver(n_sets):
    w = wl.WORKLOADS["chunk_fp8"].scaled(T=2048 + 37)
    x, idx, wts = wl.make(w)
    xd, idd, wd = x.cuda(), idx.cuda(), wts.cuda()
    err = ep.error_word()
    out = ep.dispatch_chunked_forward_nosync(xd, idd, wd, num_local_experts=w.E_local, num_ranks=w.P,
                                             chunks=w.chunks, fp8=True, n_sets=n_sets, err=err)
    ref = ep.dispatch_chunked_forward(xd, idd, wd, num_local_experts=w.E_local, num_ranks=w.P, chunks=w.chunks,
                                      fp8=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_equal("nosync == sync driver", bits16(out), bits16(ref))
    assert_combine_parity("chunked fp8 nosync", bits16(out),
                          _oracle_chunked(x, idx, wts, w.P, w.E_local, w.chunks, True))


@pytest.mark.parametrize("n_sets", [1, 2])
def test_chunked_nosync_bf16_python_local_kernel(n_sets):
    w = dataclasses.replace(wl.WORKLOADS["mid"].scaled(T=1500), chunks=5)
    x, idx, wts = wl.make(w)
    seen = []

    def identity(chunk, recv_x, recv_scale, send_idx, send_w, local_out, n_rows):
        seen.append(chunk)
        assert recv_scale is None and n_rows.numel() == 1 and n_rows.is_cuda
        local_out.copy_(recv_x)                      # rows past n_rows are never combined

    err = ep.error_word()
    out = ep.dispatch_chunked_forward_nosync(x.cuda(), idx.cuda(), wts.cuda(), num_local_experts=w.E_local,
                                             num_ranks=w.P, chunks=w.chunks, local_kernel=identity, n_sets=n_sets,
                                             err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert seen == list(range(w.chunks))
    assert_combine_parity("chunked bf16 nosync", bits16(out),
                          _oracle_chunked(x, idx, wts, w.P, w.E_local, w.chunks, False))


def test_chunked_nosync_graph_replays_new_inputs():
    w = wl.WORKLOADS["chunk_fp8"].scaled(T=1024 + 5)
    f = ep.ChunkedForward(w.T, w.K, w.H, num_ranks=w.P, num_local_experts=w.E_local, chunks=w.chunks, fp8=True,
                          n_sets=2)
    xs = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((w.T, w.K), dtype=torch.int64, device="cuda")
    ws_ = torch.empty((w.T, w.K), dtype=torch.float32, device="cuda")
    out = torch.empty_like(xs)
    err = ep.error_word()
    x0, i0, w0 = wl.make(w)
    xs.copy_(x0)
    ids.copy_(i0)
    ws_.copy_(w0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        f(xs, ids, ws_, out=out, err=err)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        f(xs, ids, ws_, out=out, err=err)
    torch.cuda.synchronize()
    for seed in (11, 12, 13):
        wi = dataclasses.replace(w, seed=seed)
        x, idx, wts = wl.make(wi)
        xs.copy_(x)
        ids.copy_(idx)
        ws_.copy_(wts)
        out.fill_(0)
        err.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_combine_parity(f"replay seed {seed}", bits16(out),
                              _oracle_chunked(x, idx, wts, w.P, w.E_local, w.chunks, True))


def test_chunked_nosync_capacity_is_flagged():
    w = wl.WORKLOADS["chunk_fp8"].scaled(T=1024)
    x, idx, wts = wl.make(w)
    f = ep.ChunkedForward(w.T, w.K, w.H, num_ranks=w.P, num_local_experts=w.E_local, chunks=w.chunks, fp8=True,
                          n_sets=2, max_rows=64)       # far fewer rows than any chunk uses
    err = ep.error_word()
    f(x.cuda(), idx.cuda(), wts.cuda(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ep.EP_ERR_CAPACITY
    for c in range(w.chunks):                         # the true counts are still reported
        assert int(f.t["rank_offsets"][c, w.P].item()) > 64
    assert int(f.t["token_pos"].max().item()) < 64    # nothing placed past the capacity


def test_chunked_nosync_empty():
    f = ep.ChunkedForward(0, 8, 256, num_ranks=4, num_local_experts=2, chunks=3, fp8=True, n_sets=2)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 8), dtype=torch.int64, device="cuda")
    wts = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    err = ep.error_word()
    out = f(x, idx, wts, err=err)
    torch.cuda.synchronize()
    assert out.shape == (0, 256) and int(err.item()) == 0
    assert int(f.t["rank_offsets"].abs().sum().item()) == 0


def test_chunked_nosync_full_size_sampled():
    w = wl.WORKLOADS["chunk_fp8"]
    x, idx, wts = wl.make(w)
    err = ep.error_word()
    out = ep.dispatch_chunked_forward_nosync(x.cuda(), idx.cuda(), wts.cuda(), num_local_experts=w.E_local,
                                             num_ranks=w.P, chunks=w.chunks, fp8=True, n_sets=2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    outb = bits16(out)
    g = np.random.Generator(np.random.PCG64(322))
    for t in np.sort(g.choice(w.T, size=64, replace=False)).tolist():
        r = oracle.send_path(x[t:t + 1], idx[t:t + 1], wts[t:t + 1], None, w.P, w.E_local)
        lay = r["layout"]
        q, sc = oracle.dispatch_fp8(x[t:t + 1], lay["send_token_idx"])
        want = oracle.combine(oracle.local_expert_fp8(q, sc, lay["send_idx"], lay["send_w"]), lay["token_pos"])
        assert_combine_parity(f"token {t}", outb[t:t + 1], want)


# ----------------------------------------- items with more sources than buffers --
# With H = 7168 the combine's shared-memory ring holds 8 rows; these cases give
# every token 16 or 32 source rows, so each item reuses ring buffers within
# itself (the producer must issue it in rounds).
@pytest.mark.parametrize("T,K,P", [(600, 16, 16), (300, 32, 32)])
def test_combine_items_longer_than_the_ring(T, K, P):
    H, E_local = 7168, 1
    idx, wts = _routing(T, K, P * E_local, seed=T + K, frac_unrouted=0.0)
    x = _randn(T, H, 5)
    o = oracle.send_path(x, idx, wts, None, P, E_local)
    assert int((o["layout"]["token_pos"] >= 0).sum(1).min()) == P      # every token hits every rank
    y = _randn(o["layout"]["n"], H, 6)
    o["out"] = oracle.combine(y, o["layout"]["token_pos"])
    g = gpu_send_path(x, idx, wts, y, P, E_local)
    compare_send_path(x, idx, wts, y, P, E_local, g, o)


def test_batched_combine_items_longer_than_the_ring():
    T, H, K, E, E_local, rank, M = 300, 7168, 32, 32, 32, 0, 400
    idx, wts = _routing(T, K, E, seed=77, frac_unrouted=0.0)           # all 32 experts local
    x = _randn(T, H, 7)
    o = oracle.batched_prepare(x, idx, E, E_local, rank, M)
    w = wl.Workload("long", T=T, H=H, E=E, K=K, P=1, routing="uniform", rank=rank, max_num_tokens=M)
    y = wl.batched_expert_outputs(w, o["tokens_per_expert"])
    want = oracle.batched_combine(y, idx, wts, o["slot"], E_local, rank)
    dev = "cuda"
    r = ep.batched_prepare(x.to(dev), idx.to(dev), E, E_local, rank, M)
    got = ep.batched_combine(y.to(dev), idx.to(dev), wts.to(dev), r["slot"], rank, err=r["err"])
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    assert_combine_parity("batched combine", bits16(got), want)


def test_batched_prepare_many_local_experts():
    # E_local = 128 > 64 takes the two-kernel slot path instead of the fused one
    T, H, K, E, E_local, rank, M = 700, 64, 8, 256, 128, 1, 300
    idx, wts = _routing(T, K, E, seed=31, dup=True)
    x = _randn(T, H, 8)
    o = oracle.batched_prepare(x, idx, E, E_local, rank, M)
    dev = "cuda"
    r = ep.batched_prepare(x.to(dev), idx.to(dev), E, E_local, rank, M)
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o["tokens_per_expert"])
    assert_equal("slot", np_(r["slot"]), o["slot"])


# ----------------------------------- route + dispatch as one no-sync call --
@pytest.mark.parametrize("name,fp8", [("mid", False), ("large", False), ("large", True), ("chunk_fp8", True)])
def test_dispatch_nosync_matches_oracle(name, fp8):
    w = wl.WORKLOADS[name]
    if name == "chunk_fp8":
        w = w.scaled(T=3000)
    x, idx, wts = wl.make(w)
    dev = "cuda"
    T, K, P, El, H = w.T, w.K, w.P, w.E_local, w.H
    W = T * min(K, P)
    i32 = torch.int32
    outs = dict(dest=torch.empty((T, K), dtype=i32, device=dev),
                is_in_rank=torch.empty((T, P), dtype=torch.uint8, device=dev),
                send_counts=torch.empty(P, dtype=i32, device=dev),
                rank_offsets=torch.empty(P + 1, dtype=i32, device=dev),
                send_token_idx=torch.empty(W, dtype=i32, device=dev),
                send_rank=torch.empty(W, dtype=i32, device=dev),
                send_idx=torch.empty((W, K), dtype=torch.int64, device=dev),
                send_w=torch.empty((W, K), dtype=torch.float32, device=dev),
                token_pos=torch.empty((T, P), dtype=i32, device=dev))
    recv = torch.empty((W, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    scale = torch.empty((W, H // 128), dtype=torch.float32, device=dev) if fp8 else None
    err = ep.error_word()
    ep.ep_dispatch_nosync(x.to(dev), idx.to(dev), wts.to(dev), T, K, H, P, El, W, int(fp8), outs["dest"],
                          outs["is_in_rank"], outs["send_counts"], outs["rank_offsets"], None, outs["send_token_idx"],
                          outs["send_rank"], outs["send_idx"], outs["send_w"], outs["token_pos"], recv, scale,
                          ep.workspace(T, K, P, El), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = oracle.send_path(x, idx, wts, None, P, El)
    ol = o["layout"]
    N = ol["n"]
    assert int(outs["rank_offsets"][P].item()) == N
    for k in ("send_token_idx", "send_rank", "send_idx"):
        assert_equal(k, np_(outs[k])[:N], ol[k])
    assert_equal("token_pos", np_(outs["token_pos"]), ol["token_pos"])
    if fp8:
        q, sc = oracle.dispatch_fp8(x, ol["send_token_idx"])
        assert_equal("fp8 codes", np_(recv)[:N], q)
        assert_equal("fp8 scales (bits)", np_(scale)[:N].view(np.uint32), sc.view(np.uint32))
    else:
        assert_equal("recv_x", bits16(recv)[:N], o["recv_x"])
