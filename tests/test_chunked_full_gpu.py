"""The chunked fp8 workload at full size (T = 32768, H = 7168, E = 256, K = 8,
P = 16, 4 chunks), every buffer compared element by element with the oracle,
through each chunked driver: the host-sync driver, the no-sync driver with one
and with two row sets, and the two-set driver replayed from a CUDA graph.

axolotl integrations.expert_parallel.torch_dispatch, dispatch_chunked_forward
(one count pass over all chunks, then per chunk layout -> dispatch -> local
kernel -> combine) and chunk_bounds; the dispatch carries the fp8 payload of
NeMo uccl_ep.buffer, Buffer.dispatch; the local kernel is the workload's
synthetic expert (expert l maps a token to its dequantised row times
1 + l/64, weighted and summed over K).

The oracle runs once per chunk for the whole module (about half a minute per
chunk, the four chunks in threads: the C oracle releases the GIL).  To see
every chunk's rows, the local kernel given to a driver is a wrapper that
copies the chunk's rows, calls the library's own synthetic expert through its
C callback with the driver's arguments, and copies the expert's output; the
drivers are also run with the library's callback passed directly, and their
outputs must be the same bits."""
import concurrent.futures as cf
import dataclasses

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.WORKLOADS["chunk_fp8"]


def _oracle_chunk(x, idx, wts, s, e):
    oc = oracle.compute_send_counts(idx[s:e], W.P, W.E_local, with_tokens_per_expert=False)
    ol = oracle.build_send_layout(idx[s:e], wts[s:e], oc["dest"], oc["is_in_rank"], W.E_local)
    q, sc = oracle.dispatch_fp8(x[s:e], ol["send_token_idx"])
    local = oracle.local_expert_fp8(q, sc, ol["send_idx"], ol["send_w"])
    out = oracle.combine(local, ol["token_pos"])
    return dict(send_counts=oc["send_counts"], n=ol["n"], send_token_idx=ol["send_token_idx"],
                send_rank=ol["send_rank"], send_idx=ol["send_idx"], send_w=ol["send_w"].view(np.int32),
                token_pos=ol["token_pos"], q=q, scale=sc.view(np.int32), local=local.view(np.int16),
                out=out.view(np.int16))


@pytest.fixture(scope="module")
def full():
    x, idx, wts = wl.make(W)
    b = [int(v) for v in oracle.chunk_bounds(W.T, W.chunks)]
    assert b == ep.chunk_bounds(W.T, W.chunks)
    whole = oracle.compute_send_counts(idx, W.P, W.E_local, with_tokens_per_expert=False)
    with cf.ThreadPoolExecutor(W.chunks) as ex:
        chunks = list(ex.map(lambda c: _oracle_chunk(x, idx, wts, b[c], b[c + 1]), range(W.chunks)))
    dev = "cuda"
    want = [{k: (torch.from_numpy(np.ascontiguousarray(v)).to(dev) if isinstance(v, np.ndarray) else v)
             for k, v in c.items()} for c in chunks]
    ro = np.concatenate([np.zeros((W.chunks, 1), np.int64),
                         np.cumsum(np.stack([c["send_counts"] for c in chunks]), axis=1)], axis=1)
    return dict(x=x.to(dev), idx=idx.to(dev), wts=wts.to(dev), bounds=b, chunks=want,
                dest=torch.from_numpy(whole["dest"]).to(dev),
                is_in_rank=torch.from_numpy(whole["is_in_rank"]).to(dev),
                send_counts=torch.from_numpy(np.stack([c["send_counts"] for c in chunks])).to(dev),
                rank_offsets=torch.from_numpy(ro.astype(np.int32)).to(dev),
                out=torch.cat([c["out"] for c in want]))


def _eq(name, got, want):
    """Element-by-element equality on the device; the first mismatch is reported."""
    assert got.shape == want.shape, (name, tuple(got.shape), tuple(want.shape))
    if not torch.equal(got, want):
        bad = (got != want).nonzero()
        i = tuple(bad[0].tolist())
        raise AssertionError(f"{name}: {bad.shape[0]} mismatches, first at {i}: got {got[i].item()} "
                             f"want {want[i].item()}")


def _i16(t):
    return t.contiguous().view(torch.int16)


def _i32(t):
    return t.contiguous().view(torch.int32)


def _check_routing(f, name, dest, is_in_rank, send_counts, rank_offsets, token_pos):
    _eq(f"{name} dest", dest, f["dest"])
    _eq(f"{name} is_in_rank", is_in_rank, f["is_in_rank"])
    _eq(f"{name} send_counts", send_counts, f["send_counts"])
    _eq(f"{name} rank_offsets", rank_offsets, f["rank_offsets"])
    for c in range(W.chunks):
        s, e = f["bounds"][c], f["bounds"][c + 1]
        _eq(f"{name} chunk {c} token_pos", token_pos[s:e], f["chunks"][c]["token_pos"])


def _check_rows(name, c, want, q, scale, send_idx, send_w, local, send_token_idx=None, send_rank=None):
    """The first n rows of a chunk's buffers (the rest are worst-case room)."""
    n = want["n"]
    _eq(f"{name} chunk {c} fp8 codes", q[:n], want["q"])
    _eq(f"{name} chunk {c} fp8 scales (bits)", _i32(scale[:n]), want["scale"])
    _eq(f"{name} chunk {c} send_idx", send_idx[:n], want["send_idx"])
    _eq(f"{name} chunk {c} send_w (bits)", _i32(send_w[:n]), want["send_w"])
    _eq(f"{name} chunk {c} synthetic expert", _i16(local[:n]), want["local"])
    if send_token_idx is not None:
        _eq(f"{name} chunk {c} send_token_idx", send_token_idx[:n], want["send_token_idx"])
    if send_rank is not None:
        _eq(f"{name} chunk {c} send_rank", send_rank[:n], want["send_rank"])


def test_host_sync_driver_full_size_every_buffer(full):
    native = ep.ep_local_expert_fp8_callback()
    err = ep.error_word()
    snaps = []

    def expert(chunk, recv_x, recv_scale, send_idx, send_w, local_out):
        s = dict(q=recv_x.clone(), scale=recv_scale.clone(), send_idx=send_idx.clone(), send_w=send_w.clone())
        rc = native(None, chunk, recv_x.shape[0], W.K, W.H, recv_x.data_ptr(), recv_scale.data_ptr(),
                    send_idx.data_ptr(), send_w.data_ptr(), local_out.data_ptr(), err.data_ptr(),
                    torch.cuda.current_stream().cuda_stream)
        if rc != ep.EP_OK:
            raise ep.EPError(rc, "synthetic expert")
        s["local"] = local_out.clone()
        snaps.append(s)

    keep = {}
    out = ep.dispatch_chunked_forward(full["x"], full["idx"], full["wts"], num_local_experts=W.E_local,
                                      num_ranks=W.P, chunks=W.chunks, fp8=True, local_kernel=expert, err=err,
                                      keep=keep)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert len(snaps) == W.chunks
    _check_routing(full, "host-sync", keep["dest"], keep["is_in_rank"], keep["send_counts"], keep["rank_offsets"],
                   keep["token_pos"])
    for c, s in enumerate(snaps):
        want = full["chunks"][c]
        assert s["q"].shape[0] == want["n"]            # the host-sync driver gives the exact row count
        _check_rows("host-sync", c, want, s["q"], s["scale"], s["send_idx"], s["send_w"], s["local"])
    last = full["chunks"][-1]                          # the row buffers still hold the last chunk
    _eq("host-sync last chunk send_token_idx", keep["send_token_idx"][:last["n"]], last["send_token_idx"])
    _eq("host-sync last chunk send_rank", keep["send_rank"][:last["n"]], last["send_rank"])
    _eq("host-sync combined output (bits)", _i16(out), full["out"])

    # the same driver with the library's callback passed directly
    err2 = ep.error_word()
    out2 = ep.dispatch_chunked_forward(full["x"], full["idx"], full["wts"], num_local_experts=W.E_local,
                                       num_ranks=W.P, chunks=W.chunks, fp8=True, err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    _eq("host-sync (native expert) combined output (bits)", _i16(out2), full["out"])


@pytest.mark.parametrize("n_sets", [1, 2])
def test_nosync_driver_full_size_every_buffer(full, n_sets):
    native = ep.ep_local_expert_fp8_dev_callback()
    err = ep.error_word()
    snaps = []
    f = None

    def expert(chunk, recv_x, recv_scale, send_idx, send_w, local_out, n_rows):
        st = f.sets[chunk % f.n_sets]
        s = dict(q=recv_x.clone(), scale=recv_scale.clone(), send_idx=send_idx.clone(), send_w=send_w.clone(),
                 send_token_idx=st["send_token_idx"].clone(), send_rank=st["send_rank"].clone(),
                 n_rows=n_rows.clone())
        rc = native(None, chunk, recv_x.shape[0], n_rows.data_ptr(), W.K, W.H, recv_x.data_ptr(),
                    recv_scale.data_ptr(), send_idx.data_ptr(), send_w.data_ptr(), local_out.data_ptr(),
                    err.data_ptr(), torch.cuda.current_stream().cuda_stream)
        if rc != ep.EP_OK:
            raise ep.EPError(rc, "synthetic expert")
        s["local"] = local_out.clone()
        snaps.append(s)

    f = ep.ChunkedForward(W.T, W.K, W.H, num_ranks=W.P, num_local_experts=W.E_local, chunks=W.chunks, fp8=True,
                          n_sets=n_sets, local_kernel=expert)
    out = f(full["x"], full["idx"], full["wts"], err=err)
    torch.cuda.synchronize()
    name = f"no-sync {n_sets} set(s)"
    assert int(err.item()) == 0
    assert len(snaps) == W.chunks
    _check_routing(full, name, f.t["dest"], f.t["is_in_rank"], f.t["send_counts"], f.t["rank_offsets"],
                   f.t["token_pos"])
    for c, s in enumerate(snaps):
        want = full["chunks"][c]
        assert int(s["n_rows"].item()) == want["n"]
        _check_rows(name, c, want, s["q"], s["scale"], s["send_idx"], s["send_w"], s["local"],
                    s["send_token_idx"], s["send_rank"])
    _eq(f"{name} combined output (bits)", _i16(out), full["out"])

    # the same driver with the library's callback passed directly
    g = ep.ChunkedForward(W.T, W.K, W.H, num_ranks=W.P, num_local_experts=W.E_local, chunks=W.chunks, fp8=True,
                          n_sets=n_sets)
    err2 = ep.error_word()
    out2 = g(full["x"], full["idx"], full["wts"], err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    _eq(f"{name} (native expert) combined output (bits)", _i16(out2), full["out"])
    _check_routing(full, f"{name} (native expert)", g.t["dest"], g.t["is_in_rank"], g.t["send_counts"],
                   g.t["rank_offsets"], g.t["token_pos"])


def test_nosync_driver_graph_replay_full_size(full):
    # captured on other inputs, replayed on the workload's: every output is
    # recomputed by the replay
    f = ep.ChunkedForward(W.T, W.K, W.H, num_ranks=W.P, num_local_experts=W.E_local, chunks=W.chunks, fp8=True,
                          n_sets=2)
    xs, ids, ws_ = (torch.empty_like(full[k]) for k in ("x", "idx", "wts"))
    out = torch.empty_like(xs)
    err = ep.error_word()
    x0, i0, w0 = wl.make(dataclasses.replace(W, seed=W.seed + 1))
    xs.copy_(x0)
    ids.copy_(i0)
    ws_.copy_(w0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        f(xs, ids, ws_, out=out, err=err)              # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        f(xs, ids, ws_, out=out, err=err)
    torch.cuda.synchronize()
    xs.copy_(full["x"])
    ids.copy_(full["idx"])
    ws_.copy_(full["wts"])
    out.fill_(0)
    err.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _check_routing(full, "graph replay", f.t["dest"], f.t["is_in_rank"], f.t["send_counts"], f.t["rank_offsets"],
                   f.t["token_pos"])
    _eq("graph replay combined output (bits)", _i16(out), full["out"])
    # the two row sets hold the last two chunks
    for c in (W.chunks - 2, W.chunks - 1):
        st = f.sets[c % 2]
        _check_rows("graph replay", c, full["chunks"][c], st["recv_x"], st["recv_scale"], st["send_idx"],
                    st["send_w"], st["local_out"], st["send_token_idx"], st["send_rank"])
