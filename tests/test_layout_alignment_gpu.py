"""The send layout written into buffers that have only their elements' natural
alignment (the C ABI promises no more for send_idx, send_w, is_in_rank):
send_idx 8-byte, send_w 4-byte and is_in_rank 1-byte aligned.  The kernels
take wider stores only where the caller's pointers allow them, so these
layouts must equal the oracle bit for bit like the aligned ones, on both the
host-synchronising path (ep_compute_send_counts + ep_build_send_layout) and
the single-launch route (ep_route_nosync)."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_equal, np_, routing_inputs

pytestmark = pytest.mark.gpu


def _buf(shape, dtype, offset):
    """A contiguous tensor of `shape` starting `offset` elements into a fresh
    allocation (the allocation itself is 256-byte aligned)."""
    n = int(np.prod(shape))
    return torch.empty(n + offset, dtype=dtype, device="cuda")[offset:].view(shape)


def _check_layout(o, N, dest, iir, sc, ro, sti, sr, si, sw, tp):
    oc, ol = o["counts"], o["layout"]
    assert_equal("dest", np_(dest), oc["dest"])
    assert_equal("is_in_rank", np_(iir), oc["is_in_rank"])
    assert_equal("send_counts", np_(sc).reshape(-1), oc["send_counts"])
    assert_equal("rank_offsets", np_(ro).reshape(-1)[: len(oc["send_counts"]) + 1],
                 np.concatenate([[0], np.cumsum(oc["send_counts"])]))
    assert_equal("send_token_idx", np_(sti)[:N], ol["send_token_idx"])
    assert_equal("send_rank", np_(sr)[:N], ol["send_rank"])
    assert_equal("send_idx", np_(si)[:N], ol["send_idx"])
    assert_equal("send_w (bits)", np_(sw)[:N].view(np.uint32), ol["send_w"].view(np.uint32))
    assert_equal("token_pos", np_(tp), ol["token_pos"])


@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("T,K,P,El", [(3000, 8, 8, 4), (1777, 6, 4, 8), (2049, 4, 16, 2), (999, 2, 8, 2),
                                      (513, 5, 8, 4)])
def test_host_sync_layout_with_natural_alignment(T, K, P, El, offset):
    idx, wts = routing_inputs(T, K, P * El, T + K, 0.1)
    o = oracle.send_path(torch.zeros((T, 8), dtype=torch.bfloat16), idx, wts, None, P, El)
    N = o["layout"]["n"]
    dev = "cuda"
    idd, wd = idx.to(dev), wts.to(dev)
    err = ep.error_word()
    dest = _buf((T, K), torch.int32, offset)
    iir = _buf((T, P), torch.uint8, offset)
    sc = _buf((P,), torch.int32, offset)
    ro = _buf((P + 1,), torch.int32, offset)
    ws = ep.workspace(T, K, P, El)
    ep.ep_compute_send_counts(idd, T, K, P, El, None, 1, dest, iir, sc, ro, None, ws, err)
    sti = _buf((N,), torch.int32, offset)
    sr = _buf((N,), torch.int32, offset)
    si = _buf((N, K), torch.int64, offset)
    sw = _buf((N, K), torch.float32, offset)
    tp = _buf((T, P), torch.int32, offset)
    ep.ep_build_send_layout(idd, wd, dest, iir, T, K, P, El, N, sti, sr, si, sw, tp, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
    _check_layout(o, N, dest, iir, sc, ro, sti, sr, si, sw, tp)


@pytest.mark.parametrize("offset", [1, 3])
@pytest.mark.parametrize("T,K,P,El", [(3000, 8, 8, 4), (1777, 6, 4, 8), (2049, 4, 16, 2), (513, 5, 8, 4)])
def test_route_nosync_with_natural_alignment(T, K, P, El, offset):
    idx, wts = routing_inputs(T, K, P * El, T + 7 * K, 0.1)
    o = oracle.send_path(torch.zeros((T, 8), dtype=torch.bfloat16), idx, wts, None, P, El)
    N = o["layout"]["n"]
    W = T * min(K, P)
    dev = "cuda"
    err = ep.error_word()
    dest = _buf((T, K), torch.int32, offset)
    iir = _buf((T, P), torch.uint8, offset)
    sc = _buf((P,), torch.int32, offset)
    ro = _buf((P + 1,), torch.int32, offset)
    sti = _buf((W,), torch.int32, offset)
    sr = _buf((W,), torch.int32, offset)
    si = _buf((W, K), torch.int64, offset)
    sw = _buf((W, K), torch.float32, offset)
    tp = _buf((T, P), torch.int32, offset)
    ws = ep.workspace(T, K, P, El)
    ep.ep_route_nosync(idx.to(dev), wts.to(dev), T, K, P, El, W, dest, iir, sc, ro, None, sti, sr, si, sw, tp, ws,
                       err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
    assert int(ro[P].item()) == N
    _check_layout(o, N, dest, iir, sc, ro, sti, sr, si, sw, tp)
