"""ep_compute_send_counts_noalloc: the counts entry point for callers that
cannot allocate device memory (an engine that plans all device memory before
it runs and forbids allocation during its enqueue step, or code running while
a CUDA graph is captured).  It keeps its scratch in the library's own fixed
device array instead of a caller workspace.

Its results must equal those of ep_compute_send_counts with a caller
workspace, call after call, whatever the previous call left in the shared
array.  This file is collected last on purpose; it builds and loads the
library itself, so it also passes alone in a fresh process."""
import ctypes

import pytest
import torch

import combine_send_counts_gb300 as ep
from combine_send_counts_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _outputs(T, K, P, E_local, C, dev):
    return dict(dest=torch.full((T, K), -7, dtype=torch.int32, device=dev),
                is_in_rank=torch.full((T, P), 9, dtype=torch.uint8, device=dev),
                send_counts=torch.full((C, P), -7, dtype=torch.int32, device=dev),
                rank_offsets=torch.full((C, P + 1), -7, dtype=torch.int32, device=dev),
                tokens_per_expert=torch.full((P * E_local,), -7, dtype=torch.int32, device=dev))


def _run(noalloc, idx, P, E_local, bounds):
    T, K = idx.shape
    C = len(bounds) - 1 if bounds is not None else 1
    o = _outputs(T, K, P, E_local, C, idx.device)
    err = ep.error_word()
    if noalloc:
        ep.ep_compute_send_counts_noalloc(idx, T, K, P, E_local, bounds, C, o["dest"], o["is_in_rank"],
                                          o["send_counts"], o["rank_offsets"], o["tokens_per_expert"], err)
    else:
        ws = ep.workspace(T, K, P, E_local, C)
        ep.ep_compute_send_counts(idx, T, K, P, E_local, bounds, C, o["dest"], o["is_in_rank"],
                                  o["send_counts"], o["rank_offsets"], o["tokens_per_expert"], ws, err)
    torch.cuda.synchronize()
    o["err"] = int(err.item())
    return o


def _same(a, b):
    for k in ("dest", "is_in_rank", "send_counts", "rank_offsets", "tokens_per_expert"):
        assert torch.equal(a[k], b[k]), k
    assert a["err"] == b["err"] == 0


def test_noalloc_counts_match_the_workspace_entry_point_on_consecutive_calls():
    dev = "cuda"
    # two different problems back to back: the second call runs on whatever
    # the first one left in the shared array
    big = wl.WORKLOADS["chunk_fp8"]
    idx_big, _ = wl.routing(big)
    idx_big = idx_big.to(dev)
    bounds = ep.chunk_bounds(big.T, big.chunks)
    small = wl.WORKLOADS["mid"]
    idx_small, _ = wl.routing(small)
    idx_small = idx_small.to(dev)

    first = _run(True, idx_big, big.P, big.E_local, bounds)
    _same(first, _run(False, idx_big, big.P, big.E_local, bounds))
    second = _run(True, idx_small, small.P, small.E_local, None)
    _same(second, _run(False, idx_small, small.P, small.E_local, None))
    again = _run(True, idx_big, big.P, big.E_local, bounds)
    _same(again, first)


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = ep.load()
    # 2^22 tokens over 64 ranks need far more than the fixed array holds:
    # rejected on the host, before any pointer is touched
    rc = lib.ep_compute_send_counts_noalloc(None, 1 << 22, 8, 64, 128, None, 1, None, None, None, None, None,
                                            None, ctypes.c_void_p(0))
    assert rc == ep.EP_ERR_UNSUPPORTED
