"""ep_compute_send_counts_noalloc: the counts entry point for callers that
cannot allocate device memory (an engine that plans all device memory before
it runs and forbids allocation during its enqueue step).  It keeps its
scratch in the library's own fixed device array instead of a caller
workspace.

Its results must equal the oracle's counts and those of
ep_compute_send_counts with a caller workspace, call after call, whatever the
previous call left in the shared array, and a call must not change the
device's free memory.  This file is collected last on purpose; it builds and
loads the library itself, so it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _outputs(T, K, P, E_local, C, dev, with_tpe):
    return dict(dest=torch.full((T, K), -7, dtype=torch.int32, device=dev),
                is_in_rank=torch.full((T, P), 9, dtype=torch.uint8, device=dev),
                send_counts=torch.full((C, P), -7, dtype=torch.int32, device=dev),
                rank_offsets=torch.full((C, P + 1), -7, dtype=torch.int32, device=dev),
                tokens_per_expert=torch.full((P * E_local,), -7, dtype=torch.int32, device=dev) if with_tpe
                else None)


def _run(noalloc, idx, P, E_local, bounds, with_tpe=True, free_bytes=None):
    """One counts call; with free_bytes (a list) the device's free memory is
    read right before the call and right after it has finished."""
    T, K = idx.shape
    C = len(bounds) - 1 if bounds is not None else 1
    o = _outputs(T, K, P, E_local, C, idx.device, with_tpe)
    err = ep.error_word()
    ws = None if noalloc else ep.workspace(T, K, P, E_local, C)
    torch.cuda.synchronize()
    if free_bytes is not None:
        free_bytes.append(torch.cuda.mem_get_info()[0])
    if noalloc:
        ep.ep_compute_send_counts_noalloc(idx, T, K, P, E_local, bounds, C, o["dest"], o["is_in_rank"],
                                          o["send_counts"], o["rank_offsets"], o["tokens_per_expert"], err)
    else:
        ep.ep_compute_send_counts(idx, T, K, P, E_local, bounds, C, o["dest"], o["is_in_rank"],
                                  o["send_counts"], o["rank_offsets"], o["tokens_per_expert"], ws, err)
    torch.cuda.synchronize()
    if free_bytes is not None:
        free_bytes.append(torch.cuda.mem_get_info()[0])
    o["err"] = int(err.item())
    return o


def _same(a, b):
    for k in ("dest", "is_in_rank", "send_counts", "rank_offsets", "tokens_per_expert"):
        if a[k] is None or b[k] is None:
            assert a[k] is None and b[k] is None, k
        else:
            assert torch.equal(a[k], b[k]), k
    assert a["err"] == b["err"] == 0


def _matches_oracle(g, idx_cpu, P, E_local, bounds):
    """axolotl compute_send_counts: dest, is_in_rank and tokens_per_expert over
    all tokens; send_counts of each chunk from the oracle run on that chunk's
    tokens alone, rank_offsets their exclusive prefix per chunk."""
    o = oracle.compute_send_counts(idx_cpu, P, E_local)
    assert o["err"] == 0
    np.testing.assert_array_equal(g["dest"].cpu().numpy(), o["dest"])
    np.testing.assert_array_equal(g["is_in_rank"].cpu().numpy(), o["is_in_rank"])
    if g["tokens_per_expert"] is not None:
        np.testing.assert_array_equal(g["tokens_per_expert"].cpu().numpy(), o["tokens_per_expert"])
    b = [0, idx_cpu.shape[0]] if bounds is None else list(bounds)
    want = np.stack([oracle.compute_send_counts(idx_cpu[b[c]:b[c + 1]], P, E_local,
                                                with_tokens_per_expert=False)["send_counts"]
                     for c in range(len(b) - 1)])
    np.testing.assert_array_equal(g["send_counts"].cpu().numpy(), want)
    offs = np.concatenate([np.zeros((want.shape[0], 1), np.int64), np.cumsum(want, axis=1)], axis=1)
    np.testing.assert_array_equal(g["rank_offsets"].cpu().numpy(), offs.astype(np.int32))


def test_noalloc_counts_match_the_oracle_and_the_workspace_entry_on_consecutive_calls():
    dev = "cuda"
    # different problems back to back: each call runs on whatever the one
    # before it left in the shared array
    big = wl.WORKLOADS["chunk_fp8"]
    idx_big_cpu, _ = wl.routing(big)
    idx_big = idx_big_cpu.to(dev)
    bounds = ep.chunk_bounds(big.T, big.chunks)
    small = wl.WORKLOADS["mid"]
    idx_small_cpu, _ = wl.routing(small)
    idx_small = idx_small_cpu.to(dev)

    first = _run(True, idx_big, big.P, big.E_local, bounds)
    _matches_oracle(first, idx_big_cpu, big.P, big.E_local, bounds)
    _same(first, _run(False, idx_big, big.P, big.E_local, bounds))

    second = _run(True, idx_small, small.P, small.E_local, None)
    _matches_oracle(second, idx_small_cpu, small.P, small.E_local, None)
    _same(second, _run(False, idx_small, small.P, small.E_local, None))

    # without tokens_per_expert the per-expert partials are skipped
    third = _run(True, idx_big, big.P, big.E_local, bounds, with_tpe=False)
    _matches_oracle(third, idx_big_cpu, big.P, big.E_local, bounds)
    _same(third, _run(False, idx_big, big.P, big.E_local, bounds, with_tpe=False))

    again = _run(True, idx_small, small.P, small.E_local, None)
    _same(again, second)


def test_noalloc_call_leaves_free_device_memory_unchanged():
    dev = "cuda"
    w = wl.WORKLOADS["large"]
    idx_cpu, _ = wl.routing(w)
    idx = idx_cpu.to(dev)
    _run(True, idx, w.P, w.E_local, None)          # loads the kernels and sets up the array's address
    free = []
    for with_tpe in (True, False, True):
        g = _run(True, idx, w.P, w.E_local, None, with_tpe=with_tpe, free_bytes=free)
        assert g["err"] == 0
    assert len(set(free)) == 1, f"free device memory changed across the calls: {free}"
    _matches_oracle(g, idx_cpu, w.P, w.E_local, None)


def test_noalloc_rejects_sizes_beyond_its_array_and_bad_arguments():
    lib = ep.load()
    call = lambda T, K, P, El, bounds, C: lib.ep_compute_send_counts_noalloc(
        None, T, K, P, El, bounds, C, None, None, None, None, None, None, ctypes.c_void_p(0))
    # 2^22 tokens over 64 ranks need far more than the fixed array holds:
    # rejected on the host, before any pointer is touched
    assert call(1 << 22, 8, 64, 128, None, 1) == ep.EP_ERR_UNSUPPORTED
    assert call(-1, 8, 8, 32, None, 1) == ep.EP_ERR_INVALID_ARG
    assert call(16, 8, 0, 32, None, 1) == ep.EP_ERR_INVALID_ARG
    bad = (ctypes.c_int64 * 3)(0, 9, 8)              # decreasing chunk bounds
    assert call(8, 2, 2, 2, bad, 2) == ep.EP_ERR_INVALID_ARG
