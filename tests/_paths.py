"""Shared drivers for the GPU parity tests: run one workload through the CUDA
library (via the C ABI binding) and through the CPU oracle on the same seeded
inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def routing_inputs(T, K, E, seed, frac_unrouted=0.1, dup=False):
    """Seeded top-k ids (distinct per token, or with duplicates) with a share
    of masked (-1) slots, and uniform weights (0 where masked)."""
    g = np.random.Generator(np.random.PCG64(seed))
    idx = (g.integers(0, E, size=(T, K)) if dup else np.argsort(g.random((T, E)), 1)[:, :K]).astype(np.int64)
    idx[g.random((T, K)) < frac_unrouted] = -1
    w = g.random((T, K)).astype(np.float32)
    w[idx < 0] = 0
    return torch.from_numpy(idx), torch.from_numpy(w)


def randn_bf16(T, H, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return torch.from_numpy(g.standard_normal((T, H), dtype=np.float32)).to(torch.bfloat16)


def assert_equal(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches, first at {i}: got {got[i]} want {want[i]}")


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (monotone integer mapping)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))
    return np.abs(key(a_bits) - key(b_bits))


def assert_combine_parity(name, got_bits, want_bits, max_ulp=0):
    """The combine target is within 1 bf16 ulp of the fp32-accumulated oracle;
    both sides add in the same order with the same roundings, so the claim
    checked here is max_ulp (0 = bit-exact unless a test says otherwise)."""
    d = bf16_ulp_distance(got_bits, want_bits)
    assert d.max(initial=0) <= max_ulp, f"{name}: max ulp distance {d.max()} > {max_ulp} ({int((d > 0).sum())} differ)"


def gpu_send_path(x, idx, w, y, P, E_local, fp8=False, out_f32=False, chunk_bounds=None):
    """counts -> (one D2H of the counts) -> layout -> dispatch -> combine on the GPU."""
    dev = "cuda"
    xd, idd, wd = x.to(dev), idx.to(dev), w.to(dev)
    err = ep.error_word()
    c = ep.compute_send_counts(idd, P, E_local, err=err)
    N = int(c["send_counts"].sum().item())
    lay = ep.build_send_layout(idd, wd, c["dest"], c["is_in_rank"], N, E_local, err=err)
    if fp8:
        recv = ep.dispatch_rows(xd, lay["token_pos"], N, fp8=True, err=err)
    else:
        recv = ep.dispatch_rows(xd, lay["token_pos"], N, err=err)
    out = None
    if y is not None:
        yd = y[:N].to(dev) if isinstance(y, torch.Tensor) else y
        out = ep.combine_rows(yd, lay["token_pos"], out_dtype=torch.float32 if out_f32 else torch.bfloat16,
                              err=err)
    torch.cuda.synchronize()
    return dict(counts=c, layout=lay, recv=recv, out=out, N=N, err=int(err.item()))


def compare_send_path(x, idx, w, y, P, E_local, g, o, check_out=True):
    """g = gpu_send_path result, o = oracle.send_path result."""
    oc, ol = o["counts"], o["layout"]
    assert g["err"] == 0, ep.EPError(g["err"])
    assert_equal("dest", np_(g["counts"]["dest"]), oc["dest"])
    assert_equal("is_in_rank", np_(g["counts"]["is_in_rank"]), oc["is_in_rank"])
    assert_equal("send_counts", np_(g["counts"]["send_counts"])[0], oc["send_counts"])
    assert_equal("rank_offsets", np_(g["counts"]["rank_offsets"])[0],
                 np.concatenate([[0], np.cumsum(oc["send_counts"])]))
    assert_equal("tokens_per_expert", np_(g["counts"]["tokens_per_expert"]), oc["tokens_per_expert"])
    assert g["N"] == ol["n"]
    for k in ("send_token_idx", "send_rank", "send_idx", "token_pos"):
        assert_equal(k, np_(g["layout"][k]), ol[k])
    assert_equal("send_w(bits)", np_(g["layout"]["send_w"]).view(np.uint32), ol["send_w"].view(np.uint32))
    assert_equal("recv_x", bits16(g["recv"]), o["recv_x"])
    if check_out and g["out"] is not None:
        assert_combine_parity("combine", bits16(g["out"]), o["out"])
