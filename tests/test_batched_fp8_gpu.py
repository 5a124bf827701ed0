"""GPU parity of the fp8 expert-batched prepare (vLLM BatchedPrepareAndFinalize
.prepare, quantised branch; NeMo uccl_ep.buffer Buffer.low_latency_dispatch
scale formats) against the oracle: codes, scales in every layout, slots and
tokens_per_expert bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from combine_send_counts_gb300 import workloads as wl
from _paths import assert_equal, np_, routing_inputs

pytestmark = pytest.mark.gpu

COMBOS = [(ep.EP_SCALE_ROW_F32, 0), (ep.EP_SCALE_COL_F32, 0), (ep.EP_SCALE_ROW_F32, 1), (ep.EP_SCALE_COL_F32, 1),
          (ep.EP_SCALE_COL_UE8M0, 1)]


def _wide_rows(T, H, seed):
    """bf16 rows whose 128-groups span magnitudes 2^-120 .. 2^120 (plus an
    all-zero group and a group at exactly 448)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    mag = 2.0 ** rng.integers(-120, 120, size=(T, H // 128, 1))
    f = (rng.standard_normal((T, H // 128, 128)) * mag).astype(np.float32).reshape(T, H)
    f[0, :128] = 0.0
    if T > 1:
        f[1, :128] = 448.0
    bits = oracle.f32_to_bf16_bits(f).reshape(T, H)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def _compare(r, o, fmt, check_all=True):
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o["tokens_per_expert"])
    assert_equal("slot", np_(r["slot"]), o["slot"])
    if check_all:
        assert_equal("codes", np_(r["b_q"]), o["b_q"])
        assert_equal("scales (bits)", np_(r["b_scale"]).view(np.uint32), o["b_scale"].view(np.uint32))
        return
    tpe = o["tokens_per_expert"]
    for e in range(len(tpe)):
        c = int(tpe[e])
        assert_equal(f"codes e={e}", np_(r["b_q"][e, :c]), o["b_q"][e, :c])
        gs = np_(r["b_scale"][e])
        ws = o["b_scale"][e]
        if fmt == ep.EP_SCALE_ROW_F32:
            gs, ws = gs[:c], ws[:c]
        else:
            gs, ws = gs[:, :c], ws[:, :c]
        assert_equal(f"scales e={e}", gs.view(np.uint32), ws.view(np.uint32))


@pytest.mark.parametrize("fmt,rs", COMBOS)
@pytest.mark.parametrize("zero_pad", [0, 1])
def test_batched_fp8_small_all_layouts(fmt, rs, zero_pad):
    T, H, K, E, El, rank, M = 1537, 1024, 6, 48, 12, 2, 300
    idx, _ = routing_inputs(T, K, E, 31 + fmt, 0.15)
    x = _wide_rows(T, H, 32)
    o = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, bool(rs), zero_pad=True)
    r = ep.batched_prepare_fp8(x.cuda(), idx.cuda(), E, El, rank, M, fmt, bool(rs), zero_pad=bool(zero_pad))
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    _compare(r, o, fmt, check_all=bool(zero_pad))


@pytest.mark.parametrize("fmt,rs", [(ep.EP_SCALE_COL_F32, 0), (ep.EP_SCALE_COL_UE8M0, 1)])
def test_batched_fp8_workload_full_size(fmt, rs):
    w = wl.WORKLOADS["batched"]
    x, idx, _ = wl.make(w)
    o = oracle.batched_prepare_fp8(x, idx, w.E, w.E_local, w.rank, w.max_num_tokens, fmt, bool(rs))
    r = ep.batched_prepare_fp8(x.cuda(), idx.cuda(), w.E, w.E_local, w.rank, w.max_num_tokens, fmt, bool(rs))
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0 and o["err"] == 0
    _compare(r, o, fmt, check_all=False)


def test_batched_fp8_padding_left_untouched():
    T, H, K, E, El, rank, M = 700, 512, 4, 16, 8, 1, 400
    idx, _ = routing_inputs(T, K, E, 33, 0.0)
    x = _wide_rows(T, H, 34)
    dev = "cuda"
    b_q = torch.full((El, M, H), 0xAB, dtype=torch.uint8, device=dev)
    shape, dt = ep.batched_scale_storage(El, M, H, ep.EP_SCALE_COL_UE8M0)
    b_s = torch.full(shape, 0x7F7F7F7F, dtype=dt, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    err = ep.error_word()
    ep.ep_batched_prepare_fp8(x.cuda(), idx.cuda(), T, K, H, E, El, rank, M, b_q, b_s, ep.EP_SCALE_COL_UE8M0, 1,
                              tpe, slot, 0, ep.workspace(T, K, E // El, El), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, 2, True, False,
                                   np.full((El, M, H), 0xAB, np.uint8), np.full(shape, 0x7F7F7F7F, np.int32))
    assert_equal("codes incl. untouched padding", np_(b_q), o["b_q"])
    assert_equal("packed scales incl. untouched padding", np_(b_s), o["b_scale"])


def test_batched_fp8_capacity_overflow():
    T, H, K, E, El, rank, M = 900, 256, 4, 8, 8, 0, 100
    idx, _ = routing_inputs(T, K, E, 35, 0.0)
    x = _wide_rows(T, H, 36)
    o = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, 1, False, zero_pad=True)
    r = ep.batched_prepare_fp8(x.cuda(), idx.cuda(), E, El, rank, M, 1, False, zero_pad=True)
    torch.cuda.synchronize()
    assert int(r["err"].item()) & ep.EP_ERR_CAPACITY and o["err"] & oracle.ERR_CAPACITY
    _compare(r, o, 1)


def test_batched_fp8_empty_and_host_checks():
    dev = "cuda"
    r = ep.batched_prepare_fp8(torch.empty((0, 512), dtype=torch.bfloat16, device=dev),
                               torch.empty((0, 4), dtype=torch.int64, device=dev), 8, 4, 1, 16, 2, True,
                               zero_pad=True)
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0
    assert int(r["tokens_per_expert"].abs().sum().item()) == 0
    assert int(r["b_q"].abs().sum().item()) == 0 and int(r["b_scale"].abs().sum().item()) == 0
    x = torch.zeros((4, 384), dtype=torch.bfloat16, device=dev)
    idx = torch.zeros((4, 2), dtype=torch.int64, device=dev)
    with pytest.raises(ep.EPError):
        ep.batched_prepare_fp8(x, idx, 4, 4, 0, 8, ep.EP_SCALE_COL_UE8M0, True)    # H % 512
    with pytest.raises(ep.EPError):
        ep.batched_prepare_fp8(torch.zeros((4, 512), dtype=torch.bfloat16, device=dev), idx, 4, 4, 0, 8,
                               ep.EP_SCALE_COL_UE8M0, False)                                 # no round_scale


def _min_workspace(T, El):
    """The smallest workspace the batched prepare accepts: a header, one count
    per (256-token block, local expert) and the kept counts.  Too small for the
    cooperative slot kernel's flags, so larger problems take the count and
    slot kernels."""
    kept = -(-El * 4 // 256) * 256
    return torch.zeros(256 + (-(-T // 256)) * El * 4 + kept, dtype=torch.uint8, device="cuda")


# T, H, K, E, E_local, rank, M, workspace: every slot kernel in front of the
# fp8 row scatter
SLOT_FORMS = [
    (3000, 256, 6, 192, 96, 1, 1000, "full"),      # more than 64 local experts: count + slot kernels
    (3000, 256, 8, 64, 32, 1, 1000, "min"),        # one cluster (needs no workspace)
    (50000, 128, 8, 64, 32, 1, 8000, "min"),       # past the cluster's size, no room for flags: count + slot kernels
    (160000, 128, 8, 64, 32, 1, 22000, "full"),    # past the cluster's size: the cooperative slot kernel
]


@pytest.mark.parametrize("T,H,K,E,El,rank,M,wsk", SLOT_FORMS)
def test_batched_fp8_every_slot_kernel_matches_oracle(T, H, K, E, El, rank, M, wsk):
    fmt, rs = ep.EP_SCALE_COL_F32, 0
    idx, _ = routing_inputs(T, K, E, T + 7, 0.1)
    x = _wide_rows(T, H, T + 8)
    dev = "cuda"
    b_q = torch.empty((El, M, H), dtype=torch.uint8, device=dev)
    shape, dt = ep.batched_scale_storage(El, M, H, fmt)
    b_s = torch.empty(shape, dtype=dt, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws = ep.workspace(T, K, E // El, El) if wsk == "full" else _min_workspace(T, El)
    err = ep.error_word()
    ep.ep_batched_prepare_fp8(x.cuda(), idx.cuda(), T, K, H, E, El, rank, M, b_q, b_s, fmt, rs, tpe, slot, 0, ws,
                              err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ep.ep_status_str(int(err.item()))
    o = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, False)
    _compare(dict(tokens_per_expert=tpe, slot=slot, b_q=b_q, b_scale=b_s), o, fmt, check_all=False)


def test_batched_helpers_take_a_callers_workspace():
    # one workspace, reused by the three expert-batched helpers in turn
    T, H, K, E, El, rank, M = 900, 512, 4, 32, 8, 2, 400
    idx, _ = routing_inputs(T, K, E, 61, 0.1)
    x = _wide_rows(T, H, 62)
    ws = ep.workspace(T, K, E // El, El)
    xd, idd = x.cuda(), idx.cuda()
    r0 = ep.batched_prepare(xd, idd, E, El, rank, M, zero_pad=True, ws=ws)
    r1 = ep.batched_prepare_fp8(xd, idd, E, El, rank, M, ep.EP_SCALE_COL_F32, False, zero_pad=True, ws=ws)
    r2 = ep.batched_prepare_ex(xd, idd, E, El, rank, M, capacity=20, alignment=16, scale_fmt=ep.EP_SCALE_ROW_F32,
                               zero_pad=True, ws=ws)
    torch.cuda.synchronize()
    o0 = oracle.batched_prepare(x, idx, E, El, rank, M, zero_pad=True)
    assert_equal("bf16 rows", np_(r0["b_x"].view(torch.int16)).view(np.uint16), o0["b_x"])
    assert_equal("bf16 slots", np_(r0["slot"]), o0["slot"])
    _compare(r1, oracle.batched_prepare_fp8(x, idx, E, El, rank, M, ep.EP_SCALE_COL_F32, False, zero_pad=True),
             ep.EP_SCALE_COL_F32, check_all=True)
    o2 = oracle.batched_prepare_ex(x, idx, E, El, rank, M, 20, 16, fmt=oracle.SCALE_ROW_F32, zero_pad=True)
    assert_equal("capacity rows", np_(r2["b_rows"]), o2["b_rows"])
    assert_equal("capacity slots", np_(r2["slot"]), o2["slot"])
    assert_equal("dropped", np_(r2["dropped"]), o2["dropped"])
