"""fp8 (1x128) quantisation of rows holding NaN and +-inf, on both layouts,
against the oracle (NeMo uccl_ep.buffer, Buffer.dispatch fp8 payload and
Buffer.low_latency_dispatch scale formats; the pages are silent on
non-finite inputs, and the reading both sides follow is: NaN elements do not
enter a group's maximum; a group holding +-inf gets scale +inf and reciprocal
+0, UE8M0 code 255, so its finite elements give +-0 codes and its
infinities NaN codes).  Codes are compared bit for bit except that a NaN
code's sign bit is not compared (IEEE leaves the sign of the NaN that
inf * 0 makes to the implementation); scales bit for bit."""
import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_equal, bits16, np_, routing_inputs

pytestmark = pytest.mark.gpu

COMBOS = [(ep.EP_SCALE_ROW_F32, 0), (ep.EP_SCALE_COL_F32, 0), (ep.EP_SCALE_ROW_F32, 1), (ep.EP_SCALE_COL_F32, 1),
          (ep.EP_SCALE_COL_UE8M0, 1)]


def _rows_with_non_finite(T, H, seed):
    """bf16 rows of N(0, 1) values with NaN, +inf and -inf planted in about a
    tenth of the 128-groups (one to three elements each), and some groups
    holding only NaNs and zeros."""
    rng = np.random.Generator(np.random.PCG64(seed))
    f = rng.standard_normal((T, H)).astype(np.float32)
    bits = oracle.f32_to_bf16_bits(f).reshape(T, H)
    G = H // 128
    specials = np.array([0x7FC0, 0xFFC0, 0x7F80, 0xFF80], np.uint16)   # +NaN, -NaN, +inf, -inf
    for t in range(T):
        for g in range(G):
            u = rng.random()
            if u < 0.1:
                cols = g * 128 + rng.choice(128, size=int(rng.integers(1, 4)), replace=False)
                bits[t, cols] = rng.choice(specials, size=cols.size)
            elif u < 0.12:
                bits[t, g * 128:(g + 1) * 128] = 0
                bits[t, g * 128 + int(rng.integers(0, 128))] = 0x7FC0
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def _assert_codes(name, got, want):
    got, want = np.asarray(got, np.uint8), np.asarray(want, np.uint8)
    nan_g, nan_w = (got & 0x7F) == 0x7F, (want & 0x7F) == 0x7F
    assert_equal(name + " (NaN positions)", nan_g, nan_w)
    assert_equal(name + " (non-NaN codes)", np.where(nan_w, 0, got), np.where(nan_w, 0, want))


def test_send_layout_fp8_dispatch_non_finite():
    T, H, K, E, P = 900, 1024, 6, 64, 8
    idx, w = routing_inputs(T, K, E, seed=71, frac_unrouted=0.1)
    x = _rows_with_non_finite(T, H, 72)
    xb = bits16(x)
    assert (((xb & 0x7F80) == 0x7F80) & ((xb & 0x7F) == 0)).any()     # infinities planted
    o = oracle.send_path(x, idx, w, None, P, E // P)
    sti = o["layout"]["send_token_idx"]
    oq, os_ = oracle.dispatch_fp8(x, sti)
    assert np.isinf(os_).any()
    err = ep.error_word()
    c = ep.compute_send_counts(idx.cuda(), P, E // P, err=err)
    N = int(c["send_counts"].sum().item())
    lay = ep.build_send_layout(idx.cuda(), w.cuda(), c["dest"], c["is_in_rank"], N, E // P, err=err)
    q, s = ep.dispatch_rows(x.cuda(), lay["token_pos"], N, fp8=True, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and N == sti.size
    _assert_codes("codes", np_(q), oq)
    assert_equal("scales (bits)", np_(s).view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("fmt,rs", COMBOS)
def test_batched_fp8_prepare_non_finite(fmt, rs):
    T, H, K, E, El, rank, M = 1100, 1024, 8, 64, 16, 1, 400
    idx, _ = routing_inputs(T, K, E, seed=73 + fmt, frac_unrouted=0.1)
    x = _rows_with_non_finite(T, H, 74)
    o = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, bool(rs), zero_pad=True)
    r = ep.batched_prepare_fp8(x.cuda(), idx.cuda(), E, El, rank, M, fmt, bool(rs), zero_pad=True)
    torch.cuda.synchronize()
    assert int(r["err"].item()) == 0 and o["err"] == 0
    assert_equal("tokens_per_expert", np_(r["tokens_per_expert"]), o["tokens_per_expert"])
    assert_equal("slot", np_(r["slot"]), o["slot"])
    _assert_codes("codes", np_(r["b_q"]), o["b_q"])
    got_s = np_(r["b_scale"])
    if fmt == ep.EP_SCALE_COL_UE8M0:
        assert_equal("UE8M0 codes", got_s.view(np.uint8), o["b_scale"].view(np.uint8))
        assert (o["b_scale"].view(np.uint8) == 255).any()
    else:
        assert_equal("scales (bits)", got_s.view(np.uint32), o["b_scale"].view(np.uint32))
        assert np.isinf(o["b_scale"]).any()
