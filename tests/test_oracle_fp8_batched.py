"""Pins of the oracle's fp8 expert-batched prepare and its scale formats
(NeMo uccl_ep.buffer Buffer.low_latency_dispatch: round_scale, use_ue8m0,
column-major scales; vLLM BatchedPrepareAndFinalize.prepare, quantised
branch).  Checked against hand-worked values, closed-form properties of
power-of-two scales, the already pinned per-token quantiser and slot
assignment, and layout identities."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fp8_pow2.json")


def _bf16(a) -> np.ndarray:
    """float32 values exactly representable in bf16 -> their bit patterns."""
    f = np.asarray(a, np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _golden_row():
    g = json.load(open(GOLDEN))
    H = g["H"]
    row = np.zeros(H, np.float32)
    for gi, head in enumerate(g["x_heads"]):
        row[gi * 128: gi * 128 + len(head)] = head
    return g, _bf16(row)[None, :]


def test_pow2_quantiser_matches_hand_worked_groups():
    g, x = _golden_row()
    q, s, c = oracle.quantize_fp8_rows_pow2(x)
    for gi, head in enumerate(g["q_heads"]):
        got = q[0, gi * 128: gi * 128 + len(head)].tolist()
        assert got == head, (gi, got, head)
        assert np.all(q[0, gi * 128 + len(head): (gi + 1) * 128] == 0)
    assert s[0].tolist() == g["scales"]
    assert c[0].tolist() == g["ue8m0"]
    assert int(c[0].astype("<u1").view("<i4")[0]) == g["packed_int32"]


def _random_rows(R, H, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    mag = 2.0 ** rng.integers(-30, 30, size=(R, H // 128, 1))      # one magnitude per group
    f = (rng.standard_normal((R, H // 128, 128)) * mag).astype(np.float32).reshape(R, H)
    f[0, :128] = 0.0                                                 # an all-zero group
    f[1, 128:256] = 448.0                                            # scale exactly 1
    return oracle.f32_to_bf16_bits(f).reshape(R, H)


def test_pow2_scales_closed_form():
    x = _random_rows(40, 1024, 3)
    q, s, c = oracle.quantize_fp8_rows_pow2(x)
    xf = oracle.bf16_bits_to_f32(x).reshape(40, 8, 128)
    a = np.maximum(np.abs(xf).max(-1), np.float32(1e-4)).astype(np.float32)
    s0 = (a / np.float32(448.0)).astype(np.float32)
    m, e = np.frexp(s)
    assert np.all(m == 0.5)                                  # powers of two
    assert np.all(s >= s0) and np.all(s / 2 < s0)            # the smallest one >= a/448
    assert np.all(c.astype(np.int64) == e.astype(np.int64) - 1 + 127)   # UE8M0 = biased exponent
    d = oracle.e4m3_to_f32(q).reshape(40, 8, 128)
    assert np.all(np.abs(d) <= 448.0)
    # x / scale is exact (power of two) and never above 448: the codes are the
    # plain e4m3 rounding of x / scale, within half a quantum of it
    y = xf / s[..., None]
    assert np.all(np.abs(y) <= 448.0)
    quantum = 2.0 ** (np.maximum(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))), -6) - 3)
    assert np.all(np.abs(d - y) <= quantum / 2)


def test_plain_scales_unchanged_when_round_scale_is_off():
    # round_scale=0 is the per-token quantiser of the fp8 dispatch, row for row
    x = _random_rows(6, 512, 4)
    idx = np.array([[0, 3], [1, -1], [3, 2], [2, 0], [1, 3], [0, 1]], np.int64)
    r = oracle.batched_prepare_fp8(x, idx, 4, 4, 0, 6, fmt=oracle.SCALE_ROW_F32, round_scale=False)
    qr, sr = oracle.quantize_fp8_rows(x)
    plain = oracle.batched_prepare(x, idx, 4, 4, 0, 6)
    assert r["err"] == 0
    assert np.array_equal(r["slot"], plain["slot"])
    assert np.array_equal(r["tokens_per_expert"], plain["tokens_per_expert"])
    for t in range(6):
        for k in range(2):
            e, sl = idx[t, k], r["slot"][t, k]
            if e < 0:
                continue
            assert np.array_equal(r["b_q"][e, sl], qr[t])
            assert np.array_equal(r["b_scale"][e, sl].view(np.uint32), sr[t].view(np.uint32))


def _routing(T, K, E, seed, frac=0.1):
    rng = np.random.Generator(np.random.PCG64(seed))
    idx = np.argsort(rng.random((T, E)), 1)[:, :K].astype(np.int64)
    idx[rng.random((T, K)) < frac] = -1
    return idx


@pytest.mark.parametrize("round_scale", [False, True])
def test_column_major_scales_are_the_transpose(round_scale):
    T, H, K, E, El, rank, M = 50, 1024, 4, 16, 4, 1, 40
    x = _random_rows(T, H, 5)
    idx = _routing(T, K, E, 6)
    row = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, oracle.SCALE_ROW_F32, round_scale, zero_pad=True)
    col = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, oracle.SCALE_COL_F32, round_scale, zero_pad=True)
    assert np.array_equal(row["b_q"], col["b_q"])
    assert col["b_scale"].shape == (El, H // 128, M)
    assert np.array_equal(col["b_scale"].view(np.uint32), row["b_scale"].transpose(0, 2, 1).view(np.uint32))


def test_ue8m0_packing():
    T, H, K, E, El, rank, M = 50, 1024, 4, 16, 4, 2, 40
    x = _random_rows(T, H, 7)
    idx = _routing(T, K, E, 8)
    ue = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, oracle.SCALE_COL_UE8M0, True, zero_pad=True)
    row = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, oracle.SCALE_ROW_F32, True, zero_pad=True)
    assert ue["err"] == 0 and ue["b_scale"].dtype == np.int32 and ue["b_scale"].shape == (El, H // 512, M)
    # unpack: int (e, j, s) little-endian bytes are groups 4j .. 4j+3
    b = ue["b_scale"].astype("<i4").view(np.uint8).reshape(El, H // 512, M, 4)
    codes = b.transpose(0, 2, 1, 3).reshape(El, M, H // 128)          # [e, s, g]
    used = np.arange(M)[None, :] < row["tokens_per_expert"][:, None]
    _, e = np.frexp(row["b_scale"])
    want = np.where(used[..., None], e - 1 + 127, 0)
    assert np.array_equal(codes, want)


def test_ue8m0_needs_round_scale_and_h_multiple_of_512():
    x = _random_rows(4, 512, 9)
    idx = np.zeros((4, 2), np.int64)
    assert oracle.batched_prepare_fp8(x, idx, 2, 2, 0, 4, oracle.SCALE_COL_UE8M0, False)["err"] == 16
    x = _random_rows(4, 384, 9)
    assert oracle.batched_prepare_fp8(x, idx, 2, 2, 0, 4, oracle.SCALE_COL_UE8M0, True)["err"] == 16


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_zero_pad_and_untouched_padding(fmt):
    T, H, K, E, El, rank, M = 30, 512, 2, 8, 4, 0, 25
    x = _random_rows(T, H, 10)
    idx = _routing(T, K, E, 11, 0.0)
    shape, dt = oracle.batched_scale_shape(El, M, H, fmt)
    q0 = np.full((El, M, H), 0xAB, np.uint8)
    s0 = np.full(shape, 0x7F7F7F7F if dt == np.int32 else np.nan, dt)
    keep = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, fmt == 2, False, q0, s0)
    zero = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, fmt, fmt == 2, True, q0, s0)
    tpe = keep["tokens_per_expert"]
    for e in range(El):
        c = int(tpe[e])
        assert np.all(keep["b_q"][e, c:] == 0xAB) and np.all(zero["b_q"][e, c:] == 0)
        assert np.array_equal(keep["b_q"][e, :c], zero["b_q"][e, :c])
        if fmt == 0:
            kp, zp = keep["b_scale"][e, c:], zero["b_scale"][e, c:]
        else:
            kp, zp = keep["b_scale"][e, :, c:], zero["b_scale"][e, :, c:]
        assert np.all(zp == 0)
        assert np.all(np.isnan(kp)) if dt != np.int32 else np.all(kp == 0x7F7F7F7F)


def test_capacity_drop():
    T, H, K, E, El, rank, M = 40, 256, 2, 4, 4, 0, 5
    x = _random_rows(T, H, 12)
    idx = _routing(T, K, E, 13, 0.0)
    r = oracle.batched_prepare_fp8(x, idx, E, El, rank, M, oracle.SCALE_ROW_F32, False)
    assert r["err"] & oracle.ERR_CAPACITY
    assert np.all(r["tokens_per_expert"] == M)
    assert r["slot"].max() == M - 1


# Non-finite inputs (the pages are silent; the reading: NaN elements do not
# enter a group's maximum, and a group holding +-inf has a = inf, so its scale
# is +inf and its reciprocal +0 in both forms).  Pinned by IEEE arithmetic:
# x * (+0) is +-0 with x's sign for finite x and NaN for +-inf or NaN.
NAN16, INF16, NINF16 = 0x7FC0, 0x7F80, 0xFF80


def _nonfinite_row():
    f = np.zeros((1, 512), np.float32)
    f[0, 128:131] = [3.0, -1.5, 0.25]          # group 1: finite, with a NaN at column 131
    f[0, 256:259] = [1.0, -2.0, 7.0]           # group 2: finite, with +inf at 259 and -inf at 260
    f[0, 384:387] = [5.0, -6.0, 0.5]           # group 3: finite only
    x = _bf16(f)
    x[0, 0] = NAN16                            # group 0: NaN and zeros only
    x[0, 131] = NAN16
    x[0, 259] = INF16
    x[0, 260] = NINF16
    return x


def _is_nan_code(c):
    return (np.asarray(c) & 0x7F) == 0x7F


@pytest.mark.parametrize("pow2", [False, True])
def test_quantisers_on_non_finite_inputs(pow2):
    x = _nonfinite_row()
    if pow2:
        q, s, c = oracle.quantize_fp8_rows_pow2(x)
    else:
        q, s = oracle.quantize_fp8_rows(x)
    # NaN elements do not enter the maximum: groups 0, 1 and 3 are quantised
    # exactly as with their NaNs replaced by +0, except the NaN's own code
    clean = x.copy()
    clean[0, 0] = 0
    clean[0, 131] = 0
    clean[0, 259:261] = 0
    qc = oracle.quantize_fp8_rows_pow2(clean) if pow2 else oracle.quantize_fp8_rows(clean)
    for g in (0, 1, 3):
        cols = np.arange(g * 128, (g + 1) * 128)
        keep = (cols != 0) & (cols != 131)
        assert np.array_equal(q[0, cols[keep]], qc[0][0, cols[keep]]), g
        assert s[0, g] == qc[1][0, g], g
        if pow2:
            assert c[0, g] == qc[2][0, g], g
    assert _is_nan_code(q[0, 0]) and _is_nan_code(q[0, 131])
    # group 0 holds only a NaN and zeros: the floor a = 1e-4 applies
    assert s[0, 0] == qc[1][0, 0]
    # group 2 holds +-inf: scale +inf, finite elements -> +-0, infinities -> NaN codes
    assert s[0, 2] == np.inf
    assert q[0, 256] == 0x00 and q[0, 257] == 0x80 and q[0, 258] == 0x00
    assert np.all(q[0, 261:384] == 0x00)
    assert _is_nan_code(q[0, 259]) and _is_nan_code(q[0, 260])
    if pow2:
        assert c[0, 2] == 255
