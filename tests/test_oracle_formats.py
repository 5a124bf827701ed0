"""Pins for the oracle's number formats (bf16 and OCP E4M3), against torch's
CPU conversions (a library routine) and hand-worked anchors."""
import numpy as np
import pytest
import torch

import oracle


def _sample_f32_bits(n, seed=1):
    g = np.random.Generator(np.random.PCG64(seed))
    bits = g.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32)


def _e4m3_range_values():
    """Values around every E4M3 rounding boundary: for each binade from 2^-12
    to 2^9, every quantum multiple m and the points just below, at and just
    above each half-way point."""
    vals = []
    for E in range(-12, 10):
        q = 2.0 ** (max(E, -6) - 3)
        for m in range(0, 17):
            for off in (-0.5, 0.0, 0.5):
                c = np.float32((m + off) * q)
                vals += [c, np.nextafter(c, np.float32(0)), np.nextafter(c, np.float32(np.inf))]
    v = np.array(vals, dtype=np.float32)
    return np.concatenate([v, -v])


def test_bf16_rne_matches_torch():
    f = np.concatenate([_sample_f32_bits(1 << 20),
                        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 3.0e38, 1e-45,
                                  1.00390625, 1.01171875, 1.0078125 + 2**-24], np.float32)])
    ours = oracle.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.bf16_bits_to_f32(ours[nan])))


def test_bf16_ties_to_even_anchors():
    # 1 + 2^-8 is half way between 1 and 1 + 2^-7: ties to the even neighbour 1.
    # 1 + 3*2^-8 is half way between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6.
    f = np.array([1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-20], np.float32)
    got = oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(f))
    assert got.tolist() == [1.0, 1 + 2**-6, 1 + 2**-7]


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # OFP8 E4M3 anchors: max finite 448, smallest normal 2^-6, smallest subnormal 2^-9.
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0**-6 and ours[0x01] == 2.0**-9
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


@pytest.mark.parametrize("which", ["random", "boundaries"])
def test_e4m3_rn_satfinite_matches_torch_on_clamped(which):
    # torch's float->e4m3fn conversion rounds to nearest-even and maps values
    # beyond the range to NaN; saturating first (clamp to +-448) gives the
    # satfinite conversion, since rounding is monotone and 448 is representable.
    if which == "random":
        f = _sample_f32_bits(1 << 20, seed=2)
        with np.errstate(invalid="ignore", over="ignore"):
            f = np.concatenate([f, f * np.float32(2.0**-120)])   # bring many into range
    else:
        f = _e4m3_range_values()
    f = f[np.isfinite(f)]
    ours = oracle.f32_to_e4m3_bits(f)
    clamped = np.clip(f, np.float32(-448.0), np.float32(448.0))
    ref = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch may give -0 for tiny negatives where we give -0 too; compare bits directly
    assert np.array_equal(ours, ref), np.nonzero(ours != ref)[0][:10]


def test_e4m3_special_inputs():
    f = np.array([np.nan, np.inf, -np.inf, 1e30, -1e30, 449.0, 464.0, -0.0], np.float32)
    got = oracle.f32_to_e4m3_bits(f)
    assert got[0] & 0x7F == 0x7F
    assert got[1:].tolist() == [0x7E, 0xFE, 0x7E, 0xFE, 0x7E, 0x7E, 0x80]


@pytest.mark.slow
def test_e4m3_rn_satfinite_exhaustive_over_every_f32_pattern():
    # Every one of the 2^32 fp32 bit patterns through the oracle's encoder
    # (OCP OFP8 E4M3, round to nearest even, saturating to +-448; the fp8
    # payload of NeMo uccl_ep.buffer, Buffer.dispatch), against torch's
    # conversion of the value clamped to +-448.  NaN inputs must give a NaN
    # code (exponent and mantissa bits all ones), whatever the sign bit.
    import concurrent.futures as cf
    import os

    step = 1 << 24
    lo, hi = np.float32(-448.0), np.float32(448.0)

    def one(start):
        bits = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
        f = bits.view(np.float32)
        ours = oracle.f32_to_e4m3_bits(f)
        nan = np.isnan(f)
        with np.errstate(invalid="ignore"):
            clamped = np.clip(f, lo, hi)
        ref = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ok = np.all(ours[~nan] == ref[~nan]) and np.all((ours[nan] & 0x7F) == 0x7F) \
            and np.all((ref[nan] & 0x7F) == 0x7F)
        if ok:
            return None
        bad = np.nonzero(np.where(nan, (ours & 0x7F) != 0x7F, ours != ref))[0]
        i = int(bad[0])
        return f"pattern {int(bits[i]):#010x}: oracle {int(ours[i]):#04x}, torch {int(ref[i]):#04x}"

    torch_threads = torch.get_num_threads()
    torch.set_num_threads(1)                       # the pool below is the parallelism
    try:
        with cf.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
            errors = [e for e in ex.map(one, range(0, 1 << 32, step)) if e is not None]
    finally:
        torch.set_num_threads(torch_threads)
    assert not errors, errors[:5]
