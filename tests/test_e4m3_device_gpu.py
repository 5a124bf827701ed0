"""The oracle's fp32 -> fp8 e4m3 encoder against CUDA's own conversion on the
device, over every one of the 2^32 fp32 bit patterns (OCP OFP8 E4M3: round to
nearest even, saturating to +-448; the fp8 payload of NeMo uccl_ep.buffer,
Buffer.dispatch).  A small harness (tests/cvt_probe.cu, built here) applies
the pair conversion the library's quantising kernels use and the single-value
conversion; each must give the oracle's code for every non-NaN pattern, and
a NaN code (exponent and mantissa bits all ones) for every NaN pattern."""
import concurrent.futures as cf
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def cvt(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("cvt_probe") / "cvt_probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "cvt_probe.cu"), "-o", out],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.cvt_e4m3_range.restype = ctypes.c_int
    lib.cvt_e4m3_range.argtypes = [ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p]
    return lib


def _mismatch(bits, ours, dev, name):
    f = bits.view(np.float32)
    nan = np.isnan(f)
    bad = np.where(nan, (dev & 0x7F) != 0x7F, ours != dev)
    if not bad.any():
        return None
    i = int(np.nonzero(bad)[0][0])
    return f"{name}: pattern {int(bits[i]):#010x}: oracle {int(ours[i]):#04x}, device {int(dev[i]):#04x}"


def test_oracle_e4m3_encoder_matches_the_device_conversion_on_every_f32_pattern(cvt):
    step = 1 << 24
    pair = torch.empty(step, dtype=torch.uint8, device="cuda")
    single = torch.empty(step, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def oracle_chunk(start):
        bits = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
        ours = oracle.f32_to_e4m3_bits(bits.view(np.float32))
        nan = np.isnan(bits.view(np.float32))
        assert np.all((ours[nan] & 0x7F) == 0x7F), f"oracle: a NaN pattern near {start:#010x} lost its NaN code"
        return bits, ours

    errors = []
    starts = list(range(0, 1 << 32, step))
    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {s: ex.submit(oracle_chunk, s) for s in starts[:8]}
        for j, start in enumerate(starts):
            rc = cvt.cvt_e4m3_range(start, step, pair.data_ptr(), single.data_ptr(), stream.cuda_stream)
            assert rc == 0, f"CUDA error {rc}"
            dev_pair, dev_single = pair.cpu().numpy(), single.cpu().numpy()
            bits, ours = futs.pop(start).result()
            if j + 8 < len(starts):
                futs[starts[j + 8]] = ex.submit(oracle_chunk, starts[j + 8])
            for name, dev in (("pair conversion", dev_pair), ("single conversion", dev_single)):
                e = _mismatch(bits, ours, dev, name)
                if e is not None:
                    errors.append(e)
            if len(errors) >= 5:
                break
    assert not errors, errors
