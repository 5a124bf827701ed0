"""Failure detection on the GPU without a fault: the library's bounded waits
are run by a small harness (tests/wait_probe.cu, built here) on something that
never happens.  The mbarrier wait (every consumer and producer wait of the
combine's bulk-copy ring goes through it) on a phase that nothing completes,
and the grid barrier of the cooperative routing kernels with a block that
leaves without arriving, must give up after their limits with EP_ERR_TIMEOUT,
read back by the host, and the context must stay usable: a library call
afterwards still matches the oracle."""
import ctypes
import os
import shutil
import subprocess
import time

import numpy as np
import pytest
import torch

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_equal, np_, routing_inputs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("wait_probe") / "wait_probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "combine_send_counts_gb300", "csrc"),
                    "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "wait_probe.cu"), "-o", out],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.wait_probe.restype = ctypes.c_int
    lib.wait_probe.argtypes = [ctypes.c_ulonglong, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                               ctypes.POINTER(ctypes.c_ulonglong)]

    lib.barrier_probe.restype = ctypes.c_int
    lib.barrier_probe.argtypes = [ctypes.c_int, ctypes.c_ulonglong, ctypes.POINTER(ctypes.c_int32)]

    def run(limit_ns, complete_first):
        torch.cuda.synchronize()
        status, elapsed = ctypes.c_int32(-1), ctypes.c_ulonglong(0)
        rc = lib.wait_probe(limit_ns, int(complete_first), ctypes.byref(status), ctypes.byref(elapsed))
        assert rc == 0, f"CUDA error {rc}"
        return status.value, elapsed.value

    def barrier(absent_block, host_tag):
        torch.cuda.synchronize()
        status = (ctypes.c_int32 * 2)()
        t0 = time.perf_counter()
        rc = lib.barrier_probe(absent_block, host_tag, status)
        assert rc == 0, f"CUDA error {rc}"
        return list(status), time.perf_counter() - t0

    run.barrier = barrier
    return run


def test_wait_on_a_phase_nothing_completes_times_out(probe):
    limit = 20_000_000   # 20 ms
    status, elapsed = probe(limit, False)
    assert status == ep.EP_ERR_TIMEOUT
    assert limit <= elapsed < 50 * limit


def test_wait_on_a_completed_phase_returns_at_once(probe):
    status, elapsed = probe(20_000_000, True)
    assert status == ep.EP_OK
    assert elapsed < 1_000_000


def test_context_usable_after_a_timeout(probe):
    assert probe(5_000_000, False)[0] == ep.EP_ERR_TIMEOUT
    idx, _ = routing_inputs(1000, 4, 32, 9, 0.1)
    c = ep.compute_send_counts(idx.cuda(), 8, 4)
    torch.cuda.synchronize()
    o = oracle.compute_send_counts(idx, 8, 4)
    assert int(c["err"].item()) == 0
    assert_equal("send_counts", np_(c["send_counts"]).reshape(-1), o["send_counts"])
    assert_equal("is_in_rank", np_(c["is_in_rank"]), o["is_in_rank"])


def test_grid_barrier_passes_when_every_block_arrives(probe):
    status, _ = probe.barrier(-1, 0x1234)
    assert status == [ep.EP_OK, ep.EP_OK]


def test_grid_barrier_gives_up_on_a_block_that_never_arrives(probe):
    status, seconds = probe.barrier(1, 0x5678)
    assert status == [ep.EP_ERR_TIMEOUT, -1]   # block 1 left without arriving
    assert 0.45 < seconds < 10.0               # the barrier's limit is 0.5 s
    # the context is still usable
    assert probe.barrier(-1, 0x9abc)[0] == [ep.EP_OK, ep.EP_OK]
