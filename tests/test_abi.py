"""The C-ABI library builds, loads and exports every entry point that
include/ep.h declares; host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest
import torch

import combine_send_counts_gb300 as ep
from combine_send_counts_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ep.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ep_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ctypes.CDLL(_build.LIB_PATH)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ep_compute_send_counts", "ep_build_send_layout", "ep_dispatch", "ep_combine",
                     "ep_batched_prepare", "ep_batched_combine", "ep_chunk_bounds", "ep_workspace_size",
                     "ep_status_str", "ep_local_expert_fp8"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    for n in declared_functions():
        assert callable(getattr(ep, n, None)), n


def test_host_only_calls(lib):
    assert ep.ep_status_str(0) == "EP_OK"
    assert ep.ep_status_str(ep.EP_ERR_CAPACITY) == "EP_ERR_CAPACITY"
    assert ep.ep_chunk_bounds(10, 3) == [0, 3, 6, 10]
    assert ep.ep_chunk_bounds(2, 4) == [0, 0, 0, 0, 2]
    assert ep.ep_workspace_size(16384, 8, 8, 32, 1) > 0
    with pytest.raises(ep.EPError):
        ep.ep_chunk_bounds(5, 0)


def test_argument_checks_reject_before_launch(lib):
    # Null / impossible arguments are rejected on the host: no device is touched.
    vp = ctypes.c_void_p
    lib.ep_dispatch.argtypes = [vp, ctypes.c_int64, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int64, vp, vp,
                                ctypes.c_int, vp, vp]
    assert lib.ep_dispatch(None, 4, 7, None, 2, 4, None, None, 0, None, None) == ep.EP_ERR_INVALID_ARG  # H % 8
    assert lib.ep_dispatch(None, 4, 64, None, 2, 4, None, None, 1, None, None) == ep.EP_ERR_UNSUPPORTED  # fp8, H % 128
    assert lib.ep_dispatch(None, 4, 64, None, 0, 4, None, None, 0, None, None) == ep.EP_ERR_INVALID_ARG  # P = 0
    assert lib.ep_dispatch(None, 0, 64, None, 2, 0, None, None, 0, None, None) == ep.EP_OK  # empty: nothing to do
    lib.ep_combine.argtypes = [vp, ctypes.c_int64, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int64, vp,
                               ctypes.c_int, vp, ctypes.c_size_t, vp, vp]
    assert lib.ep_combine(None, 4, 64, None, 2, 4, None, 2, None, 0, None, None) == ep.EP_ERR_UNSUPPORTED  # dtype
    assert lib.ep_combine(None, 4, 64, None, 2, 4, None, 0, None, 0, None, None) == ep.EP_ERR_INVALID_ARG  # out
    f = lib.ep_batched_prepare_fp8
    f.argtypes = [vp, vp, ctypes.c_int64] + [ctypes.c_int] * 6 + [vp, vp, ctypes.c_int, ctypes.c_int, vp, vp,
                                                                  ctypes.c_int, vp, ctypes.c_size_t, vp, vp]
    args = lambda H, fmt, rs: (None, None, 4, 2, H, 8, 4, 0, 16, None, None, fmt, rs, None, None, 0, None, 0,
                               None, None)
    assert f(*args(512, 3, 1)) == ep.EP_ERR_INVALID_ARG          # unknown scale layout
    assert f(*args(512, 0, 2)) == ep.EP_ERR_INVALID_ARG          # round_scale not 0/1
    assert f(*args(192, 0, 0)) == ep.EP_ERR_UNSUPPORTED          # H % 128
    assert f(*args(512, 2, 0)) == ep.EP_ERR_UNSUPPORTED          # UE8M0 needs round_scale
    assert f(*args(384, 2, 1)) == ep.EP_ERR_UNSUPPORTED          # UE8M0 needs H % 512
    assert f(*args(512, 1, 1)) == ep.EP_ERR_INVALID_ARG          # null outputs


def test_no_entry_point_host_code_calls_exit(lib):
    # nvcc compiles a host-side call of a __device__-only function inside a
    # template into exit(1) without a diagnostic; an entry point built that
    # way ends the caller's process silently.  Inspect the host code of this
    # (locally built) library for direct calls of exit.
    import shutil
    import subprocess
    objdump = shutil.which("objdump")
    if objdump is None:
        pytest.skip("objdump not available")
    asm = subprocess.run([objdump, "-d", "--no-show-raw-insn", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    fn, offenders = None, set()
    for line in asm.splitlines():
        m = re.match(r"^[0-9a-f]+ <(.+)>:$", line)
        if m:
            fn = m.group(1)
        elif re.search(r"\s(call|bl|jmp|b)\s+[0-9a-f]+ <exit@plt>", line):
            offenders.add(fn)
    assert not offenders, offenders


def test_ctypes_structs_match_the_header(tmp_path):
    # Compile a probe against include/ep.h with the host C compiler and compare
    # every struct's size and field offsets with the ctypes mirrors.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    mirrors = {"ep_chunk_buffers": ep.EPChunkBuffers, "ep_row_set": ep.EPRowSet,
               "ep_pipeline_buffers": ep.EPPipelineBuffers}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "ep.h"', "int main(void) {"]
    for cname, cls in mirrors.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0; }"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        cname, field, v = line.split()
        got[(cname, field)] = int(v)
    for cname, cls in mirrors.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, (cname, f)


def test_helpers_reject_wrong_dtypes_before_any_device_work():
    # the C ABI takes untyped pointers; the allocating helpers check the dtypes
    # first, so these fail on the host (CPU tensors, no CUDA needed)
    x32 = torch.zeros((4, 8), dtype=torch.float32)
    idx = torch.zeros((4, 2), dtype=torch.int64)
    w = torch.zeros((4, 2), dtype=torch.float32)
    tp = torch.zeros((4, 2), dtype=torch.int32)
    with pytest.raises(TypeError, match="x must be torch.bfloat16"):
        ep.dispatch_rows(x32, tp, 4)
    with pytest.raises(TypeError, match="topk_idx must be torch.int64"):
        ep.compute_send_counts(idx.to(torch.int32), 2, 2)
    with pytest.raises(TypeError, match="topk_weights must be torch.float32"):
        ep.route_nosync(idx, w.to(torch.float64), 2, 2)
    with pytest.raises(TypeError, match="y must be torch.bfloat16"):
        ep.combine_rows(x32, tp)
    with pytest.raises(TypeError, match="slot must be torch.int32"):
        ep.batched_combine(torch.zeros((2, 4, 8), dtype=torch.bfloat16), idx, w, idx, 0)


def test_noalloc_counts_reject_bad_arguments_without_a_device(lib):
    # The no-allocation counts entry checks its arguments before it looks up
    # its device array (which would need a device): with no GPU here, a device
    # call would answer EP_ERR_CUDA instead of these host statuses.
    f = ep.load().ep_compute_send_counts_noalloc
    call = lambda T, K, P, El, bounds, C, sc=None: f(None, T, K, P, El, bounds, C, None, None, sc, None, None,
                                                     None, ctypes.c_void_p(0))
    assert call(-1, 8, 8, 32, None, 1) == ep.EP_ERR_INVALID_ARG             # T < 0
    assert call(16, 0, 8, 32, None, 1) == ep.EP_ERR_INVALID_ARG             # K = 0
    assert call(16, 8, 8, 0, None, 1) == ep.EP_ERR_INVALID_ARG              # E_local = 0
    assert call(16, 8, 8, 32, None, 1) == ep.EP_ERR_INVALID_ARG             # no send_counts
    bounds = (ctypes.c_int64 * 3)(0, 4, 15)                                   # does not end at T
    assert call(16, 8, 8, 32, bounds, 2, ctypes.c_void_p(16)) == ep.EP_ERR_INVALID_ARG
    assert call(1 << 22, 8, 64, 128, None, 1) == ep.EP_ERR_UNSUPPORTED   # beyond the fixed array
