"""CPU oracle for MoE top-k dispatch / combine (plain C behind ctypes + numpy).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``combine_send_counts_gb300``) and neither imports
the other; ``oracle.c`` states the definitions it follows and the readings
taken where the pages are silent.

Arrays are numpy; bf16 tensors travel as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

ERR_INVALID_EXPERT = 2
ERR_CAPACITY = 8

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (plain C11, no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int
    sig = {
        "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_e4m3_to_f32": (ctypes.c_float, [ctypes.c_uint8]),
        "orc_f32_to_e4m3": (ctypes.c_uint8, [ctypes.c_float]),
        "orc_f32_to_bf16_array": (None, [P, i64, P]),
        "orc_f32_to_e4m3_array": (None, [P, i64, P]),
        "orc_e4m3_to_f32_array": (None, [P, i64, P]),
        "orc_chunk_bounds": (None, [i64, i32, P]),
        "orc_compute_send_counts": (i32, [P, i64, i32, i32, i32, P, P, P, P]),
        "orc_build_send_layout": (i64, [P, P, P, P, i64, i32, i32, i32, i64, P, P, P, P, P]),
        "orc_dispatch": (None, [P, i32, P, i64, P]),
        "orc_quantize_fp8_rows": (None, [P, i64, i32, P, P]),
        "orc_dispatch_fp8": (None, [P, i64, i32, P, i64, P, P]),
        "orc_local_expert_fp8": (None, [P, P, P, P, i64, i32, i32, P]),
        "orc_combine": (None, [P, i64, i32, i32, P, i32, P]),
        "orc_batched_prepare": (i32, [P, P, i64, i32, i32, i32, i32, i32, i32, P, P, P, i32]),
        "orc_batched_combine": (None, [P, P, P, P, i64, i32, i32, i32, i32, i32, P]),
        "orc_quantize_fp8_rows_pow2": (None, [P, i64, i32, P, P, P]),
        "orc_batched_prepare_fp8": (i32, [P, P, i64, i32, i32, i32, i32, i32, i32, P, P, i32, i32, P, P, i32]),
        "orc_expert_capacity": (i64, [i64, i32, i32, ctypes.c_double]),
        "orc_batched_prepare_ex": (i32, [P, P, i64, i32, i32, i32, i32, i32, i32, i32, i32, P, P, i32, i32, P, P,
                                         P, i32]),
        "orc_align_send_layout": (i64, [P, i32, i32, i32, i64, P, P, P, P, P, P, P, P, P]),
        "orc_indices_to_multihot": (i32, [P, P, i64, i32, i32, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _bf16_bits(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bit patterns."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(a.contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


# ---------------------------------------------------------------- formats --
def f32_to_bf16_bits(f) -> np.ndarray:
    f = _c(f, np.float32).reshape(-1)
    out = np.empty(f.size, np.uint16)
    _load().orc_f32_to_bf16_array(_ptr(f), f.size, _ptr(out))
    return out


def f32_to_e4m3_bits(f) -> np.ndarray:
    f = _c(f, np.float32).reshape(-1)
    out = np.empty(f.size, np.uint8)
    _load().orc_f32_to_e4m3_array(_ptr(f), f.size, _ptr(out))
    return out


def e4m3_to_f32(b) -> np.ndarray:
    b = _c(b, np.uint8).reshape(-1)
    out = np.empty(b.size, np.float32)
    _load().orc_e4m3_to_f32_array(_ptr(b), b.size, _ptr(out))
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- routing --
def chunk_bounds(T: int, chunks: int) -> np.ndarray:
    b = np.zeros(chunks + 1, dtype=np.int64)
    _load().orc_chunk_bounds(int(T), int(chunks), _ptr(b))
    return b


def compute_send_counts(topk_idx, P: int, E_local: int, with_tokens_per_expert: bool = True):
    """-> dict(dest [T,K] i32, is_in_rank [T,P] u8, send_counts [P] i32,
    tokens_per_expert [P*E_local] i32 or None, err int)."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    dest = np.empty((T, K), np.int32)
    iir = np.empty((T, P), np.uint8)
    sc = np.empty(P, np.int32)
    tpe = np.empty(P * E_local, np.int32) if with_tokens_per_expert else None
    err = _load().orc_compute_send_counts(_ptr(idx), T, K, P, E_local, _ptr(dest), _ptr(iir),
                                          _ptr(sc), _ptr(tpe))
    return dict(dest=dest, is_in_rank=iir, send_counts=sc, tokens_per_expert=tpe, err=int(err))


def build_send_layout(topk_idx, topk_weights, dest, is_in_rank, E_local: int,
                      num_send: Optional[int] = None):
    """-> dict(send_token_idx [N] i32, send_rank [N] i32, send_idx [N,K] i64,
    send_w [N,K] f32, token_pos [T,P] i32, n int)."""
    idx = _c(topk_idx, np.int64)
    w = _c(topk_weights, np.float32)
    dest = _c(dest, np.int32)
    iir = _c(is_in_rank, np.uint8)
    T, K = idx.shape
    P = iir.shape[1]
    if num_send is None:
        num_send = int(iir.astype(np.int64).sum())
    sti = np.empty(num_send, np.int32)
    sr = np.empty(num_send, np.int32)
    si = np.empty((num_send, K), np.int64)
    sw = np.empty((num_send, K), np.float32)
    tp = np.empty((T, P), np.int32)
    n = _load().orc_build_send_layout(_ptr(idx), _ptr(w), _ptr(dest), _ptr(iir), T, K, P, E_local,
                                      num_send, _ptr(sti), _ptr(sr), _ptr(si), _ptr(sw), _ptr(tp))
    return dict(send_token_idx=sti, send_rank=sr, send_idx=si, send_w=sw, token_pos=tp, n=int(n))


# --------------------------------------------------------------- movement --
def dispatch(x, send_token_idx) -> np.ndarray:
    xb = _bf16_bits(x)
    T, H = xb.shape
    sti = _c(send_token_idx, np.int32)
    out = np.empty((sti.size, H), np.uint16)
    _load().orc_dispatch(_ptr(xb), H, _ptr(sti), sti.size, _ptr(out))
    return out


def quantize_fp8_rows(x):
    xb = _bf16_bits(x)
    R, H = xb.shape
    q = np.empty((R, H), np.uint8)
    s = np.empty((R, H // 128), np.float32)
    _load().orc_quantize_fp8_rows(_ptr(xb), R, H, _ptr(q), _ptr(s))
    return q, s


def quantize_fp8_rows_pow2(x):
    """Power-of-two group scales: -> (codes [R,H] u8, scales [R,H/128] f32, UE8M0 codes [R,H/128] u8)."""
    xb = _bf16_bits(x)
    R, H = xb.shape
    q = np.empty((R, H), np.uint8)
    s = np.empty((R, H // 128), np.float32)
    c = np.empty((R, H // 128), np.uint8)
    _load().orc_quantize_fp8_rows_pow2(_ptr(xb), R, H, _ptr(q), _ptr(s), _ptr(c))
    return q, s, c


SCALE_ROW_F32, SCALE_COL_F32, SCALE_COL_UE8M0 = 0, 1, 2


def batched_scale_shape(E_local: int, M: int, H: int, fmt: int):
    """Storage shape and dtype of the batched scales of each format (fmt 1 and
    2 are column-major in their last two dims, stored as [E_local, G, M])."""
    G = H // 128
    if fmt == SCALE_ROW_F32:
        return (E_local, M, G), np.float32
    if fmt == SCALE_COL_F32:
        return (E_local, G, M), np.float32
    return (E_local, G // 4, M), np.int32


def batched_prepare_fp8(x, topk_idx, E: int, E_local: int, rank: int, M: int, fmt: int = SCALE_ROW_F32,
                        round_scale: bool = False, zero_pad: bool = False, b_q_init=None, b_scale_init=None):
    """-> dict(b_q [E_local,M,H] u8, b_scale (storage layout of batched_scale_shape),
    tokens_per_expert, slot, err)."""
    xb = _bf16_bits(x)
    idx = _c(topk_idx, np.int64)
    T, H = xb.shape
    K = idx.shape[1]
    shape, dt = batched_scale_shape(E_local, M, H, fmt)
    b_q = np.zeros((E_local, M, H), np.uint8) if b_q_init is None else np.array(b_q_init, np.uint8, copy=True)
    b_s = np.zeros(shape, dt) if b_scale_init is None else np.array(b_scale_init, dt, copy=True)
    tpe = np.empty(E_local, np.int32)
    slot = np.empty((T, K), np.int32)
    err = _load().orc_batched_prepare_fp8(_ptr(xb), _ptr(idx), T, K, H, E, E_local, rank, M, _ptr(b_q),
                                          _ptr(b_s), int(fmt), int(round_scale), _ptr(tpe), _ptr(slot),
                                          int(zero_pad))
    return dict(b_q=b_q, b_scale=b_s, tokens_per_expert=tpe, slot=slot, err=int(err))


def expert_capacity(T: int, K: int, E: int, factor: float) -> int:
    return int(_load().orc_expert_capacity(T, K, E, float(factor)))


def batched_prepare_ex(x, topk_idx, E: int, E_local: int, rank: int, M: int, capacity: Optional[int] = None,
                       alignment: int = 1, fmt: Optional[int] = None, round_scale: bool = False,
                       zero_pad: bool = False, rows_init=None, scale_init=None):
    """Expert-batched prepare with a per-expert capacity and receive alignment.
    fmt None: bf16 rows (uint16 bits); else fp8 codes + scales in layout fmt.
    -> dict(b_rows, b_scale (or None), tokens_per_expert, slot, dropped, err)."""
    xb = _bf16_bits(x)
    idx = _c(topk_idx, np.int64)
    T, H = xb.shape
    K = idx.shape[1]
    C = M if capacity is None else int(capacity)
    if fmt is None:
        rows = np.zeros((E_local, M, H), np.uint16) if rows_init is None else np.array(rows_init, np.uint16)
        b_s = None
    else:
        rows = np.zeros((E_local, M, H), np.uint8) if rows_init is None else np.array(rows_init, np.uint8)
        shape, dt = batched_scale_shape(E_local, M, H, fmt)
        b_s = np.zeros(shape, dt) if scale_init is None else np.array(scale_init, dt)
    tpe = np.empty(E_local, np.int32)
    slot = np.empty((T, K), np.int32)
    dropped = np.empty(E_local, np.int32)
    err = _load().orc_batched_prepare_ex(_ptr(xb), _ptr(idx), T, K, H, E, E_local, rank, M, C, int(alignment),
                                         _ptr(rows), _ptr(b_s), -1 if fmt is None else int(fmt),
                                         int(round_scale), _ptr(tpe), _ptr(slot), _ptr(dropped), int(zero_pad))
    return dict(b_rows=rows, b_scale=b_s, tokens_per_expert=tpe, slot=slot, dropped=dropped, err=int(err))


def align_send_layout(layout: dict, send_counts, A: int) -> dict:
    """The send layout with every rank's segment padded to a multiple of A rows
    (pad rows: token -1, rank p, no experts); plus the aligned rank_offsets."""
    sc = _c(send_counts, np.int32)
    P = sc.shape[0]
    sti = _c(layout["send_token_idx"], np.int32)
    si = _c(layout["send_idx"], np.int64)
    sw = _c(layout["send_w"], np.float32)
    tp = _c(layout["token_pos"], np.int32)
    T = tp.shape[0]
    K = si.shape[1] if si.ndim == 2 else 1
    n = int(sum(-(-int(c) // A) * A for c in sc))
    ro = np.empty(P + 1, np.int32)
    a_ti = np.empty(max(n, 1), np.int32)
    a_r = np.empty(max(n, 1), np.int32)
    a_i = np.empty((max(n, 1), K), np.int64)
    a_w = np.empty((max(n, 1), K), np.float32)
    a_tp = np.empty((T, P), np.int32)
    got = _load().orc_align_send_layout(_ptr(sc), P, A, K, T, _ptr(sti), _ptr(si.reshape(-1, K)),
                                        _ptr(sw.reshape(-1, K)), _ptr(tp), _ptr(ro), _ptr(a_ti), _ptr(a_r),
                                        _ptr(a_i), _ptr(a_w), _ptr(a_tp))
    assert got == n
    return dict(n=n, rank_offsets=ro, send_token_idx=a_ti[:n], send_rank=a_r[:n], send_idx=a_i[:n],
                send_w=a_w[:n], token_pos=a_tp)


def indices_to_multihot(topk_idx, topk_probs, E: int):
    """-> dict(routing_map [T,E] u8, probs [T,E] f32, err)."""
    idx = _c(topk_idx, np.int64)
    pr = _c(topk_probs, np.float32)
    T, K = idx.shape
    rm = np.empty((T, E), np.uint8)
    dp = np.empty((T, E), np.float32)
    err = _load().orc_indices_to_multihot(_ptr(idx), _ptr(pr), T, K, E, _ptr(rm), _ptr(dp))
    return dict(routing_map=rm, probs=dp, err=int(err))


def dispatch_fp8(x, send_token_idx):
    xb = _bf16_bits(x)
    T, H = xb.shape
    sti = _c(send_token_idx, np.int32)
    q = np.empty((sti.size, H), np.uint8)
    s = np.empty((sti.size, H // 128), np.float32)
    _load().orc_dispatch_fp8(_ptr(xb), T, H, _ptr(sti), sti.size, _ptr(q), _ptr(s))
    return q, s


def local_expert_fp8(q, scale, send_idx, send_w) -> np.ndarray:
    q = _c(q, np.uint8)
    scale = _c(scale, np.float32)
    si = _c(send_idx, np.int64)
    sw = _c(send_w, np.float32)
    N, H = q.shape
    K = si.shape[1]
    out = np.empty((N, H), np.uint16)
    _load().orc_local_expert_fp8(_ptr(q), _ptr(scale), _ptr(si), _ptr(sw), N, K, H, _ptr(out))
    return out


def combine(y, token_pos, out_f32: bool = False) -> np.ndarray:
    yb = _bf16_bits(y)
    tp = _c(token_pos, np.int32)
    T, P = tp.shape
    H = yb.shape[1]
    out = np.empty((T, H), np.float32 if out_f32 else np.uint16)
    _load().orc_combine(_ptr(yb), T, H, P, _ptr(tp), int(out_f32), _ptr(out))
    return out


def batched_prepare(x, topk_idx, E: int, E_local: int, rank: int, M: int, zero_pad: bool = False,
                    b_x_init: Optional[np.ndarray] = None):
    """-> dict(b_x [E_local,M,H] u16, tokens_per_expert [E_local] i32, slot [T,K] i32, err)."""
    xb = _bf16_bits(x)
    idx = _c(topk_idx, np.int64)
    T, H = xb.shape
    K = idx.shape[1]
    if b_x_init is None:
        b_x = np.zeros((E_local, M, H), np.uint16)
    else:
        b_x = np.array(b_x_init, dtype=np.uint16, copy=True)
    tpe = np.empty(E_local, np.int32)
    slot = np.empty((T, K), np.int32)
    err = _load().orc_batched_prepare(_ptr(xb), _ptr(idx), T, K, H, E, E_local, rank, M,
                                      _ptr(b_x), _ptr(tpe), _ptr(slot), int(zero_pad))
    return dict(b_x=b_x, tokens_per_expert=tpe, slot=slot, err=int(err))


def batched_combine(y, topk_idx, topk_weights, slot, E_local: int, rank: int) -> np.ndarray:
    yb = _bf16_bits(y)
    idx = _c(topk_idx, np.int64)
    w = _c(topk_weights, np.float32)
    sl = _c(slot, np.int32)
    El, M, H = yb.shape
    assert El == E_local
    T, K = idx.shape
    out = np.empty((T, H), np.uint16)
    _load().orc_batched_combine(_ptr(yb), _ptr(idx), _ptr(w), _ptr(sl), T, K, H, E_local, rank,
                                M, _ptr(out))
    return out


# ------------------------------------------------------------- pipelines --
def send_path(x, topk_idx, topk_weights, y, P: int, E_local: int):
    """counts -> layout -> dispatch -> combine(y) for one problem; all results."""
    c = compute_send_counts(topk_idx, P, E_local)
    lay = build_send_layout(topk_idx, topk_weights, c["dest"], c["is_in_rank"], E_local)
    recv = dispatch(x, lay["send_token_idx"])
    out = combine(y, lay["token_pos"]) if y is not None else None
    return dict(counts=c, layout=lay, recv_x=recv, out=out)
