"""GB300 (sm_103a) MoE top-k token dispatch / combine.

Thin ctypes binding over ``libep_gb300.so`` (C ABI in ``include/ep.h``).  The
``ep_*`` functions here have the same names and argument order as the C
entry points and only marshal arguments: torch tensors become device pointers,
the current CUDA stream is passed through, and a non-OK status raises
:class:`EPError`.  Every step runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and using the binding without the built library on a
CUDA device raises.

The lower-case helpers after them allocate outputs with torch and call the
``ep_*`` entry points:

- send layout, following the axolotl ``integrations.expert_parallel.
  torch_dispatch`` page: ``compute_send_counts``, ``build_send_layout``,
  ``dispatch`` / ``combine`` (the host-synchronising call order),
  ``route_nosync`` (worst-case rows, no host round trip), ``dispatch_rows``,
  ``combine_rows``, ``chunk_bounds``, ``dispatch_chunked_forward``,
  ``dispatch_chunked_forward_nosync`` and ``ChunkedForward`` (buffers kept for
  repeated or graph-captured calls), ``local_expert_fp8`` (the synthetic
  expert of the chunked fp8 workload);
- expert-batched layout, following the vLLM ``BatchedPrepareAndFinalize``
  page and the NeMo ``uccl_ep.buffer`` low-latency calls:
  ``batched_prepare``, ``batched_prepare_fp8`` (scale layouts),
  ``batched_prepare_ex`` (capacity and alignment, NeMo token-dispatcher
  options), ``expert_capacity``, ``batched_combine``;
- ``indices_to_multihot``: the NeMo token dispatchers' routing map and dense
  probabilities;
- ``workspace``, ``combine_ws``, ``error_word``: scratch and the device error
  word, allocated the way the entry points expect.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import _build

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_INVALID_EXPERT = 2
EP_ERR_COUNT_MISMATCH = 4
EP_ERR_CAPACITY = 8
EP_ERR_UNSUPPORTED = 16
EP_ERR_CUDA = 32
EP_ERR_TIMEOUT = 64

_ERR_NAMES = {
    EP_ERR_INVALID_ARG: "EP_ERR_INVALID_ARG", EP_ERR_INVALID_EXPERT: "EP_ERR_INVALID_EXPERT",
    EP_ERR_COUNT_MISMATCH: "EP_ERR_COUNT_MISMATCH", EP_ERR_CAPACITY: "EP_ERR_CAPACITY",
    EP_ERR_UNSUPPORTED: "EP_ERR_UNSUPPORTED", EP_ERR_CUDA: "EP_ERR_CUDA",
    EP_ERR_TIMEOUT: "EP_ERR_TIMEOUT",
}


class EPError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        names = [n for b, n in _ERR_NAMES.items() if status & b] or [str(status)]
        super().__init__(f"{where}: {'|'.join(names)}" if where else "|".join(names))
        self.status = status


_lib = None
_VP, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

_SIGNATURES = {
    "ep_status_str": (ctypes.c_char_p, [_I32]),
    "ep_workspace_size": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "ep_chunk_bounds": (_I32, [_I64, _I32, _VP]),
    "ep_compute_send_counts": (_I32, [_VP, _I64, _I32, _I32, _I32, _VP, _I32, _VP, _VP, _VP, _VP, _VP,
                                      _VP, _SZ, _VP, _VP]),
    "ep_build_send_layout": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _I64, _VP, _VP, _VP, _VP,
                                    _VP, _VP, _SZ, _VP, _VP]),
    "ep_dispatch": (_I32, [_VP, _I64, _I32, _VP, _I32, _I64, _VP, _VP, _I32, _VP, _VP]),
    "ep_combine": (_I32, [_VP, _I64, _I32, _VP, _I32, _I64, _VP, _I32, _VP, _SZ, _VP, _VP]),
    "ep_batched_prepare": (_I32, [_VP, _VP, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _I32,
                                  _VP, _SZ, _VP, _VP]),
    "ep_batched_combine": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _SZ, _VP,
                                  _VP]),
    "ep_local_expert_fp8": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _VP, _VP, _VP]),
    "ep_route_nosync": (_I32, [_VP, _VP, _I64, _I32, _I32, _I32, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                               _VP, _VP, _VP, _SZ, _VP, _VP]),
    "ep_local_expert_fp8_callback": (_I32, [_VP, _I32, _I64, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "ep_compute_send_counts_noalloc": (_I32, [_VP, _I64, _I32, _I32, _I32, _VP, _I32, _VP, _VP, _VP, _VP, _VP,
                                              _VP, _VP]),
    "ep_local_expert_fp8_dev_callback": (_I32, [_VP, _I32, _I64, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                                _VP]),
    "ep_batched_prepare_fp8": (_I32, [_VP, _VP, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _I32, _I32,
                                      _VP, _VP, _I32, _VP, _SZ, _VP, _VP]),
    "ep_batched_prepare_ex": (_I32, [_VP, _VP, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _VP, _VP,
                                     _I32, _I32, _VP, _VP, _VP, _I32, _VP, _SZ, _VP, _VP]),
    "ep_expert_capacity": (_I64, [_I64, _I32, _I32, ctypes.c_double]),
    "ep_route_nosync_aligned": (_I32, [_VP, _VP, _I64, _I32, _I32, _I32, _I64, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                       _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "ep_indices_to_multihot": (_I32, [_VP, _VP, _I64, _I32, _I32, _VP, _VP, _VP, _VP]),
    "ep_dispatch_nosync": (_I32, [_VP, _VP, _VP, _I64, _I32, _I32, _I32, _I32, _I64, _I32, _VP, _VP, _VP, _VP, _VP,
                                  _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
}

EP_SCALE_ROW_F32, EP_SCALE_COL_F32, EP_SCALE_COL_UE8M0 = 0, 1, 2


class EPChunkBuffers(ctypes.Structure):
    """ep_chunk_buffers of include/ep.h."""
    _fields_ = [("dest", _VP), ("is_in_rank", _VP), ("send_counts", _VP), ("rank_offsets", _VP),
                ("token_pos", _VP), ("max_rows", _I64), ("send_token_idx", _VP), ("send_rank", _VP),
                ("send_idx", _VP), ("send_w", _VP), ("recv_x", _VP), ("recv_scale", _VP), ("local_out", _VP),
                ("ws", _VP), ("ws_bytes", _SZ), ("combine_ws", _VP)]


LOCAL_KERNEL_FN = ctypes.CFUNCTYPE(_I32, _VP, _I32, _I64, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP)


class EPRowSet(ctypes.Structure):
    """ep_row_set of include/ep.h."""
    _fields_ = [("send_token_idx", _VP), ("send_rank", _VP), ("send_idx", _VP), ("send_w", _VP),
                ("recv_x", _VP), ("recv_scale", _VP), ("local_out", _VP)]


class EPPipelineBuffers(ctypes.Structure):
    """ep_pipeline_buffers of include/ep.h."""
    _fields_ = [("dest", _VP), ("is_in_rank", _VP), ("send_counts", _VP), ("rank_offsets", _VP),
                ("token_pos", _VP), ("max_rows", _I64), ("n_sets", _I32), ("sets", EPRowSet * 2),
                ("ws", _VP), ("ws_bytes", _SZ), ("combine_ws", _VP)]


LOCAL_KERNEL_DEV_FN = ctypes.CFUNCTYPE(_I32, _VP, _I32, _I64, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP)


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libep_gb300.so (building it first if asked and needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libep_gb300.so is not built ({path}); run combine_send_counts_gb300._build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    lib.ep_dispatch_chunked_forward.restype = _I32
    lib.ep_dispatch_chunked_forward.argtypes = [_VP, _VP, _VP, _I64, _I32, _I32, _I32, _I32, _I32, _I32,
                                                LOCAL_KERNEL_FN, _VP, _VP, ctypes.POINTER(EPChunkBuffers), _VP,
                                                _VP, _VP]
    lib.ep_dispatch_chunked_forward_nosync.restype = _I32
    lib.ep_dispatch_chunked_forward_nosync.argtypes = [_VP, _VP, _VP, _I64, _I32, _I32, _I32, _I32, _I32, _I32,
                                                       LOCAL_KERNEL_DEV_FN, _VP, _VP,
                                                       ctypes.POINTER(EPPipelineBuffers), _VP, _VP, _VP]
    _lib = lib
    return lib


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str):
    if rc != EP_OK:
        raise EPError(rc, where)


def _expect(where: str, **tensors):
    """dtype checks of the allocating helpers: name=(tensor, dtype or tuple of
    dtypes); None tensors are skipped.  The C ABI takes untyped pointers, so a
    tensor of the wrong type would otherwise be read as the expected one."""
    for name, (t, dt) in tensors.items():
        if t is None:
            continue
        want = dt if isinstance(dt, tuple) else (dt,)
        if t.dtype not in want:
            raise TypeError(f"{where}: {name} must be {' or '.join(str(d) for d in want)}, got {t.dtype}")


# ------------------------------------------------------------- C ABI names --
def ep_status_str(status: int) -> str:
    return load().ep_status_str(int(status)).decode()


def ep_workspace_size(T: int, K: int, P: int, E_local: int, chunks: int = 1) -> int:
    return int(load().ep_workspace_size(int(T), int(K), int(P), int(E_local), int(chunks)))


def ep_chunk_bounds(T: int, chunks: int) -> list:
    buf = (ctypes.c_int64 * (chunks + 1))()
    _check(load().ep_chunk_bounds(int(T), int(chunks), buf), "ep_chunk_bounds")
    return list(buf)


def ep_compute_send_counts(topk_idx, T, K, P, E_local, h_chunk_bounds, chunks, dest, is_in_rank,
                           send_counts, rank_offsets, tokens_per_expert, ws, err, stream=None):
    hb = None
    if h_chunk_bounds is not None:
        hb = (ctypes.c_int64 * len(h_chunk_bounds))(*[int(v) for v in h_chunk_bounds])
    rc = load().ep_compute_send_counts(_p(topk_idx), int(T), int(K), int(P), int(E_local), hb, int(chunks),
                                       _p(dest), _p(is_in_rank), _p(send_counts), _p(rank_offsets),
                                       _p(tokens_per_expert), _p(ws), ws.numel() * ws.element_size(),
                                       _p(err), _stream(stream))
    _check(rc, "ep_compute_send_counts")


def ep_build_send_layout(topk_idx, topk_weights, dest, is_in_rank, T, K, P, E_local, num_send,
                         send_token_idx, send_rank, send_idx, send_w, token_pos, ws, err, stream=None):
    rc = load().ep_build_send_layout(_p(topk_idx), _p(topk_weights), _p(dest), _p(is_in_rank), int(T), int(K),
                                     int(P), int(E_local), int(num_send), _p(send_token_idx), _p(send_rank),
                                     _p(send_idx), _p(send_w), _p(token_pos), _p(ws),
                                     ws.numel() * ws.element_size(), _p(err), _stream(stream))
    _check(rc, "ep_build_send_layout")


def ep_route_nosync(topk_idx, topk_weights, T, K, P, E_local, num_worst_rows, dest, is_in_rank, send_counts,
                    rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w, token_pos, ws, err,
                    stream=None):
    rc = load().ep_route_nosync(_p(topk_idx), _p(topk_weights), int(T), int(K), int(P), int(E_local),
                                int(num_worst_rows), _p(dest), _p(is_in_rank), _p(send_counts), _p(rank_offsets),
                                _p(tokens_per_expert), _p(send_token_idx), _p(send_rank), _p(send_idx), _p(send_w),
                                _p(token_pos), _p(ws), ws.numel() * ws.element_size(), _p(err), _stream(stream))
    _check(rc, "ep_route_nosync")


def ep_route_nosync_aligned(topk_idx, topk_weights, T, K, P, E_local, num_worst_rows, alignment, dest, is_in_rank,
                            send_counts, rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx,
                            send_w, token_pos, ws, err, stream=None):
    rc = load().ep_route_nosync_aligned(_p(topk_idx), _p(topk_weights), int(T), int(K), int(P), int(E_local),
                                        int(num_worst_rows), int(alignment), _p(dest), _p(is_in_rank),
                                        _p(send_counts), _p(rank_offsets), _p(tokens_per_expert),
                                        _p(send_token_idx), _p(send_rank), _p(send_idx), _p(send_w), _p(token_pos),
                                        _p(ws), ws.numel() * ws.element_size(), _p(err), _stream(stream))
    _check(rc, "ep_route_nosync_aligned")


def ep_dispatch(x, T, H, token_pos, P, num_send, recv_x, recv_scale, fp8, err, stream=None):
    rc = load().ep_dispatch(_p(x), int(T), int(H), _p(token_pos), int(P), int(num_send), _p(recv_x),
                            _p(recv_scale), int(fp8), _p(err), _stream(stream))
    _check(rc, "ep_dispatch")


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def ep_combine(y, T, H, token_pos, P, num_send, out, out_dtype, ws, err, stream=None):
    rc = load().ep_combine(_p(y), int(T), int(H), _p(token_pos), int(P), int(num_send), _p(out),
                           int(out_dtype), _p(ws), _nbytes(ws), _p(err), _stream(stream))
    _check(rc, "ep_combine")


def ep_batched_prepare(x, topk_idx, T, K, H, E, E_local, rank, max_num_tokens, b_x, tokens_per_expert,
                       slot, zero_pad, ws, err, stream=None):
    rc = load().ep_batched_prepare(_p(x), _p(topk_idx), int(T), int(K), int(H), int(E), int(E_local),
                                   int(rank), int(max_num_tokens), _p(b_x), _p(tokens_per_expert), _p(slot),
                                   int(zero_pad), _p(ws), ws.numel() * ws.element_size(), _p(err),
                                   _stream(stream))
    _check(rc, "ep_batched_prepare")


def ep_batched_prepare_fp8(x, topk_idx, T, K, H, E, E_local, rank, max_num_tokens, b_q, b_scale, scale_fmt,
                           round_scale, tokens_per_expert, slot, zero_pad, ws, err, stream=None):
    rc = load().ep_batched_prepare_fp8(_p(x), _p(topk_idx), int(T), int(K), int(H), int(E), int(E_local),
                                       int(rank), int(max_num_tokens), _p(b_q), _p(b_scale), int(scale_fmt),
                                       int(round_scale), _p(tokens_per_expert), _p(slot), int(zero_pad), _p(ws),
                                       ws.numel() * ws.element_size(), _p(err), _stream(stream))
    _check(rc, "ep_batched_prepare_fp8")


def ep_batched_combine(y, topk_idx, topk_weights, slot, T, K, H, E_local, rank, max_num_tokens, out, ws, err,
                       stream=None):
    rc = load().ep_batched_combine(_p(y), _p(topk_idx), _p(topk_weights), _p(slot), int(T), int(K), int(H),
                                   int(E_local), int(rank), int(max_num_tokens), _p(out), _p(ws), _nbytes(ws),
                                   _p(err), _stream(stream))
    _check(rc, "ep_batched_combine")


def ep_local_expert_fp8(recv_q, recv_scale, send_idx, send_w, N, K, H, out, err, stream=None):
    rc = load().ep_local_expert_fp8(_p(recv_q), _p(recv_scale), _p(send_idx), _p(send_w), int(N), int(K),
                                    int(H), _p(out), _p(err), _stream(stream))
    _check(rc, "ep_local_expert_fp8")


def ep_compute_send_counts_noalloc(topk_idx, T, K, P, E_local, h_chunk_bounds, chunks, dest, is_in_rank,
                                   send_counts, rank_offsets, tokens_per_expert, err, stream=None):
    """ep_compute_send_counts without a workspace argument, for callers that
    cannot allocate device memory: the library's own fixed device array holds
    the scratch (its size limit and sharing rules are stated beside the C
    declaration)."""
    hb = None
    if h_chunk_bounds is not None:
        hb = (ctypes.c_int64 * len(h_chunk_bounds))(*[int(v) for v in h_chunk_bounds])
    rc = load().ep_compute_send_counts_noalloc(_p(topk_idx), int(T), int(K), int(P), int(E_local), hb,
                                               int(chunks), _p(dest), _p(is_in_rank), _p(send_counts),
                                               _p(rank_offsets), _p(tokens_per_expert), _p(err), _stream(stream))
    _check(rc, "ep_compute_send_counts_noalloc")


def ep_dispatch_chunked_forward(x, topk_idx, topk_weights, T, K, H, P, E_local, chunks, fp8, local_kernel, user,
                                out, buffers: EPChunkBuffers, h_counts, err, stream=None):
    """local_kernel: a LOCAL_KERNEL_FN (ctypes callback or the library's
    ep_local_expert_fp8_callback); h_counts: pinned host int32 [chunks*P]."""
    rc = load().ep_dispatch_chunked_forward(_p(x), _p(topk_idx), _p(topk_weights), int(T), int(K), int(H), int(P),
                                            int(E_local), int(chunks), int(fp8), local_kernel, user, _p(out),
                                            ctypes.byref(buffers), ctypes.c_void_p(h_counts.data_ptr()), _p(err),
                                            _stream(stream))
    _check(rc, "ep_dispatch_chunked_forward")


def ep_local_expert_fp8_callback():
    """The library's synthetic fp8 expert as a LOCAL_KERNEL_FN."""
    return LOCAL_KERNEL_FN(ctypes.cast(load().ep_local_expert_fp8_callback, ctypes.c_void_p).value)


def ep_dispatch_chunked_forward_nosync(x, topk_idx, topk_weights, T, K, H, P, E_local, chunks, fp8, local_kernel,
                                       user, out, buffers: EPPipelineBuffers, err, stream=None, aux_stream=None):
    """local_kernel: a LOCAL_KERNEL_DEV_FN (ctypes callback or the library's
    ep_local_expert_fp8_dev_callback); aux_stream: the producer stream (two
    row sets) or None (one set)."""
    aux = None if aux_stream is None else _stream(aux_stream)
    rc = load().ep_dispatch_chunked_forward_nosync(_p(x), _p(topk_idx), _p(topk_weights), int(T), int(K), int(H),
                                                   int(P), int(E_local), int(chunks), int(fp8), local_kernel, user,
                                                   _p(out), ctypes.byref(buffers), _p(err), _stream(stream), aux)
    _check(rc, "ep_dispatch_chunked_forward_nosync")


def ep_local_expert_fp8_dev_callback():
    """The library's synthetic fp8 expert as a LOCAL_KERNEL_DEV_FN."""
    return LOCAL_KERNEL_DEV_FN(ctypes.cast(load().ep_local_expert_fp8_dev_callback, ctypes.c_void_p).value)


# ------------------------------------------------------------------ helpers --
def workspace(T: int, K: int, P: int, E_local: int, chunks: int = 1, device=None) -> torch.Tensor:
    """A device workspace of ep_workspace_size bytes (torch allocations are 256-B aligned)."""
    n = max(ep_workspace_size(T, K, P, E_local, chunks), 256)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def error_word(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def raise_device_error(err: torch.Tensor, where: str = "device"):
    """Synchronise and raise EPError if the device error word is non-zero."""
    v = int(err.item())
    if v:
        raise EPError(v, where)


def chunk_bounds(num_tokens: int, chunks: int) -> list:
    return ep_chunk_bounds(num_tokens, chunks)


def compute_send_counts(topk_idx: torch.Tensor, num_ranks: int, num_local_experts: int,
                        chunk_bounds: Optional[Sequence[int]] = None, ws=None, err=None, stream=None,
                        with_tokens_per_expert: bool = True):
    """-> dict(dest, is_in_rank, send_counts [C,P], rank_offsets [C,P+1], tokens_per_expert)."""
    _expect("compute_send_counts", topk_idx=(topk_idx, torch.int64))
    T, K = topk_idx.shape
    P, El = num_ranks, num_local_experts
    C = len(chunk_bounds) - 1 if chunk_bounds is not None else 1
    dev = topk_idx.device
    out = dict(
        dest=torch.empty((T, K), dtype=torch.int32, device=dev),
        is_in_rank=torch.empty((T, P), dtype=torch.uint8, device=dev),
        send_counts=torch.empty((C, P), dtype=torch.int32, device=dev),
        rank_offsets=torch.empty((C, P + 1), dtype=torch.int32, device=dev),
        tokens_per_expert=torch.empty(P * El, dtype=torch.int32, device=dev) if with_tokens_per_expert else None,
    )
    ws = ws if ws is not None else workspace(T, K, P, El, C, dev)
    err = err if err is not None else error_word(dev)
    ep_compute_send_counts(topk_idx, T, K, P, El, chunk_bounds if C > 1 else None, C, out["dest"],
                           out["is_in_rank"], out["send_counts"], out["rank_offsets"], out["tokens_per_expert"],
                           ws, err, stream)
    out["err"] = err
    return out


def build_send_layout(topk_idx, topk_weights, dest, is_in_rank, num_send: int, num_local_experts: int,
                      ws=None, err=None, stream=None):
    """-> dict(send_token_idx [N], send_rank [N], send_idx [N,K], send_w [N,K], token_pos [T,P])."""
    _expect("build_send_layout", topk_idx=(topk_idx, torch.int64), topk_weights=(topk_weights, torch.float32),
            dest=(dest, torch.int32), is_in_rank=(is_in_rank, torch.uint8))
    T, K = topk_idx.shape
    P = is_in_rank.shape[1]
    dev = topk_idx.device
    N = int(num_send)
    out = dict(
        send_token_idx=torch.empty(N, dtype=torch.int32, device=dev),
        send_rank=torch.empty(N, dtype=torch.int32, device=dev),
        send_idx=torch.empty((N, K), dtype=torch.int64, device=dev),
        send_w=torch.empty((N, K), dtype=torch.float32, device=dev),
        token_pos=torch.empty((T, P), dtype=torch.int32, device=dev),
    )
    ws = ws if ws is not None else workspace(T, K, P, num_local_experts, 1, dev)
    err = err if err is not None else error_word(dev)
    ep_build_send_layout(topk_idx, topk_weights, dest, is_in_rank, T, K, P, num_local_experts, N,
                         out["send_token_idx"], out["send_rank"], out["send_idx"], out["send_w"],
                         out["token_pos"], ws, err, stream)
    out["err"] = err
    return out


def route_nosync(topk_idx, topk_weights, num_ranks: int, num_local_experts: int, num_worst_rows: Optional[int] = None,
                 ws=None, err=None, stream=None, with_tokens_per_expert: bool = True, alignment: int = 1):
    """Counts and send layout in one call with rows sized for the worst case
    (no host round trip).  rank_offsets[P] holds the number of rows used.
    alignment > 1 starts every rank segment at a multiple of it (pad rows
    carry no token) and rounds tokens_per_expert up."""
    _expect("route_nosync", topk_idx=(topk_idx, torch.int64), topk_weights=(topk_weights, torch.float32))
    T, K = topk_idx.shape
    P, El = num_ranks, num_local_experts
    W = T * min(K, P) + P * (alignment - 1) if num_worst_rows is None else int(num_worst_rows)
    dev = topk_idx.device
    out = dict(
        dest=torch.empty((T, K), dtype=torch.int32, device=dev),
        is_in_rank=torch.empty((T, P), dtype=torch.uint8, device=dev),
        send_counts=torch.empty(P, dtype=torch.int32, device=dev),
        rank_offsets=torch.empty(P + 1, dtype=torch.int32, device=dev),
        tokens_per_expert=torch.empty(P * El, dtype=torch.int32, device=dev) if with_tokens_per_expert else None,
        send_token_idx=torch.empty(W, dtype=torch.int32, device=dev),
        send_rank=torch.empty(W, dtype=torch.int32, device=dev),
        send_idx=torch.empty((W, K), dtype=torch.int64, device=dev),
        send_w=torch.empty((W, K), dtype=torch.float32, device=dev),
        token_pos=torch.empty((T, P), dtype=torch.int32, device=dev),
        num_worst_rows=W,
    )
    ws = ws if ws is not None else workspace(T, K, P, El, 1, dev)
    err = err if err is not None else error_word(dev)
    ep_route_nosync_aligned(topk_idx, topk_weights, T, K, P, El, W, alignment, out["dest"], out["is_in_rank"],
                            out["send_counts"], out["rank_offsets"], out["tokens_per_expert"], out["send_token_idx"],
                            out["send_rank"], out["send_idx"], out["send_w"], out["token_pos"], ws, err, stream)
    out["err"] = err
    return out


def dispatch_rows(x: torch.Tensor, token_pos: torch.Tensor, num_send: int, fp8: bool = False, err=None,
                  stream=None):
    """recv_x [N,H] bf16, or (recv_q [N,H] e4m3 as uint8, recv_scale [N,H/128] fp32) when fp8."""
    _expect("dispatch_rows", x=(x, torch.bfloat16), token_pos=(token_pos, torch.int32))
    T, H = x.shape
    P = token_pos.shape[1]
    err = err if err is not None else error_word(x.device)
    if fp8:
        q = torch.empty((num_send, H), dtype=torch.uint8, device=x.device)
        s = torch.empty((num_send, H // 128), dtype=torch.float32, device=x.device)
        ep_dispatch(x, T, H, token_pos, P, num_send, q, s, 1, err, stream)
        return q, s
    recv = torch.empty((num_send, H), dtype=x.dtype, device=x.device)
    ep_dispatch(x, T, H, token_pos, P, num_send, recv, None, 0, err, stream)
    return recv


EP_COMBINE_WS_BYTES = 16


def combine_ws(device=None) -> torch.Tensor:
    """Scratch for ep_combine / ep_batched_combine (lets the SMs share work)."""
    return torch.empty(256, dtype=torch.uint8, device=device or "cuda")


def combine_rows(y: torch.Tensor, token_pos: torch.Tensor, out_dtype=torch.bfloat16, err=None, stream=None,
                 ws="auto"):
    """ws: "auto" (a fresh scratch), a device tensor, or None (static work split)."""
    _expect("combine_rows", y=(y, torch.bfloat16), token_pos=(token_pos, torch.int32))
    T, P = token_pos.shape
    N, H = y.shape
    out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    err = err if err is not None else error_word(y.device)
    ws = combine_ws(y.device) if isinstance(ws, str) else ws
    ep_combine(y, T, H, token_pos, P, N, out, 1 if out_dtype == torch.float32 else 0, ws, err, stream)
    return out


def dispatch(x, topk_idx, topk_weights, *, num_local_experts: int, num_ranks: int, fp8: bool = False):
    """The collective-free local path of the axolotl dispatch: counts, one
    device-to-host copy of the counts, layout, row scatter.
    Returns (recv_x, recv_idx, recv_w, handle)."""
    c = compute_send_counts(topk_idx, num_ranks, num_local_experts, with_tokens_per_expert=False)
    num_send = int(c["send_counts"].sum().item())
    lay = build_send_layout(topk_idx, topk_weights, c["dest"], c["is_in_rank"], num_send, num_local_experts)
    recv = dispatch_rows(x, lay["token_pos"], num_send, fp8=fp8)
    handle = dict(num_tokens=x.shape[0], token_pos=lay["token_pos"], send_counts=c["send_counts"],
                  send_token_idx=lay["send_token_idx"], err=c["err"])
    return recv, lay["send_idx"], lay["send_w"], handle


def combine(local_out: torch.Tensor, handle: dict, dtype=None):
    return combine_rows(local_out, handle["token_pos"], out_dtype=dtype or torch.bfloat16)


def batched_prepare(x, topk_idx, num_experts: int, num_local_experts: int, rank: int, max_num_tokens: int,
                    zero_pad: bool = False, err=None, stream=None, ws=None):
    """-> dict(b_x [E_local,M,H], tokens_per_expert [E_local], slot [T,K]).
    ws: a workspace of at least ep_workspace_size bytes, or None for a new one."""
    _expect("batched_prepare", x=(x, torch.bfloat16), topk_idx=(topk_idx, torch.int64))
    T, H = x.shape
    K = topk_idx.shape[1]
    El = num_local_experts
    dev = x.device
    b_x = torch.empty((El, max_num_tokens, H), dtype=x.dtype, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws = ws if ws is not None else workspace(T, K, num_experts // El, El, 1, dev)
    err = err if err is not None else error_word(dev)
    ep_batched_prepare(x, topk_idx, T, K, H, num_experts, El, rank, max_num_tokens, b_x, tpe, slot,
                       int(zero_pad), ws, err, stream)
    return dict(b_x=b_x, tokens_per_expert=tpe, slot=slot, err=err)


def ep_batched_prepare_ex(x, topk_idx, T, K, H, E, E_local, rank, max_num_tokens, capacity, alignment, b_rows,
                          b_scale, scale_fmt, round_scale, tokens_per_expert, slot, dropped, zero_pad, ws, err,
                          stream=None):
    rc = load().ep_batched_prepare_ex(_p(x), _p(topk_idx), int(T), int(K), int(H), int(E), int(E_local), int(rank),
                                      int(max_num_tokens), int(capacity), int(alignment), _p(b_rows), _p(b_scale),
                                      int(scale_fmt), int(round_scale), _p(tokens_per_expert), _p(slot),
                                      _p(dropped), int(zero_pad), _p(ws), ws.numel() * ws.element_size(), _p(err),
                                      _stream(stream))
    _check(rc, "ep_batched_prepare_ex")


def ep_dispatch_nosync(x, topk_idx, topk_weights, T, K, H, P, E_local, num_worst_rows, fp8, dest, is_in_rank,
                       send_counts, rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w,
                       token_pos, recv_x, recv_scale, ws, err, stream=None):
    rc = load().ep_dispatch_nosync(_p(x), _p(topk_idx), _p(topk_weights), int(T), int(K), int(H), int(P),
                                   int(E_local), int(num_worst_rows), int(fp8), _p(dest), _p(is_in_rank),
                                   _p(send_counts), _p(rank_offsets), _p(tokens_per_expert), _p(send_token_idx),
                                   _p(send_rank), _p(send_idx), _p(send_w), _p(token_pos), _p(recv_x),
                                   _p(recv_scale), _p(ws), ws.numel() * ws.element_size(), _p(err), _stream(stream))
    _check(rc, "ep_dispatch_nosync")


def ep_indices_to_multihot(topk_idx, topk_probs, T, K, E, routing_map, probs, err, stream=None):
    rc = load().ep_indices_to_multihot(_p(topk_idx), _p(topk_probs), int(T), int(K), int(E), _p(routing_map),
                                       _p(probs), _p(err), _stream(stream))
    _check(rc, "ep_indices_to_multihot")


def indices_to_multihot(topk_idx, topk_probs, num_experts: int, err=None, stream=None):
    """-> (routing_map [T,E] bool, probs [T,E] fp32): the multihot view of top-k routing."""
    _expect("indices_to_multihot", topk_idx=(topk_idx, torch.int64), topk_probs=(topk_probs, torch.float32))
    T, K = topk_idx.shape
    dev = topk_idx.device
    rm = torch.empty((T, num_experts), dtype=torch.bool, device=dev)
    pr = torch.empty((T, num_experts), dtype=torch.float32, device=dev)
    err = err if err is not None else error_word(dev)
    ep_indices_to_multihot(topk_idx, topk_probs, T, K, num_experts, rm, pr, err, stream)
    return rm, pr


def ep_expert_capacity(T: int, K: int, E: int, factor: float) -> int:
    v = int(load().ep_expert_capacity(int(T), int(K), int(E), float(factor)))
    if v < 0:
        raise EPError(EP_ERR_INVALID_ARG, "ep_expert_capacity")
    return v


def expert_capacity(num_tokens: int, topk: int, num_experts: int, capacity_factor: float) -> int:
    """Tokens each expert keeps under a capacity factor: ceil(factor * T * K / E)."""
    return ep_expert_capacity(num_tokens, topk, num_experts, capacity_factor)


def batched_prepare_ex(x, topk_idx, num_experts: int, num_local_experts: int, rank: int, max_num_tokens: int, *,
                       capacity: int = 0, alignment: int = 1, scale_fmt: Optional[int] = None,
                       round_scale: bool = False, zero_pad: bool = False, err=None, stream=None, ws=None):
    """Expert-batched prepare with a per-expert capacity (0: max_num_tokens,
    overflow is an error; else later tokens are dropped and counted) and a
    receive alignment.  scale_fmt None: bf16 rows; else fp8 codes + scales.
    ws: a workspace of at least ep_workspace_size bytes, or None for a new one.
    -> dict(b_rows, b_scale, tokens_per_expert, slot, dropped, err)."""
    _expect("batched_prepare_ex", x=(x, torch.bfloat16), topk_idx=(topk_idx, torch.int64))
    T, H = x.shape
    K = topk_idx.shape[1]
    El, M = num_local_experts, max_num_tokens
    dev = x.device
    fp8 = scale_fmt is not None
    b_rows = torch.empty((El, M, H), dtype=torch.uint8 if fp8 else x.dtype, device=dev)
    b_s = None
    if fp8:
        shape, dt = batched_scale_storage(El, M, H, scale_fmt)
        b_s = torch.empty(shape, dtype=dt, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    dropped = torch.empty(El, dtype=torch.int32, device=dev)
    ws = ws if ws is not None else workspace(T, K, num_experts // El, El, 1, dev)
    err = err if err is not None else error_word(dev)
    ep_batched_prepare_ex(x, topk_idx, T, K, H, num_experts, El, rank, M, capacity, alignment, b_rows, b_s,
                          -1 if not fp8 else scale_fmt, int(round_scale), tpe, slot, dropped, int(zero_pad), ws,
                          err, stream)
    return dict(b_rows=b_rows, b_scale=b_s, tokens_per_expert=tpe, slot=slot, dropped=dropped, err=err)


def batched_scale_storage(E_local: int, M: int, H: int, scale_fmt: int):
    """(shape, dtype) of the scale tensor of each EP_SCALE_* layout, in storage
    order: the column-major layouts are stored as [E_local, groups, M]."""
    G = H // 128
    if scale_fmt == EP_SCALE_ROW_F32:
        return (E_local, M, G), torch.float32
    if scale_fmt == EP_SCALE_COL_F32:
        return (E_local, G, M), torch.float32
    return (E_local, G // 4, M), torch.int32


def batched_prepare_fp8(x, topk_idx, num_experts: int, num_local_experts: int, rank: int, max_num_tokens: int,
                        scale_fmt: int = EP_SCALE_ROW_F32, round_scale: bool = False, zero_pad: bool = False,
                        err=None, stream=None, ws=None):
    """-> dict(b_q [E_local,M,H] uint8 (e4m3 codes), b_scale (batched_scale_storage),
    tokens_per_expert [E_local], slot [T,K]).  ws: a workspace of at least
    ep_workspace_size bytes, or None for a new one."""
    _expect("batched_prepare_fp8", x=(x, torch.bfloat16), topk_idx=(topk_idx, torch.int64))
    T, H = x.shape
    K = topk_idx.shape[1]
    El = num_local_experts
    dev = x.device
    b_q = torch.empty((El, max_num_tokens, H), dtype=torch.uint8, device=dev)
    shape, dt = batched_scale_storage(El, max_num_tokens, H, scale_fmt)
    b_s = torch.empty(shape, dtype=dt, device=dev)
    tpe = torch.empty(El, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws = ws if ws is not None else workspace(T, K, num_experts // El, El, 1, dev)
    err = err if err is not None else error_word(dev)
    ep_batched_prepare_fp8(x, topk_idx, T, K, H, num_experts, El, rank, max_num_tokens, b_q, b_s, scale_fmt,
                           int(round_scale), tpe, slot, int(zero_pad), ws, err, stream)
    return dict(b_q=b_q, b_scale=b_s, tokens_per_expert=tpe, slot=slot, err=err)


def batched_combine(y, topk_idx, topk_weights, slot, rank: int, err=None, stream=None, ws="auto"):
    _expect("batched_combine", y=(y, torch.bfloat16), topk_idx=(topk_idx, torch.int64),
            topk_weights=(topk_weights, torch.float32), slot=(slot, torch.int32))
    El, M, H = y.shape
    T, K = topk_idx.shape
    out = torch.empty((T, H), dtype=y.dtype, device=y.device)
    err = err if err is not None else error_word(y.device)
    ws = combine_ws(y.device) if isinstance(ws, str) else ws
    ep_batched_combine(y, topk_idx, topk_weights, slot, T, K, H, El, rank, M, out, ws, err, stream)
    return out


def local_expert_fp8(recv_q, recv_scale, send_idx, send_w, err=None, stream=None):
    _expect("local_expert_fp8", recv_q=(recv_q, (torch.uint8, torch.float8_e4m3fn)), recv_scale=(recv_scale, torch.float32),
            send_idx=(send_idx, torch.int64), send_w=(send_w, torch.float32))
    N, H = recv_q.shape
    K = send_idx.shape[1]
    out = torch.empty((N, H), dtype=torch.bfloat16, device=recv_q.device)
    err = err if err is not None else error_word(recv_q.device)
    ep_local_expert_fp8(recv_q, recv_scale, send_idx, send_w, N, K, H, out, err, stream)
    return out


def dispatch_chunked_forward(x, topk_idx, topk_weights, *, num_local_experts: int, num_ranks: int, chunks: int,
                             fp8: bool = False, local_kernel=None, err=None, stream=None, keep=None):
    """The axolotl dispatch_chunked_forward on one GPU through the native driver.

    local_kernel: None for the library's synthetic fp8 expert (fp8 only), or a
    Python callable f(chunk, recv_x, recv_scale, send_idx, send_w, local_out)
    receiving torch views of the chunk's n rows, which must fill local_out
    (bf16 [n, H]) with the weighted sum over K of its experts on the current
    stream.  keep: an optional dict that receives the driver's buffers (the
    counts and token_pos of every chunk, and the row buffers, which hold the
    last chunk's rows once the call has run).  Returns out [T,H] bf16."""
    T, H = x.shape
    K = topk_idx.shape[1]
    P, El = num_ranks, num_local_experts
    dev = x.device
    bounds = chunk_bounds(T, chunks)
    max_len = max(bounds[i + 1] - bounds[i] for i in range(chunks))
    R = max(max_len * min(K, P), 1)
    t = dict(
        dest=torch.empty((T, K), dtype=torch.int32, device=dev),
        is_in_rank=torch.empty((T, P), dtype=torch.uint8, device=dev),
        send_counts=torch.empty((chunks, P), dtype=torch.int32, device=dev),
        rank_offsets=torch.empty((chunks, P + 1), dtype=torch.int32, device=dev),
        token_pos=torch.empty((T, P), dtype=torch.int32, device=dev),
        send_token_idx=torch.empty(R, dtype=torch.int32, device=dev),
        send_rank=torch.empty(R, dtype=torch.int32, device=dev),
        send_idx=torch.empty((R, K), dtype=torch.int64, device=dev),
        send_w=torch.empty((R, K), dtype=torch.float32, device=dev),
        recv_x=torch.empty((R, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
        recv_scale=torch.empty((R, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
        local_out=torch.empty((R, H), dtype=torch.bfloat16, device=dev),
        ws=workspace(T, K, P, El, chunks, dev),
        combine_ws=combine_ws(dev),
    )
    b = EPChunkBuffers()
    for f, _ in EPChunkBuffers._fields_:
        if f == "max_rows":
            b.max_rows = R
        elif f == "ws_bytes":
            b.ws_bytes = t["ws"].numel()
        else:
            v = t[f]
            setattr(b, f, None if v is None else v.data_ptr())
    h_counts = torch.empty(chunks * P, dtype=torch.int32, pin_memory=True)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    err = err if err is not None else error_word(dev)
    if local_kernel is None:
        if not fp8:
            raise ValueError("the built-in local kernel is the fp8 synthetic expert")
        cb = ep_local_expert_fp8_callback()
    else:
        def _py_kernel(user, chunk, n, K_, H_, rx, rs, si, sw, lo, err_p, stream_p):
            try:
                local_kernel(chunk, t["recv_x"][:n], None if t["recv_scale"] is None else t["recv_scale"][:n],
                             t["send_idx"][:n], t["send_w"][:n], t["local_out"][:n])
                return EP_OK
            except Exception:  # reported to the driver as a failed step
                return EP_ERR_INVALID_ARG
        cb = LOCAL_KERNEL_FN(_py_kernel)
    ep_dispatch_chunked_forward(x, topk_idx, topk_weights, T, K, H, P, El, chunks, int(fp8), cb, None, out, b,
                                h_counts, err, stream)
    if keep is not None:
        keep.update(t)
    return out


class ChunkedForward:
    """Buffers of ep_dispatch_chunked_forward_nosync, allocated once for
    T tokens and reused by every call (eager, or captured in a CUDA graph and
    replayed on new contents of the same input tensors).

    local_kernel: None for the library's synthetic fp8 expert (fp8 only), or a
    Python callable f(chunk, recv_x, recv_scale, send_idx, send_w, local_out,
    n_rows) receiving torch views of all max_rows rows of the chunk's row set
    and n_rows, a one-element device int32 tensor with the chunk's row count;
    it must fill local_out[:n_rows] (bf16) with the weighted sum over K of its
    experts, enqueued on the current stream, and may write rows past n_rows.
    n_sets: 2 pipelines chunk c+1's routing and dispatch (on an internal
    producer stream) with chunk c's local kernel and combine; 1 runs in order."""

    def __init__(self, T: int, K: int, H: int, *, num_ranks: int, num_local_experts: int, chunks: int,
                 fp8: bool = False, n_sets: int = 2, max_rows: Optional[int] = None, local_kernel=None,
                 device=None):
        dev = torch.device(device or "cuda")
        P, El = num_ranks, num_local_experts
        bounds = chunk_bounds(T, chunks)
        max_len = max(bounds[i + 1] - bounds[i] for i in range(chunks))
        R = max(max_len * min(K, P), 1) if max_rows is None else int(max_rows)
        self.T, self.K, self.H, self.P, self.El, self.chunks, self.fp8 = T, K, H, P, El, chunks, fp8
        self.max_rows, self.n_sets = R, n_sets
        self.t = dict(
            dest=torch.empty((T, K), dtype=torch.int32, device=dev),
            is_in_rank=torch.empty((T, P), dtype=torch.uint8, device=dev),
            send_counts=torch.empty((chunks, P), dtype=torch.int32, device=dev),
            rank_offsets=torch.empty((chunks, P + 1), dtype=torch.int32, device=dev),
            token_pos=torch.empty((T, P), dtype=torch.int32, device=dev),
            ws=workspace(T, K, P, El, chunks, dev),
            combine_ws=combine_ws(dev),
        )
        self.sets = []
        for _ in range(n_sets):
            self.sets.append(dict(
                send_token_idx=torch.empty(R, dtype=torch.int32, device=dev),
                send_rank=torch.empty(R, dtype=torch.int32, device=dev),
                send_idx=torch.empty((R, K), dtype=torch.int64, device=dev),
                send_w=torch.empty((R, K), dtype=torch.float32, device=dev),
                recv_x=torch.empty((R, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
                recv_scale=torch.empty((R, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
                local_out=torch.empty((R, H), dtype=torch.bfloat16, device=dev),
            ))
        b = EPPipelineBuffers()
        for f in ("dest", "is_in_rank", "send_counts", "rank_offsets", "token_pos", "ws", "combine_ws"):
            setattr(b, f, self.t[f].data_ptr())
        b.max_rows, b.n_sets, b.ws_bytes = R, n_sets, self.t["ws"].numel()
        for i, st in enumerate(self.sets):
            for f, _ in EPRowSet._fields_:
                setattr(b.sets[i], f, None if st[f] is None else st[f].data_ptr())
        self.buffers = b
        self.aux = torch.cuda.Stream(dev) if n_sets == 2 else None
        if local_kernel is None:
            if not fp8:
                raise ValueError("the built-in local kernel is the fp8 synthetic expert")
            self._cb = ep_local_expert_fp8_dev_callback()
        else:
            def _py_kernel(user, chunk, max_rows_, n_rows_p, K_, H_, rx, rs, si, sw, lo, err_p, stream_p):
                try:
                    st = self.sets[chunk % self.n_sets]
                    n_rows = self.t["rank_offsets"][chunk, self.P:self.P + 1]
                    local_kernel(chunk, st["recv_x"], st["recv_scale"], st["send_idx"], st["send_w"],
                                 st["local_out"], n_rows)
                    return EP_OK
                except Exception:  # reported to the driver as a failed step
                    return EP_ERR_INVALID_ARG
            self._cb = LOCAL_KERNEL_DEV_FN(_py_kernel)

    def __call__(self, x, topk_idx, topk_weights, out=None, err=None, stream=None):
        """Enqueue the chunked forward on `stream` (default: current); returns out [T,H] bf16."""
        if out is None:
            out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=x.device)
        err = err if err is not None else error_word(x.device)
        ep_dispatch_chunked_forward_nosync(x, topk_idx, topk_weights, self.T, self.K, self.H, self.P, self.El,
                                           self.chunks, int(self.fp8), self._cb, None, out, self.buffers, err,
                                           stream, self.aux)
        return out


def dispatch_chunked_forward_nosync(x, topk_idx, topk_weights, *, num_local_experts: int, num_ranks: int,
                                    chunks: int, fp8: bool = False, local_kernel=None, n_sets: int = 2, err=None,
                                    stream=None):
    """One call of the no-sync chunked forward (see ChunkedForward)."""
    T, H = x.shape
    f = ChunkedForward(T, topk_idx.shape[1], H, num_ranks=num_ranks, num_local_experts=num_local_experts,
                       chunks=chunks, fp8=fp8, n_sets=n_sets, local_kernel=local_kernel, device=x.device)
    out = f(x, topk_idx, topk_weights, err=err, stream=stream)
    torch.cuda.synchronize(x.device)   # the buffers of f die with this call
    return out
