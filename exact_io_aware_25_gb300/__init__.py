"""Exact, IO-aware tiled attention for GB300 (sm_103a) -- Python binding.

A thin ctypes layer over ``libfa.so`` (C ABI in ``include/fa.h``).  The
functions carry the C names and only marshal arguments: tensors may be given
as objects with ``data_ptr()`` (e.g. torch CUDA tensors) or as integer device
addresses; ``stream`` is a ``torch.cuda.Stream``, an integer ``cudaStream_t``
or None (legacy default stream).  Every computation runs in the library's
CUDA kernels; there is no fallback of any kind.  A non-OK status raises
:class:`FaError`.

Build the library with ``python -m exact_io_aware_25_gb300.build`` (done by
``__graft_entry__.build()``); importing this package does not compile
anything, and :func:`lib` raises if ``libfa.so`` is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "FaError", "lib", "fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_check",
    "fa_status_string", "fa_set_wait_timeout_ns", "fa_debug_starve_next_fwd",
    "fa_set_bwd_main_events", "fa_bwd_noalloc", "fa_bwd_noalloc_max_scratch_bytes",
    "fa_host_arena_size", "fa_fwd_host", "fa_fwd_bwd_host",
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED", "FA_ERR_CUDA",
    "FA_ERR_TIMEOUT", "FA_ERR_WORKSPACE", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_MISALIGNED = -3
FA_ERR_CUDA = -4
FA_ERR_TIMEOUT = -5
FA_ERR_WORKSPACE = -6

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded libfa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m exact_io_aware_25_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, vp, vp, vp]
            L.fa_fwd.restype = ci
            L.fa_bwd_workspace_size.argtypes = [ci, ci, ci, ci]
            L.fa_bwd_workspace_size.restype = sz
            L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, vp,
                                 vp, vp, sz, vp]
            L.fa_bwd.restype = ci
            u64 = ctypes.c_ulonglong
            L.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, vp, vp, cf,
                                         u64, vp]
            L.fa_fwd_dropout.restype = ci
            L.fa_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, cf,
                                         ci, vp, vp, cf, u64, vp, sz, vp]
            L.fa_bwd_dropout.restype = ci
            L.fa_fwd_splitkv_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci]
            L.fa_fwd_splitkv_workspace_size.restype = sz
            L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, ci, vp,
                                         sz, vp]
            L.fa_fwd_splitkv.restype = ci
            L.fa_fwd_stats.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, vp,
                                       vp, vp]
            L.fa_fwd_stats.restype = ci
            L.fa_fwd_csr.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, vp, vp, vp, ci,
                                     vp]
            L.fa_fwd_csr.restype = ci
            L.fa_bwd_csr_workspace_size.argtypes = [ci, ci, ci, ci]
            L.fa_bwd_csr_workspace_size.restype = sz
            L.fa_bwd_csr.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci,
                                     vp, vp, vp, ci, vp, sz, vp]
            L.fa_bwd_csr.restype = ci
            L.fa_fwd_qk.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, vp]
            L.fa_fwd_qk.restype = ci
            L.fa_bwd_qk.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf,
                                    ci, vp, vp, sz, vp]
            L.fa_bwd_qk.restype = ci
            L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, cf,
                                         ci, vp, vp, vp]
            L.fa_bwd_noalloc.restype = ci
            L.fa_bwd_noalloc_max_scratch_bytes.argtypes = []
            L.fa_bwd_noalloc_max_scratch_bytes.restype = sz
            L.fa_host_arena_size.argtypes = [ci, ci, ci, ci]
            L.fa_host_arena_size.restype = sz
            L.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, vp, vp, ci, vp,
                                      sz, vp]
            L.fa_fwd_host.restype = ci
            L.fa_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, cf,
                                          ci, vp, vp, ci, vp, sz, vp]
            L.fa_fwd_bwd_host.restype = ci
            L.fa_check.argtypes = [vp]
            L.fa_check.restype = ci
            L.fa_status_string.argtypes = [ci]
            L.fa_status_string.restype = ctypes.c_char_p
            L.fa_set_wait_timeout_ns.argtypes = [ctypes.c_longlong]
            L.fa_set_wait_timeout_ns.restype = None
            L.fa_set_bwd_main_events.argtypes = [vp, vp]
            L.fa_set_bwd_main_events.restype = None
            L.fa_debug_starve_next_fwd.argtypes = [ci]
            L.fa_debug_starve_next_fwd.restype = None
            _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return getattr(s, "cuda_stream", s) or None


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FaError(status, where)


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal=0, kv_len=None, block_mask=None,
           stream=None) -> None:
    """Enqueue the forward pass (see include/fa.h for shapes and rules)."""
    _check(lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                        int(d), float(scale), int(bool(causal)), _ptr(kv_len), _ptr(block_mask),
                        _stream(stream)), "fa_fwd")


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(lib().fa_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal=0, kv_len=None,
           block_mask=None, workspace=None, workspace_bytes=0, stream=None) -> None:
    """Enqueue the backward pass; ``workspace`` holds >= fa_bwd_workspace_size bytes."""
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                        _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), float(scale),
                        int(bool(causal)), _ptr(kv_len), _ptr(block_mask), _ptr(workspace),
                        int(workspace_bytes), _stream(stream)), "fa_bwd")


def fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, causal=0, kv_len=None, block_mask=None,
                   p=0.0, seed=0, stream=None) -> None:
    """fa_fwd with dropout of probability p on P (keep mask from ``seed``; see
    include/fa.h for its definition)."""
    _check(lib().fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                int(N), int(d), float(scale), int(bool(causal)), _ptr(kv_len),
                                _ptr(block_mask), float(p), int(seed) & (2**64 - 1),
                                _stream(stream)), "fa_fwd_dropout")


def fa_bwd_dropout(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal=0, kv_len=None,
                   block_mask=None, p=0.0, seed=0, workspace=None, workspace_bytes=0,
                   stream=None) -> None:
    """fa_bwd of the dropped-out forward (same p and seed as fa_fwd_dropout)."""
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d),
                                float(scale), int(bool(causal)), _ptr(kv_len), _ptr(block_mask),
                                float(p), int(seed) & (2**64 - 1), _ptr(workspace),
                                int(workspace_bytes), _stream(stream)), "fa_bwd_dropout")


def fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits=0) -> int:
    return int(lib().fa_fwd_splitkv_workspace_size(int(B), int(H), int(Nq), int(Nk), int(d),
                                                    int(num_splits)))


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, kv_len=None, num_splits=0,
                   workspace=None, workspace_bytes=0, stream=None) -> None:
    """Forward of Nq query rows against Nk key rows with the key range split
    across CTAs and merged (see include/fa.h)."""
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                int(Nq), int(Nk), int(d), float(scale), _ptr(kv_len),
                                int(num_splits), _ptr(workspace), int(workspace_bytes),
                                _stream(stream)), "fa_fwd_splitkv")


def fa_fwd_stats(q, k, v, o, lse, row_max, row_sum, B, H, N, d, scale, causal=0, kv_len=None,
                 block_mask=None, stream=None) -> None:
    """fa_fwd that also writes the row statistics m (row max of scale*QK^T)
    and l (sum of exp(s - m)) as fp32 [B, H, N]."""
    _check(lib().fa_fwd_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(row_max),
                              _ptr(row_sum), int(B), int(H), int(N), int(d), float(scale),
                              int(bool(causal)), _ptr(kv_len), _ptr(block_mask),
                              _stream(stream)), "fa_fwd_stats")


def fa_fwd_csr(q, k, v, o, lse, B, H, N, d, scale, causal=0, kv_len=None, row_ptr=None,
               col_idx=None, nnz=0, stream=None) -> None:
    """fa_fwd with the block mask as CSR over query tiles (device int32
    row_ptr [nb + 1] and col_idx [nnz])."""
    _check(lib().fa_fwd_csr(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                            int(N), int(d), float(scale), int(bool(causal)), _ptr(kv_len),
                            _ptr(row_ptr), _ptr(col_idx), int(nnz), _stream(stream)),
           "fa_fwd_csr")


def fa_bwd_csr_workspace_size(B, H, N, d) -> int:
    return int(lib().fa_bwd_csr_workspace_size(int(B), int(H), int(N), int(d)))


def fa_bwd_csr(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal=0, kv_len=None,
               row_ptr=None, col_idx=None, nnz=0, workspace=None, workspace_bytes=0,
               stream=None) -> None:
    """Backward of fa_fwd_csr (workspace of fa_bwd_csr_workspace_size bytes)."""
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_csr(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                            _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), float(scale),
                            int(bool(causal)), _ptr(kv_len), _ptr(row_ptr), _ptr(col_idx),
                            int(nnz), _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "fa_bwd_csr")


def fa_fwd_qk(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal=0, kv_len=None,
              stream=None) -> None:
    """Forward of Nq query rows against Nk key rows; causal is aligned to the
    bottom right (query i keeps key j iff j <= i + Nk - Nq)."""
    _check(lib().fa_fwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                           int(Nq), int(Nk), int(d), float(scale), int(bool(causal)),
                           _ptr(kv_len), _stream(stream)), "fa_fwd_qk")


def fa_bwd_qk(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, causal=0,
              kv_len=None, workspace=None, workspace_bytes=0, stream=None) -> None:
    """Backward of fa_fwd_qk (workspace: fa_bwd_workspace_size(B, H, Nq, d) bytes)."""
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                           _ptr(dk), _ptr(dv), int(B), int(H), int(Nq), int(Nk), int(d),
                           float(scale), int(bool(causal)), _ptr(kv_len), _ptr(workspace),
                           int(workspace_bytes), _stream(stream)), "fa_bwd_qk")


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal=0,
                   kv_len=None, block_mask=None, stream=None) -> None:
    """fa_bwd for callers that cannot allocate device memory: the scratch is a
    fixed array inside the library (see include/fa.h for its limit and the
    rule that overlapping calls race)."""
    _check(lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d),
                                float(scale), int(bool(causal)), _ptr(kv_len),
                                _ptr(block_mask), _stream(stream)), "fa_bwd_noalloc")


def fa_bwd_noalloc_max_scratch_bytes() -> int:
    return int(lib().fa_bwd_noalloc_max_scratch_bytes())


def fa_host_arena_size(B, H, N, d) -> int:
    return int(lib().fa_host_arena_size(int(B), int(H), int(N), int(d)))


def _nbytes(t, given):
    if t is not None and not isinstance(t, int) and not given:
        return t.numel() * t.element_size()
    return int(given)


def fa_fwd_host(q, k, v, o, lse, B, H, N, d, scale, causal=0, kv_len=None, block_mask=None,
                n_chunks=0, arena=None, arena_bytes=0, stream=None) -> None:
    """Forward of tensors in (pinned) HOST memory, with the copies overlapped
    with the kernels; ``arena`` is device scratch of >= fa_host_arena_size
    bytes.  The outputs are ready once ``stream`` has completed."""
    _check(lib().fa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                             int(N), int(d), float(scale), int(bool(causal)), _ptr(kv_len),
                             _ptr(block_mask), int(n_chunks), _ptr(arena),
                             _nbytes(arena, arena_bytes), _stream(stream)), "fa_fwd_host")


def fa_fwd_bwd_host(q, k, v, dout, o, lse, dq, dk, dv, B, H, N, d, scale, causal=0,
                    kv_len=None, block_mask=None, n_chunks=0, arena=None, arena_bytes=0,
                    stream=None) -> None:
    """Forward and backward of tensors in (pinned) HOST memory (see
    fa_fwd_host and include/fa.h)."""
    _check(lib().fa_fwd_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d),
                                 float(scale), int(bool(causal)), _ptr(kv_len), _ptr(block_mask),
                                 int(n_chunks), _ptr(arena), _nbytes(arena, arena_bytes),
                                 _stream(stream)), "fa_fwd_bwd_host")


def fa_check(stream=None) -> None:
    """Synchronise ``stream``; raise FaError if a kernel recorded an error."""
    _check(lib().fa_check(_stream(stream)), "fa_check")


def fa_set_wait_timeout_ns(ns: int) -> None:
    lib().fa_set_wait_timeout_ns(int(ns))


def fa_set_bwd_main_events(start_event=None, stop_event=None) -> None:
    """Record these events (torch.cuda.Event or raw cudaEvent_t) around the
    main backward kernel of later fa_bwd calls; None, None stops it."""
    def raw(e):
        if e is None:
            return None
        return e if isinstance(e, int) else e.cuda_event
    lib().fa_set_bwd_main_events(raw(start_event), raw(stop_event))


def fa_debug_starve_next_fwd(enable: bool = True) -> None:
    lib().fa_debug_starve_next_fwd(int(bool(enable)))
