"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never does, and this package
imports nothing from it: the two meet only through the seeded inputs of
``workloads.py``.

The arithmetic lives in ``fa_oracle.c`` (plain C, double precision, plain
loops); this module only compiles it with gcc and marshals numpy arrays.

Function -> definition it follows (page titles as in ``fa_oracle.c``):

* ``forward``      the plain definition S = scale*Q K^T, P = softmax(S), O = P V,
                   lse = m + ln l  ("FlashAttention: Fast and Memory-Efficient
                   Exact Attention with IO-Awareness" explainer, "Problem and
                   motivation"; masks from "Key ideas" (fusion) and "Extension:
                   Block-Sparse FlashAttention").
* ``probs``        the same P, materialised for one head (tiny cases).
* ``forward_tiled`` the explainer's "Method" steps 1-4 with running (m, l);
                   used only to pin the streaming merge against ``forward``.
* ``backward``     the textbook gradient of O = softmax(scale Q K^T) V
                   (dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(dO o O)),
                   dQ = scale dS K, dK = scale dS^T Q).
* ``forward_qk`` / ``backward_qk``  the same with Nq query rows and Nk key
                   rows, causal aligned to the bottom right (key j is kept
                   for query i iff j <= i + Nk - Nq).

Pins (tests/test_oracle_pins.py): rows of P sum to 1, constant V gives that
constant, every block split of the tiled forward equals the one-shot
forward, Q = 0 gives the mean of the allowed values and lse = ln|A_i|, a
single allowed key returns that key's value, a key shift moves lse by
scale*<q, c>, joint K/V permutations leave O unchanged, central finite
differences of sum(dO o O) equal ``backward``, an all-ones block mask equals
no mask, and hand-derived closed-form values in tests/golden/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "libfa_oracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128  # block-mask granularity (rows and columns per mask entry)


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into libfa_oracle.so with gcc (-O2, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci, cd, cl = ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.fa_oracle_fwd.argtypes = [dp, dp, dp, ci, ci, ci, ci, cd, ci, i32p, u8p, ci,
                                          i64p, cl, dp, dp, ci]
            lib.fa_oracle_fwd.restype = ci
            lib.fa_oracle_probs.argtypes = [dp, dp, ci, ci, ci, ci, cd, ci, i32p, u8p, ci, ci, dp]
            lib.fa_oracle_probs.restype = ci
            lib.fa_oracle_fwd_tiled.argtypes = [dp, dp, dp, ci, ci, ci, ci, cd, ci, i32p, u8p,
                                                ci, ci, ci, dp, dp]
            lib.fa_oracle_fwd_tiled.restype = ci
            lib.fa_oracle_bwd.argtypes = [dp, dp, dp, dp, ci, ci, ci, ci, cd, ci, i32p, u8p, ci,
                                          i64p, cl, i64p, cl, dp, dp, dp, ci]
            lib.fa_oracle_bwd.restype = ci
            u64 = ctypes.c_uint64
            lib.fa_oracle_fwd_dropout.argtypes = [dp, dp, dp, ci, ci, ci, ci, cd, ci, i32p, u8p,
                                                  ci, ci, u64, i64p, cl, dp, dp, ci]
            lib.fa_oracle_fwd_dropout.restype = ci
            lib.fa_oracle_bwd_dropout.argtypes = [dp, dp, dp, dp, ci, ci, ci, ci, cd, ci, i32p,
                                                  u8p, ci, ci, u64, i64p, cl, i64p, cl, dp, dp,
                                                  dp, ci]
            lib.fa_oracle_bwd_dropout.restype = ci
            lib.fa_oracle_fwd_qk.argtypes = [dp, dp, dp, ci, ci, ci, ci, ci, cd, ci, i32p, i64p,
                                             cl, dp, dp, ci]
            lib.fa_oracle_bwd_qk.argtypes = [dp, dp, dp, dp, ci, ci, ci, ci, ci, cd, ci, i32p,
                                             i64p, cl, i64p, cl, dp, dp, dp, ci]
            lib.fa_oracle_bwd_qk.restype = ci
            lib.fa_oracle_fwd_stats.argtypes = [dp, dp, dp, ci, ci, ci, ci, cd, ci, i32p, u8p,
                                                ci, i64p, cl, dp, dp, dp, dp, ci]
            lib.fa_oracle_fwd_stats.restype = ci
            lib.fa_oracle_fwd_qk.restype = ci
            lib.fa_oracle_keep.argtypes = [u64, ci, ci, ci, ci]
            lib.fa_oracle_keep.restype = ci
            _lib = lib
    return _lib


def _f64(x):
    a = np.ascontiguousarray(x, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _opt_i32(x):
    if x is None:
        return None, None
    a = np.ascontiguousarray(x, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _opt_u8(x):
    if x is None:
        return None, None
    a = np.ascontiguousarray(x, dtype=np.uint8)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _opt_i64(x):
    if x is None:
        return None, None
    a = np.ascontiguousarray(x, dtype=np.int64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _shape(q):
    if q.ndim != 4:
        raise ValueError("expected [B, H, N, d]")
    return q.shape


def drop_p8(p):
    """Dropout threshold in 1/256 units for drop probability p in [0, 1):
    p * 256 rounded to nearest, ties to even, at most 255."""
    return min(int(np.rint(np.float32(p) * np.float32(256.0))), 255)


def keep(seed, p8, bh, i, j):
    """Dropout keep mask Z_ij (1 kept, 0 dropped) of head bh."""
    return int(_load().fa_oracle_keep(int(seed), int(p8), int(bh), int(i), int(j)))


def forward(q, k, v, scale, causal=False, kv_len=None, block_mask=None, rows=None,
            nthreads=None, block=BLOCK, p8=0, seed=0):
    """Exact forward.  q, k, v: float64 [B, H, N, d].

    rows: optional int64 array of global row ids (bh * N + i).  Returns
    (o, lse): o [B, H, N, d] and lse [B, H, N] for rows=None, else o [nrows, d]
    and lse [nrows].  p8 > 0 applies dropout with keep mask keep(seed, p8, ...)
    and keep scale 256 / (256 - p8) to P before the product with V.
    """
    lib = _load()
    B, H, N, d = _shape(q)
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    va, vp = _f64(v)
    kl, klp = _opt_i32(kv_len)
    bm, bmp = _opt_u8(block_mask)
    ra, rp = _opt_i64(rows)
    nrows = B * H * N if rows is None else len(ra)
    o = np.zeros((nrows, d), np.float64)
    lse = np.zeros((nrows,), np.float64)
    rc = lib.fa_oracle_fwd_dropout(qp, kp, vp, B, H, N, d, float(scale), int(bool(causal)), klp,
                                   bmp, int(block), int(p8), int(seed), rp, nrows, _f64(o)[1],
                                   _f64(lse)[1], _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"fa_oracle_fwd failed ({rc})")
    if rows is None:
        return o.reshape(B, H, N, d), lse.reshape(B, H, N)
    return o, lse


def forward_qk(q, k, v, scale, kv_len=None, rows=None, nthreads=None, causal=False):
    """Forward with Nq query rows and Nk key rows (q [B, H, Nq, d]; k, v
    [B, H, Nk, d]; no block mask; causal keeps key j for query i iff
    j <= i + Nk - Nq, bottom-right aligned).  Returns (o, lse) like forward,
    row ids bh * Nq + i."""
    lib = _load()
    B, H, Nq, d = _shape(q)
    Nk = _shape(k)[2]
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    va, vp = _f64(v)
    kl, klp = _opt_i32(kv_len)
    ra, rp = _opt_i64(rows)
    nrows = B * H * Nq if rows is None else len(ra)
    o = np.zeros((nrows, d), np.float64)
    lse = np.zeros((nrows,), np.float64)
    rc = lib.fa_oracle_fwd_qk(qp, kp, vp, B, H, Nq, Nk, d, float(scale), int(bool(causal)), klp,
                              rp, nrows, _f64(o)[1], _f64(lse)[1], _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"fa_oracle_fwd_qk failed ({rc})")
    if rows is None:
        return o.reshape(B, H, Nq, d), lse.reshape(B, H, Nq)
    return o, lse


def forward_stats(q, k, v, scale, causal=False, kv_len=None, block_mask=None, rows=None,
                  nthreads=None, block=BLOCK):
    """forward() plus the row statistics: returns (o, lse, m, l) with
    m_i = max_j s_ij and l_i = sum_j exp(s_ij - m_i) over the allowed keys
    (-inf and 0 for a row without any)."""
    lib = _load()
    B, H, N, d = _shape(q)
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    va, vp = _f64(v)
    kl, klp = _opt_i32(kv_len)
    bm, bmp = _opt_u8(block_mask)
    ra, rp = _opt_i64(rows)
    nrows = B * H * N if rows is None else len(ra)
    o = np.zeros((nrows, d), np.float64)
    lse, m, l = (np.zeros((nrows,), np.float64) for _ in range(3))
    rc = lib.fa_oracle_fwd_stats(qp, kp, vp, B, H, N, d, float(scale), int(bool(causal)), klp,
                                 bmp, int(block), rp, nrows, _f64(o)[1], _f64(lse)[1],
                                 _f64(m)[1], _f64(l)[1], _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"fa_oracle_fwd_stats failed ({rc})")
    if rows is None:
        return (o.reshape(B, H, N, d), lse.reshape(B, H, N), m.reshape(B, H, N),
                l.reshape(B, H, N))
    return o, lse, m, l


def probs(q, k, scale, bh=0, causal=False, kv_len=None, block_mask=None, block=BLOCK):
    """Dense P [N, N] of head bh (exactly 0 outside the allowed set)."""
    lib = _load()
    B, H, N, d = _shape(q)
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    kl, klp = _opt_i32(kv_len)
    bm, bmp = _opt_u8(block_mask)
    P = np.zeros((N, N), np.float64)
    rc = lib.fa_oracle_probs(qp, kp, B, H, N, d, float(scale), int(bool(causal)), klp, bmp,
                             int(block), int(bh), _f64(P)[1])
    if rc != 0:
        raise RuntimeError(f"fa_oracle_probs failed ({rc})")
    return P


def forward_tiled(q, k, v, scale, Br, Bc, causal=False, kv_len=None, block_mask=None,
                  block=BLOCK):
    """The pages' tiled forward (steps 1-4) with query blocks Br, key blocks Bc."""
    lib = _load()
    B, H, N, d = _shape(q)
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    va, vp = _f64(v)
    kl, klp = _opt_i32(kv_len)
    bm, bmp = _opt_u8(block_mask)
    o = np.zeros((B, H, N, d), np.float64)
    lse = np.zeros((B, H, N), np.float64)
    rc = lib.fa_oracle_fwd_tiled(qp, kp, vp, B, H, N, d, float(scale), int(bool(causal)), klp,
                                 bmp, int(block), int(Br), int(Bc), _f64(o)[1], _f64(lse)[1])
    if rc != 0:
        raise RuntimeError(f"fa_oracle_fwd_tiled failed ({rc})")
    return o, lse


def backward(q, k, v, dout, scale, causal=False, kv_len=None, block_mask=None, q_rows=None,
             k_rows=None, nthreads=None, block=BLOCK, p8=0, seed=0):
    """Textbook backward (of the dropped-out forward when p8 > 0).  Returns (dq, dk, dv).

    With q_rows/k_rows None the results are full [B, H, N, d] arrays;
    otherwise dq is [len(q_rows), d] and dk, dv are [len(k_rows), d].  Pass an
    empty array to skip one side.
    """
    lib = _load()
    B, H, N, d = _shape(q)
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    va, vp = _f64(v)
    da, dp = _f64(dout)
    kl, klp = _opt_i32(kv_len)
    bm, bmp = _opt_u8(block_mask)
    qr, qrp = _opt_i64(q_rows)
    kr, krp = _opt_i64(k_rows)
    nq = B * H * N if q_rows is None else len(qr)
    nk = B * H * N if k_rows is None else len(kr)
    dq = np.zeros((max(nq, 1), d), np.float64)
    dk = np.zeros((max(nk, 1), d), np.float64)
    dv = np.zeros((max(nk, 1), d), np.float64)
    rc = lib.fa_oracle_bwd_dropout(qp, kp, vp, dp, B, H, N, d, float(scale), int(bool(causal)),
                                   klp, bmp, int(block), int(p8), int(seed), qrp, nq, krp, nk,
                                   _f64(dq)[1], _f64(dk)[1], _f64(dv)[1], _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"fa_oracle_bwd failed ({rc})")
    dq, dk, dv = dq[:nq], dk[:nk], dv[:nk]
    if q_rows is None:
        dq = dq.reshape(B, H, N, d)
    if k_rows is None:
        dk, dv = dk.reshape(B, H, N, d), dv.reshape(B, H, N, d)
    return dq, dk, dv


def backward_qk(q, k, v, dout, scale, kv_len=None, q_rows=None, k_rows=None, nthreads=None,
                causal=False):
    """Backward of forward_qk: q, dout [B, H, Nq, d]; k, v [B, H, Nk, d];
    causal bottom-right aligned.  Returns (dq, dk, dv) shaped like q, k, v, or
    [len(q_rows), d] / [len(k_rows), d] for selected rows (bh * Nq + i,
    bh * Nk + j)."""
    lib = _load()
    B, H, Nq, d = _shape(q)
    Nk = _shape(k)[2]
    qa, qp = _f64(q)
    ka, kp = _f64(k)
    va, vp = _f64(v)
    da, dp = _f64(dout)
    kl, klp = _opt_i32(kv_len)
    qr, qrp = _opt_i64(q_rows)
    kr, krp = _opt_i64(k_rows)
    nq = B * H * Nq if q_rows is None else len(qr)
    nk = B * H * Nk if k_rows is None else len(kr)
    dq = np.zeros((max(nq, 1), d), np.float64)
    dk = np.zeros((max(nk, 1), d), np.float64)
    dv = np.zeros((max(nk, 1), d), np.float64)
    rc = lib.fa_oracle_bwd_qk(qp, kp, vp, dp, B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                              klp, qrp, nq, krp, nk, _f64(dq)[1], _f64(dk)[1], _f64(dv)[1],
                              _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"fa_oracle_bwd_qk failed ({rc})")
    dq, dk, dv = dq[:nq], dk[:nk], dv[:nk]
    if q_rows is None:
        dq = dq.reshape(B, H, Nq, d)
    if k_rows is None:
        dk, dv = dk.reshape(B, H, Nk, d), dv.reshape(B, H, Nk, d)
    return dq, dk, dv
