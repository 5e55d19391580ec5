"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/fa.h declares, and rejects bad arguments before touching CUDA
(these calls return from host-side validation; nothing is launched)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
FAKE = 0x10000  # a 16-byte aligned non-null address that is never dereferenced


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_check", "fa_status_string"} <= names


def test_library_exports_every_declared_symbol(fa_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa_lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(fa_\w+)", out))
    missing = set(declared_symbols()) - exported
    assert not missing, missing
    lib = fa_lib.lib()
    for name in declared_symbols():
        assert hasattr(lib, name)


def test_status_strings(fa_lib):
    for code in range(0, -7, -1):
        s = fa_lib.fa_status_string(code)
        assert s.startswith("FA_")
    assert fa_lib.fa_status_string(42) == "unknown fa_status"


def test_workspace_size_formula(fa_lib):
    # per (b, h) and padded row: D (4 B) + base-2 lse (4 B) + d fp32 dQ accumulators;
    # plus the block-sparse column lists: nl int32 counts, nl*nl int16 indices and
    # nl int16 key tiles by count (nl = min(nt, 1024), the most tiles a block mask
    # may have), and one int32 work counter
    up = lambda x: -(-x // 256) * 256
    for B, H, N in [(1, 1, 1), (2, 3, 129), (16, 16, 512), (1, 8, 65536), (1, 1, 1 << 20)]:
        for d in (64, 128):
            n_pad = -(-N // 128) * 128
            nl = min(n_pad // 128, 1024)
            bh = B * H
            want = up(bh * n_pad * 4)
            want = up(want + bh * n_pad * 4)
            want = up(want + bh * n_pad * d * 4)
            want = up(want + nl * 4)
            want = up(want + nl * nl * 2)
            want = up(want + nl * 2)
            want = up(want + 4)
            assert fa_lib.fa_bwd_workspace_size(B, H, N, d) == want
    assert fa_lib.fa_bwd_workspace_size(1, 1, 128, 96) == 0
    assert fa_lib.fa_bwd_workspace_size(0, 1, 128, 64) == 0
    assert fa_lib.fa_bwd_workspace_size(1, 1, 65536 * 128, 64) == 0  # too many tiles


def _fwd_status(fa, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125,
             causal=0, kv_len=None, block_mask=None, stream=None)
    a.update(kw)
    L = fa.lib()
    return L.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                    a["scale"], a["causal"], a["kv_len"], a["block_mask"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(lse=None), -1), (dict(B=0), -1), (dict(N=0), -1),
    (dict(H=-1), -1), (dict(scale=0.0), -1), (dict(scale=-1.0), -1),
    (dict(scale=float("inf")), -1), (dict(scale=float("nan")), -1),
    (dict(d=96), -2), (dict(d=32), -2), (dict(d=256), -2), (dict(N=1 << 20, block_mask=FAKE), -2),
    (dict(d=128, lse=FAKE + 4), -3),  # d = 128 passes the head-dim check (forward only)
    (dict(k=FAKE + 8), -3), (dict(lse=FAKE + 4), -3),
    (dict(B=1 << 16, H=1 << 16, N=1), -1), (dict(N=65535 * 128 + 1), -2),
])
def test_forward_validation_without_gpu(fa_lib, kw, status):
    assert _fwd_status(fa_lib, **kw) == status


def test_backward_validation_without_gpu(fa_lib):
    L = fa_lib.lib()
    need = fa_lib.fa_bwd_workspace_size(1, 1, 128, 64)

    def call(ws=FAKE, nbytes=need, d=64, dq=FAKE):
        return L.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, 1, 1, 128, d, 0.125,
                        0, None, None, ws, nbytes, None)

    assert call(dq=None) == -1
    assert call(d=96) == -2
    assert call(dq=FAKE + 2) == -3
    assert call(ws=None) == -6
    assert call(nbytes=need - 1) == -6
    assert call(ws=FAKE + 8) == -6


def test_product_path_never_touches_the_oracle():
    """The package and the header neither import, load nor name the oracle."""
    bad = []
    for base in ("exact_io_aware_25_gb300", "include"):
        for dirpath, _, files in os.walk(os.path.join(ROOT, base)):
            for f in files:
                if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                    text = open(os.path.join(dirpath, f)).read()
                    if re.search(r"\boracle\b|fa_oracle", text):
                        bad.append(os.path.join(dirpath, f))
    assert not bad, bad


def _fwd_drop_status(fa, p, N=128, seed=1, lse=FAKE):
    L = fa.lib()
    return L.fa_fwd_dropout(FAKE, FAKE, FAKE, FAKE, lse, 1, 1, N, 64, 0.125, 0, None, None,
                            p, seed, None)


@pytest.mark.parametrize("p,N,status", [
    (-0.1, 128, -1), (1.0, 128, -1), (1.5, 128, -1), (float("nan"), 128, -1),
    (float("inf"), 128, -1), (0.1, 131072 + 1, -2), (0.0, 131072 + 1, -3),
])
def test_dropout_validation_without_gpu(fa_lib, p, N, status):
    """Bad drop probabilities are rejected before anything else happens; a
    positive one needs N <= 131072; p = 0 is plain attention at any N (here it
    gets as far as the alignment check, which a misaligned lse fails: no call
    of this test reaches a device)."""
    got = _fwd_drop_status(fa_lib, p, N, lse=FAKE + 4)
    assert got == status
    L = fa_lib.lib()
    need = fa_lib.fa_bwd_workspace_size(1, 1, 128, 64)
    if status in (-1,):
        assert L.fa_bwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64,
                                0.125, 0, None, None, p, 1, FAKE, need, None) == -1


def test_splitkv_workspace_and_validation_without_gpu(fa_lib):
    """Workspace: S * B * H * Nq_pad rows of 64 fp32 partial outputs plus one
    fp32 lse each (each part 256-byte aligned), S chosen as documented."""
    up = lambda x: -(-x // 256) * 256
    for B, H, Nq, Nk, S in [(1, 1, 1, 1000, 3), (2, 8, 16, 32768, 0), (4, 2, 300, 129, 5)]:
        nq_pad = -(-Nq // 128) * 128
        nk_t = -(-Nk // 128)
        if S == 0:
            units = B * H * (nq_pad // 128)
            S_eff = min(-(-304 // units), 256)
        else:
            S_eff = S
        S_eff = max(1, min(S_eff, nk_t))
        rows = S_eff * B * H * nq_pad
        for d in (64, 128):
            want = up(up(rows * d * 4) + rows * 4)
            got = fa_lib.fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, S)
            assert got == want, (B, H, Nq, Nk, S, d)
    assert fa_lib.fa_fwd_splitkv_workspace_size(1, 1, 1, 128, 96, 0) == 0
    assert fa_lib.fa_fwd_splitkv_workspace_size(1, 1, 1, 128, 64, 2000) == 0
    L = fa_lib.lib()
    need = fa_lib.fa_fwd_splitkv_workspace_size(1, 1, 1, 256, 64, 0)

    def call(**kw):
        a = dict(q=FAKE, o=FAKE, Nq=1, Nk=256, d=64, scale=0.125, S=0, ws=FAKE, nbytes=need)
        a.update(kw)
        return L.fa_fwd_splitkv(a["q"], FAKE, FAKE, a["o"], FAKE, 1, 1, a["Nq"], a["Nk"], a["d"],
                                a["scale"], None, a["S"], a["ws"], a["nbytes"], None)

    assert call(q=None) == -1
    assert call(Nq=0) == -1 and call(Nk=0) == -1
    assert call(scale=-1.0) == -1
    assert call(S=-1) == -1 and call(S=1025) == -1
    assert call(d=96) == -2
    assert call(d=128, nbytes=need) == -6   # the d = 128 partials need twice the bytes
    assert call(d=128, o=FAKE + 8) == -3
    assert call(o=FAKE + 8) == -3
    assert call(ws=None) == -6 and call(nbytes=need - 1) == -6


def test_api_variant_validation_without_gpu(fa_lib):
    """fa_fwd_stats, fa_fwd_csr, fa_fwd_qk and fa_bwd_csr reject bad arguments
    on the host; every call here stops before the device (a misaligned
    pointer is the last check passed arguments meet)."""
    L = fa_lib.lib()

    def stats(rm=FAKE, rs=FAKE, lse=FAKE, d=64):
        return L.fa_fwd_stats(FAKE, FAKE, FAKE, FAKE, lse, rm, rs, 1, 1, 128, d, 0.125, 0, None,
                              None, None)

    assert stats(rm=None) == -1 and stats(rs=None) == -1
    assert stats(rm=FAKE + 4) == -3 and stats(lse=FAKE + 4) == -3
    assert stats(d=96) == -2
    assert stats(d=128, rs=FAKE + 8) == -3

    def csr(rp=FAKE, ci=FAKE, nnz=4, N=1000, lse=FAKE + 4, d=64):
        return L.fa_fwd_csr(FAKE, FAKE, FAKE, FAKE, lse, 1, 1, N, d, 0.125, 0, None, rp, ci, nnz,
                            None)

    assert csr(rp=None) == -1 and csr(nnz=-1) == -1 and csr(ci=None) == -1
    assert csr(ci=None, nnz=0) == -3             # no entries: col_idx may be NULL
    assert csr(N=1024 * 128 + 1) == -2           # more than 1024 tiles per row
    assert csr() == -3 and csr(d=128) == -3

    def qk(Nq=5, Nk=300, d=64, lse=FAKE + 4):
        return L.fa_fwd_qk(FAKE, FAKE, FAKE, FAKE, lse, 2, 3, Nq, Nk, d, 0.125, 1, None, None)

    assert qk(Nk=0) == -1 and qk(Nq=0) == -1 and qk(d=32) == -2
    assert qk() == -3 and qk(d=128) == -3 and qk(Nq=300, Nk=5) == -3

    def bqk(Nq=5, Nk=300, d=64, dk=FAKE, ws=FAKE, nbytes=None):
        if nbytes is None:
            nbytes = fa_lib.fa_bwd_workspace_size(2, 3, max(Nq, 1), 64)
        return L.fa_bwd_qk(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dk, FAKE, 2, 3, Nq, Nk, d,
                           0.125, 1, None, ws, nbytes, None)

    assert bqk(Nk=0) == -1 and bqk(Nq=0) == -1 and bqk(d=32) == -2
    assert bqk(dk=FAKE + 2) == -3 and bqk(d=128, dk=FAKE + 8) == -3
    assert bqk(ws=None) == -6 and bqk(nbytes=1) == -6
    assert bqk(Nq=300, Nk=5, ws=None) == -6

    up = lambda x: -(-x // 256) * 256
    for N in (1, 128, 1000, 65536):
        nt = -(-N // 128)
        want = fa_lib.fa_bwd_workspace_size(2, 3, N, 64) + up(nt * nt)
        assert fa_lib.fa_bwd_csr_workspace_size(2, 3, N, 64) == want
    assert fa_lib.fa_bwd_csr_workspace_size(1, 1, 1024 * 128 + 1, 64) == 0
    assert fa_lib.fa_bwd_csr_workspace_size(1, 1, 128, 96) == 0
    need = fa_lib.fa_bwd_csr_workspace_size(1, 1, 1000, 64)

    def bcsr(rp=FAKE, ws=FAKE, nbytes=need, dq=FAKE):
        return L.fa_bwd_csr(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, 1, 1, 1000, 64,
                            0.125, 0, None, rp, FAKE, 3, ws, nbytes, None)

    assert bcsr(rp=None) == -1
    assert bcsr(nbytes=need - 1) == -6 and bcsr(ws=None) == -6
    assert bcsr(dq=FAKE + 2) == -3


@pytest.mark.parametrize("kw", [
    dict(dq=None), dict(B=0), dict(scale=-1.0), dict(d=96), dict(dq=FAKE + 2),
    dict(N=65535 * 128 + 1),                     # too many query tiles: unsupported
    dict(N=1024 * 128 + 1, block_mask=FAKE),     # block mask wider than 1024 tiles: unsupported
    dict(B=1 << 16, H=1 << 16, N=1),
    dict(H=8, N=65536),                          # valid, but beyond the fixed scratch
])
def test_noalloc_status_equals_fa_bwd_status_without_gpu(fa_lib, kw):
    """fa_bwd_noalloc gives every argument set fa_bwd rejects the code fa_bwd
    gives it; arguments fa_bwd accepts but whose workspace exceeds the fixed
    scratch get FA_ERR_WORKSPACE.  No call here reaches a device."""
    L = fa_lib.lib()
    a = dict(dq=FAKE, B=1, H=1, N=128, d=64, scale=0.125, block_mask=None)
    a.update(kw)
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["dq"], FAKE, FAKE, a["B"], a["H"], a["N"], a["d"],
            a["scale"], 0, None, a["block_mask"])
    want = L.fa_bwd(*args, None, 0, None)
    got = L.fa_bwd_noalloc(*args, None)
    assert got == want
    if kw.get("N") == 65536:
        assert want == -6 and got == -6


def test_host_arena_size_formula(fa_lib):
    # device copies of q, k, v, dout, o, dq, dk, dv; the lse region with one
    # 256-byte boundary of slack per head group (at most 64); kv_len; the
    # block mask (when it may exist); the backward workspace of the whole problem
    L = fa_lib.lib()
    up = lambda x: -(-x // 256) * 256
    for B, H, N, d in [(1, 1, 1, 64), (2, 3, 301, 128), (1, 8, 65536, 64), (1, 1, 1 << 18, 64)]:
        nb = -(-N // 128)
        want = 8 * up(B * H * N * d * 2) + up(B * H * N * 4) + 256 * 64 + up(B * 4)
        want += up(nb * nb) if nb <= 1024 else 0
        want += fa_lib.fa_bwd_workspace_size(B, H, N, d)
        assert L.fa_host_arena_size(B, H, N, d) == want
    assert L.fa_host_arena_size(1, 1, 128, 96) == 0
    assert L.fa_host_arena_size(0, 1, 128, 64) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(dout=None), -1), (dict(n_chunks=-1), -1), (dict(n_chunks=65), -1),
    (dict(B=0), -1), (dict(scale=float("nan")), -1), (dict(d=96), -2),
    (dict(N=1024 * 128 + 1, mask=FAKE), -2), (dict(N=65535 * 128 + 1), -2),
    (dict(arena=None), -6), (dict(arena=FAKE + 16), -6), (dict(short=1), -6),
])
def test_host_api_validation_without_gpu(fa_lib, kw, status):
    """Both host-buffer entry points reject bad arguments before any CUDA
    call, with fa_fwd's code for the arguments they share."""
    L = fa_lib.lib()
    a = dict(q=FAKE, dout=FAKE, B=1, H=1, N=128, d=64, scale=0.125, mask=None, n_chunks=0,
             arena=FAKE, short=0)
    a.update(kw)
    need = L.fa_host_arena_size(a["B"], a["H"], a["N"], a["d"])
    nbytes = max(need - a["short"], 0) if need else 1 << 40
    got = L.fa_fwd_bwd_host(a["q"], FAKE, FAKE, a["dout"], FAKE, FAKE, FAKE, FAKE, FAKE, a["B"],
                            a["H"], a["N"], a["d"], a["scale"], 0, None, a["mask"],
                            a["n_chunks"], a["arena"], nbytes, None)
    assert got == status
    if "dout" not in kw:
        got_f = L.fa_fwd_host(a["q"], FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["N"], a["d"],
                              a["scale"], 0, None, a["mask"], a["n_chunks"], a["arena"], nbytes,
                              None)
        assert got_f == status
    if status in (-1, -2) and not {"n_chunks", "dout"} & set(kw):
        want = L.fa_fwd(a["q"], FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["N"], a["d"],
                        a["scale"], 0, None, a["mask"], None)
        assert got == want
