"""Out-of-bounds writes, caught with guard bands (compute-sanitizer is not
available on this pool).

Every buffer a call writes -- O, lse, dQ, dK, dV, the row statistics, the
backward and split-KV workspaces -- is carved out of a larger allocation with
a band of at least 4 KiB on each side, filled with a known byte.  After the
call (and fa_check) every band byte must be unchanged, and every output
element must have been written (the buffers start as all-ones bytes, a NaN in
bf16 and fp32).  The sizes sit at tile edges (N = 1, 17, 129, 300, 4097),
with empty and one-key rows, a CSR mask, split-KV, N_q != N_k and the
allocation-free backward, where a store past the end of a buffer would not
show in a parity comparison."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BAND = 4096          # bytes on each side; a multiple of 256 keeps the payload aligned
FILL = 0xA5
UNSET = 0xFF         # payload start value: NaN in bf16 and in fp32


class Guarded:
    """A payload of `nbytes` between two guard bands of BAND bytes."""

    def __init__(self, nbytes, payload=UNSET):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * BAND,), FILL, dtype=torch.uint8, device="cuda")
        self.raw = self.buf[BAND:BAND + self.n]
        self.raw.fill_(payload)

    def as_tensor(self, dtype, shape):
        return self.raw.view(dtype).view(shape)

    def bands_intact(self):
        lo, hi = self.buf[:BAND], self.buf[BAND + self.n:]
        return bool(torch.all(lo == FILL)) and bool(torch.all(hi == FILL))


@pytest.fixture(scope="module")
def env(fa_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_25_gb300 as fa
    import gpu_harness as H
    import workloads as W
    return fa, H, W


def bf16_out(shape):
    g = Guarded(int(np.prod(shape)) * 2)
    return g, g.as_tensor(torch.bfloat16, shape)


def f32_out(shape):
    g = Guarded(int(np.prod(shape)) * 4)
    return g, g.as_tensor(torch.float32, shape)


def check(guards, outputs=()):
    torch.cuda.synchronize()
    for name, g in guards.items():
        assert g.bands_intact(), f"{name}: a guard band was overwritten"
    for name, t in outputs:
        assert not torch.any(torch.isnan(t.float())), f"{name}: element(s) left unwritten"


def fwd_bwd(fa, x, d, causal, kv_len=None, noalloc=False):
    B, Hh, N = x.B, x.H, x.N
    shape = (B, Hh, N, d)
    st = torch.cuda.current_stream()
    g = {}
    g["o"], o = bf16_out(shape)
    g["lse"], lse = f32_out((B, Hh, N))
    fa.fa_fwd(x.q, x.k, x.v, o, lse, B, Hh, N, d, x.scale, causal, kv_len, None, st)
    fa.fa_check(st)
    g["dq"], dq = bf16_out(shape)
    g["dk"], dk = bf16_out(shape)
    g["dv"], dv = bf16_out(shape)
    if noalloc:
        fa.fa_bwd_noalloc(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hh, N, d, x.scale, causal,
                          kv_len, None, st)
    else:
        need = fa.fa_bwd_workspace_size(B, Hh, N, d)
        g["ws"] = Guarded(need)
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hh, N, d, x.scale, causal, kv_len,
                  None, g["ws"].raw, need, st)
    fa.fa_check(st)
    check(g, [("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)])
    assert not torch.any(torch.isnan(lse))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 129, 300, 4097])
def test_guard_bands_plain(env, d, N):
    fa, H, W = env
    x = H.Inputs(W.make("tiny", seed=110 + N % 7, d=d, B=1, H=2, N=N))
    fwd_bwd(fa, x, d, causal=N % 2)


@pytest.mark.parametrize("d", [64, 128])
def test_guard_bands_empty_and_one_key(env, d):
    fa, H, W = env
    x = H.Inputs(W.make("tiny", seed=120, d=d, B=2, H=2, N=300))
    kv = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    fwd_bwd(fa, x, d, causal=0, kv_len=kv)


@pytest.mark.parametrize("d", [64, 128])
def test_guard_bands_noalloc(env, d):
    fa, H, W = env
    x = H.Inputs(W.make("tiny", seed=121, d=d, B=1, H=3, N=333))
    fwd_bwd(fa, x, d, causal=1, noalloc=True)


@pytest.mark.parametrize("d", [64, 128])
def test_guard_bands_csr_and_stats(env, d):
    fa, H, W = env
    N = 700
    nb = -(-N // 128)
    x = H.Inputs(W.make("tiny", seed=122, d=d, B=1, H=2, N=N))
    rng = np.random.default_rng(123)
    rows = [sorted(set(rng.integers(0, nb, size=3).tolist()) | {r}) for r in range(nb)]
    ptr = torch.tensor(np.cumsum([0] + [len(r) for r in rows]), dtype=torch.int32, device="cuda")
    idx = torch.tensor([c for r in rows for c in r], dtype=torch.int32, device="cuda")
    nnz = int(idx.numel())
    shape = (1, 2, N, d)
    st = torch.cuda.current_stream()
    g = {}
    g["o"], o = bf16_out(shape)
    g["lse"], lse = f32_out((1, 2, N))
    fa.fa_fwd_csr(x.q, x.k, x.v, o, lse, 1, 2, N, d, x.scale, 1, None, ptr, idx, nnz, st)
    fa.fa_check(st)
    g["dq"], dq = bf16_out(shape)
    g["dk"], dk = bf16_out(shape)
    g["dv"], dv = bf16_out(shape)
    need = fa.fa_bwd_csr_workspace_size(1, 2, N, d)
    g["ws"] = Guarded(need)
    fa.fa_bwd_csr(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, 1, 2, N, d, x.scale, 1, None, ptr,
                  idx, nnz, g["ws"].raw, need, st)
    fa.fa_check(st)
    check(g, [("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)])
    # the row statistics
    g2 = {}
    g2["o"], o2 = bf16_out(shape)
    g2["lse"], lse2 = f32_out((1, 2, N))
    g2["m"], m = f32_out((1, 2, N))
    g2["l"], l = f32_out((1, 2, N))
    fa.fa_fwd_stats(x.q, x.k, x.v, o2, lse2, m, l, 1, 2, N, d, x.scale, 1, None, None, st)
    fa.fa_check(st)
    check(g2, [("O", o2), ("m", m), ("l", l)])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (300, 129), (17, 4097)])
def test_guard_bands_splitkv(env, d, Nq, Nk):
    fa, H, W = env
    B, Hh = 2, 2
    rng = np.random.default_rng(124)
    mk = lambda n: H.dev_bf16(W.f32_to_bf16_bits(rng.standard_normal((B, Hh, n, d), dtype=np.float32)))
    q, k, v = mk(Nq), mk(Nk), mk(Nk)
    st = torch.cuda.current_stream()
    g = {}
    g["o"], o = bf16_out((B, Hh, Nq, d))
    g["lse"], lse = f32_out((B, Hh, Nq))
    need = fa.fa_fwd_splitkv_workspace_size(B, Hh, Nq, Nk, d, 0)
    g["ws"] = Guarded(need)
    fa.fa_fwd_splitkv(q, k, v, o, lse, B, Hh, Nq, Nk, d, 0.125, None, 0, g["ws"].raw, need, st)
    fa.fa_check(st)
    check(g, [("O", o), ("lse", lse)])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(5, 300), (300, 5), (129, 257)])
def test_guard_bands_qk(env, d, Nq, Nk):
    fa, H, W = env
    B, Hh = 1, 2
    rng = np.random.default_rng(125)
    mk = lambda n: H.dev_bf16(W.f32_to_bf16_bits(rng.standard_normal((B, Hh, n, d), dtype=np.float32)))
    q, k, v, do = mk(Nq), mk(Nk), mk(Nk), mk(Nq)
    st = torch.cuda.current_stream()
    g = {}
    g["o"], o = bf16_out((B, Hh, Nq, d))
    g["lse"], lse = f32_out((B, Hh, Nq))
    fa.fa_fwd_qk(q, k, v, o, lse, B, Hh, Nq, Nk, d, 0.125, 1, None, st)
    fa.fa_check(st)
    g["dq"], dq = bf16_out((B, Hh, Nq, d))
    g["dk"], dk = bf16_out((B, Hh, Nk, d))
    g["dv"], dv = bf16_out((B, Hh, Nk, d))
    need = fa.fa_bwd_workspace_size(B, Hh, Nq, d)
    g["ws"] = Guarded(need)
    fa.fa_bwd_qk(q, k, v, o, lse, do, dq, dk, dv, B, Hh, Nq, Nk, d, 0.125, 1, None, g["ws"].raw,
                 need, st)
    fa.fa_check(st)
    check(g, [("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)])


@pytest.mark.parametrize("d", [64, 128])
def test_guard_bands_dropout(env, d):
    fa, H, W = env
    x = H.Inputs(W.make("tiny", seed=126, d=d, B=1, H=2, N=257))
    B, Hh, N = x.B, x.H, x.N
    shape = (B, Hh, N, d)
    st = torch.cuda.current_stream()
    g = {}
    g["o"], o = bf16_out(shape)
    g["lse"], lse = f32_out((B, Hh, N))
    fa.fa_fwd_dropout(x.q, x.k, x.v, o, lse, B, Hh, N, d, x.scale, 1, None, None, 0.3, 77, st)
    fa.fa_check(st)
    g["dq"], dq = bf16_out(shape)
    g["dk"], dk = bf16_out(shape)
    g["dv"], dv = bf16_out(shape)
    need = fa.fa_bwd_workspace_size(B, Hh, N, d)
    g["ws"] = Guarded(need)
    fa.fa_bwd_dropout(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hh, N, d, x.scale, 1, None,
                      None, 0.3, 77, g["ws"].raw, need, st)
    fa.fa_check(st)
    check(g, [("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)])
