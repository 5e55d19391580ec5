"""GPU parity of the host-buffer entry points (fa_fwd_host, fa_fwd_bwd_host):
pinned host tensors in, host tensors out, with the copies of consecutive head
groups overlapped with the kernels.

* Against the fp64 oracle at the parity tolerances.
* Against the device entry points on the same inputs: O, lse, dK and dV
  bitwise (each element is produced by one CTA whose order of work does not
  depend on how the heads are grouped), dQ within the gradient tolerance of
  the device result (its fp32 partial sums are reduced in hardware order).
* Guard bands of 4 KiB around every host output and around the device arena:
  nothing is written outside the buffers, every output element is written.
* Group plans: automatic, one group, whole batches, heads within a batch, more
  groups than heads, and lse segments that do not start on a 16-byte boundary
  inside the [B, H, N] array (N odd).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BAND = 4096
FILL = 0xA5


class HostGuarded:
    """A pinned host payload of `nbytes` between two bands of BAND bytes."""

    def __init__(self, nbytes, payload=0xFF):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * BAND,), FILL, dtype=torch.uint8).pin_memory()
        self.raw = self.buf[BAND:BAND + self.n]
        self.raw.fill_(payload)

    def view(self, dtype, shape):
        return self.raw.view(dtype).view(shape)

    def bands_intact(self):
        return bool(torch.all(self.buf[:BAND] == FILL)) and bool(
            torch.all(self.buf[BAND + self.n:] == FILL))


@pytest.fixture(scope="module")
def H(fa_lib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gpu_harness
    return gpu_harness


def pinned_bits(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()


def run_host(x, n_chunks, with_bwd=True):
    """One host-API call on the workload's inputs; returns the host outputs
    (O, lse, dQ, dK, dV as numpy) after checking every guard band."""
    import exact_io_aware_25_gb300 as fa
    B, Hh, N, d = x.B, x.H, x.N, x.d
    w = x.w
    hq, hk, hv, hdo = (pinned_bits(getattr(w, n)) for n in ("q", "k", "v", "do"))
    kv = (None if x.kv_len_np is None
          else torch.from_numpy(np.asarray(x.kv_len_np, np.int32)).pin_memory())
    mask = (None if x.mask_np is None
            else torch.from_numpy(np.ascontiguousarray(x.mask_np, np.uint8)).pin_memory())
    t_bytes = B * Hh * N * d * 2
    g = {n: HostGuarded(t_bytes) for n in ("o", "dq", "dk", "dv")}
    g["lse"] = HostGuarded(B * Hh * N * 4)
    need = fa.fa_host_arena_size(B, Hh, N, d)
    assert need > 0
    arena = torch.full((need + 2 * BAND,), FILL, dtype=torch.uint8, device="cuda")
    payload = arena[BAND:BAND + need]
    st = torch.cuda.current_stream()
    o = g["o"].view(torch.int16, (B, Hh, N, d))
    lse = g["lse"].view(torch.float32, (B, Hh, N))
    if with_bwd:
        fa.fa_fwd_bwd_host(hq, hk, hv, hdo, o, lse, g["dq"].raw, g["dk"].raw, g["dv"].raw, B, Hh,
                           N, d, x.scale, x.causal, kv, mask, n_chunks, payload, need, st)
    else:
        fa.fa_fwd_host(hq, hk, hv, o, lse, B, Hh, N, d, x.scale, x.causal, kv, mask, n_chunks,
                       payload, need, st)
    fa.fa_check(st)
    torch.cuda.synchronize()
    assert bool(torch.all(arena[:BAND] == FILL)) and bool(torch.all(arena[BAND + need:] == FILL)), \
        "arena guard band overwritten"
    names = ("o", "lse", "dq", "dk", "dv") if with_bwd else ("o", "lse")
    for n in names:
        assert g[n].bands_intact(), f"{n}: a host guard band was overwritten"
    out = {"lse": lse.numpy().copy()}
    for n in ("o", "dq", "dk", "dv") if with_bwd else ("o",):
        out[n] = g[n].raw.view(torch.int16).numpy().view(np.uint16).reshape(B, Hh, N, d).copy()
    return out


def bits_of(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


CASES = [
    # (B, H, N, d, variant, n_chunks)
    (2, 3, 301, 64, "plain", 0),      # automatic plan
    (2, 3, 301, 64, "causal", 4),     # heads within each batch, odd N
    (3, 2, 257, 128, "kv_len", 5),    # 6 groups of one head
    (1, 4, 520, 64, "mask", 3),       # one batch cut into 3 head groups
    (1, 2, 129, 128, "causal", 64),   # more groups than heads: one per head
    (3, 2, 129, 64, "plain", 1),      # a single group
]


def make_inputs(H, B, Hh, N, d, variant, seed):
    import workloads as W
    w = W.make("tiny", seed=seed, d=d, B=B, H=Hh, N=N)
    kw = {}
    if variant == "causal":
        kw["causal"] = True
    elif variant == "kv_len":
        kw["kv_len"] = np.array([0, 1, N - 77][:B], np.int32)
    elif variant == "mask":
        nb = -(-N // 128)
        m = (np.random.default_rng(seed + 1).random((nb, nb)) < 0.5).astype(np.uint8)
        m[1, :] = 0
        kw["block_mask"] = m
    return H.Inputs(w, **kw)


@pytest.mark.parametrize("B,Hh,N,d,variant,n_chunks", CASES)
def test_fwd_bwd_host_matches_oracle_and_device(H, oracle_mod, B, Hh, N, d, variant, n_chunks):
    x = make_inputs(H, B, Hh, N, d, variant, seed=300 + B * 7 + N)
    got = run_host(x, n_chunks)
    # the device entry points on the same inputs
    o_dev, lse_dev = H.run_fwd(x)
    dq_dev, dk_dev, dv_dev = H.run_bwd(x, o_dev, lse_dev)
    assert np.array_equal(got["o"], bits_of(o_dev)), "O differs from fa_fwd"
    assert np.array_equal(got["lse"].view(np.uint32), lse_dev.cpu().numpy().view(np.uint32)), \
        "lse differs from fa_fwd"
    assert np.array_equal(got["dk"], bits_of(dk_dev)), "dK differs from fa_bwd"
    assert np.array_equal(got["dv"], bits_of(dv_dev)), "dV differs from fa_bwd"
    import workloads as W
    f = W.bf16_bits_to_f64
    H.assert_grad(f(got["dq"]), H.host_f64(dq_dev), "dQ vs fa_bwd")
    # the oracle
    o_r, lse_r = oracle_mod.forward(x.f64("q"), x.f64("k"), x.f64("v"), x.scale,
                                    **x.oracle_kwargs())
    H.assert_o(f(got["o"]), o_r)
    H.assert_lse(got["lse"].astype(np.float64), lse_r)
    dq_r, dk_r, dv_r = oracle_mod.backward(x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do"),
                                           x.scale, **x.oracle_kwargs())
    H.assert_grad(f(got["dq"]), dq_r, "dQ")
    H.assert_grad(f(got["dk"]), dk_r, "dK")
    H.assert_grad(f(got["dv"]), dv_r, "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_chunks", [0, 3])
def test_fwd_host_matches_device(H, d, n_chunks):
    x = make_inputs(H, 2, 3, 301, d, "causal", seed=320 + d)
    got = run_host(x, n_chunks, with_bwd=False)
    o_dev, lse_dev = H.run_fwd(x)
    assert np.array_equal(got["o"], bits_of(o_dev))
    assert np.array_equal(got["lse"].view(np.uint32), lse_dev.cpu().numpy().view(np.uint32))


def test_host_calls_back_to_back_on_two_streams(H):
    """Two host-API calls enqueued back to back on different streams (sharing
    the library's copy streams) each return their own inputs' results."""
    import exact_io_aware_25_gb300 as fa
    xs = [make_inputs(H, 1, 2, 700, 64, v, seed=330 + i) for i, v in enumerate(("plain", "causal"))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    keep = []
    for x, st in zip(xs, streams):
        B, Hh, N, d = x.B, x.H, x.N, x.d
        hq, hk, hv = (pinned_bits(getattr(x.w, n)) for n in ("q", "k", "v"))
        o = torch.full((B, Hh, N, d), -1, dtype=torch.int16).pin_memory()
        lse = torch.full((B, Hh, N), float("nan"), dtype=torch.float32).pin_memory()
        need = fa.fa_host_arena_size(B, Hh, N, d)
        arena = torch.empty((need,), dtype=torch.uint8, device="cuda")
        fa.fa_fwd_host(hq, hk, hv, o, lse, B, Hh, N, d, x.scale, x.causal, None, None, 2, arena,
                       need, st)
        outs.append((o, lse))
        keep.append((hq, hk, hv, arena))
    for st in streams:
        fa.fa_check(st)
    for x, (o, lse) in zip(xs, outs):
        o_dev, lse_dev = H.run_fwd(x)
        assert np.array_equal(o.numpy().view(np.uint16), bits_of(o_dev))
        assert np.array_equal(lse.numpy().view(np.uint32), lse_dev.cpu().numpy().view(np.uint32))
