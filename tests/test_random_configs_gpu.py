"""Seeded random configurations against the fp64 oracle (GPU).

The fixed parity cases cover each feature on its own; these draw them
together: 1-3 batches and heads, ragged lengths N in [1, 700), both head
dimensions, causal, per-batch key lengths drawn from [0, N], random block
masks (empty rows and columns included), dropout, scales from 0.05 to 0.3, and
N_q != N_k (bottom-right causal).  Each case runs the forward and backward
through the C ABI into NaN-prefilled outputs and compares every output with
the oracle at the parity tolerances (with dropout, O's absolute bound times
1/(1-p'), the factor every kept term is scaled by); some also run the
host-buffer call and check that it returns the device calls' O, lse, dK and
dV bit for bit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def H(fa_lib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gpu_harness
    return gpu_harness


def draw(case):
    rng = np.random.default_rng(case)
    c = dict(d=int(rng.choice([64, 128])), B=int(rng.integers(1, 4)), H=int(rng.integers(1, 4)),
             N=int(rng.integers(1, 700)), causal=bool(rng.integers(0, 2)),
             scale=float(rng.uniform(0.05, 0.3)))
    c["Nk"] = c["N"]
    c["kv"] = rng.integers(0, c["N"] + 1, size=c["B"]).astype(np.int32) if rng.random() < 0.4 else None
    nb = -(-c["N"] // 128)
    c["mask"] = ((rng.random((nb, nb)) < rng.uniform(0.2, 0.9)).astype(np.uint8)
                 if rng.random() < 0.4 else None)
    c["p"] = float(rng.choice([0.0, 0.0, 0.15, 0.5]))
    c["seed"] = int(rng.integers(0, 2**40))
    c["host"] = c["p"] == 0.0 and rng.random() < 0.5
    if c["mask"] is None and c["p"] == 0.0 and rng.random() < 0.35:
        c["Nk"] = int(rng.integers(1, 700))     # N_q != N_k, bottom-right causal
        c["host"] = False
    return c


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_qk(H, c, q, k, v, do):
    import exact_io_aware_25_gb300 as fa
    B, Hh, Nq, Nk, d = c["B"], c["H"], c["N"], c["Nk"], c["d"]
    dev = H.dev_bf16
    tq, tk, tv, tdo = dev(q), dev(k), dev(v), dev(do)
    kl = None if c["kv"] is None else torch.from_numpy(c["kv"]).cuda()
    o = H.nan_like_bf16((B, Hh, Nq, d))
    lse = torch.full((B, Hh, Nq), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_qk(tq, tk, tv, o, lse, B, Hh, Nq, Nk, d, c["scale"], c["causal"], kl, st)
    dq = H.nan_like_bf16((B, Hh, Nq, d))
    dk, dv = H.nan_like_bf16((B, Hh, Nk, d)), H.nan_like_bf16((B, Hh, Nk, d))
    nbytes = fa.fa_bwd_workspace_size(B, Hh, Nq, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    fa.fa_bwd_qk(tq, tk, tv, o, lse, tdo, dq, dk, dv, B, Hh, Nq, Nk, d, c["scale"], c["causal"],
                 kl, ws, nbytes, st)
    fa.fa_check(st)
    return o, lse, dq, dk, dv


def run_host(c, x):
    import exact_io_aware_25_gb300 as fa
    B, Hh, N, d = x.B, x.H, x.N, x.d
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
    hq, hk, hv, hdo = (pin(getattr(x.w, n)) for n in ("q", "k", "v", "do"))
    out = [torch.full((B, Hh, N, d), -1, dtype=torch.int16).pin_memory() for _ in range(4)]
    hl = torch.full((B, Hh, N), float("nan"), dtype=torch.float32).pin_memory()
    kv = None if c["kv"] is None else torch.from_numpy(c["kv"]).pin_memory()
    mk = None if c["mask"] is None else torch.from_numpy(c["mask"]).pin_memory()
    need = fa.fa_host_arena_size(B, Hh, N, d)
    arena = torch.empty((need,), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_bwd_host(hq, hk, hv, hdo, out[0], hl, out[1], out[2], out[3], B, Hh, N, d,
                       c["scale"], c["causal"], kv, mk, 0, arena, need, st)
    fa.fa_check(st)
    return [t.numpy().view(np.uint16) for t in out], hl.numpy()


@pytest.mark.parametrize("case", list(range(900, 932)))
def test_random_config(H, oracle_mod, case):
    import workloads as W
    c = draw(case)
    f = W.bf16_bits_to_f64
    if c["Nk"] != c["N"]:
        rng = np.random.default_rng(case + 1)
        mk = lambda n: W.f32_to_bf16_bits(
            rng.standard_normal((c["B"], c["H"], n, c["d"]), dtype=np.float32))
        q, k, v, do = mk(c["N"]), mk(c["Nk"]), mk(c["Nk"]), mk(c["N"])
        o, lse, dq, dk, dv = run_qk(H, c, q, k, v, do)
        o_r, lse_r = oracle_mod.forward_qk(f(q), f(k), f(v), c["scale"], kv_len=c["kv"],
                                           causal=c["causal"])
        dq_r, dk_r, dv_r = oracle_mod.backward_qk(f(q), f(k), f(v), f(do), c["scale"],
                                                  kv_len=c["kv"], causal=c["causal"])
    else:
        w = W.make("tiny", seed=case, d=c["d"], B=c["B"], H=c["H"], N=c["N"])
        x = H.Inputs(w, causal=c["causal"], scale=c["scale"], kv_len=c["kv"], block_mask=c["mask"])
        kw = x.oracle_kwargs()
        if c["p"] > 0:
            o, lse = H.run_fwd_dropout(x, c["p"], c["seed"])
            dq, dk, dv = H.run_bwd_dropout(x, o, lse, c["p"], c["seed"])
            kw = dict(kw, p8=oracle_mod.drop_p8(c["p"]), seed=c["seed"])
        else:
            o, lse = H.run_fwd(x)
            dq, dk, dv = H.run_bwd(x, o, lse)
        q4 = [x.f64(n) for n in ("q", "k", "v", "do")]
        o_r, lse_r = oracle_mod.forward(q4[0], q4[1], q4[2], x.scale, **kw)
        dq_r, dk_r, dv_r = oracle_mod.backward(*q4, x.scale, **kw)
        if c["host"]:
            (ho, hdq, hdk, hdv), hl = run_host(c, x)
            assert np.array_equal(ho, bits(o)) and np.array_equal(hdk, bits(dk))
            assert np.array_equal(hdv, bits(dv))
            assert np.array_equal(hl.view(np.uint32), lse.cpu().numpy().view(np.uint32))
            H.assert_grad(f(hdq), dq_r, "dQ (host-buffer call)")
    # dropout scales O by 1/(1-p'), and with it the absolute bound (a reading
    # of the tolerance, which is stated for attention without dropout)
    keep_scale = 256.0 / (256 - oracle_mod.drop_p8(c["p"])) if c["p"] > 0 else 1.0
    H.assert_o(H.host_f64(o), o_r, maxabs_scale=keep_scale)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_r)
    H.assert_grad(H.host_f64(dq), dq_r, "dQ")
    H.assert_grad(H.host_f64(dk), dk_r, "dK")
    H.assert_grad(H.host_f64(dv), dv_r, "dV")


def test_random_configs_cover_every_feature():
    """The seeded draws include each feature at least once (checked on the
    host, so that a change of seeds cannot silently drop one)."""
    cs = [draw(case) for case in range(900, 932)]
    assert {c["d"] for c in cs} == {64, 128}
    assert any(c["causal"] for c in cs) and any(not c["causal"] for c in cs)
    assert any(c["kv"] is not None for c in cs)
    assert any(c["mask"] is not None for c in cs)
    assert any(c["p"] > 0 for c in cs)
    assert any(c["Nk"] != c["N"] for c in cs)
    assert any(c["host"] for c in cs)
    assert any(c["B"] * c["H"] > 1 and c["N"] % 128 != 0 for c in cs)
