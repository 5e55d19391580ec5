"""More GPU edge cases against the fp64 oracle: masks combined with dropout
at d = 128, an empty CSR mask, many tiny heads (the persistent backward's
scheduler with hundreds of items per CTA), concurrent calls on two streams
with their own workspaces, back-to-back backward calls sharing one workspace,
either side of the backward's ahead-zeroing length, fwd + bwd replayed from a
CUDA graph."""
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


def _check_all(H, oracle, x, o, lse, grads, **extra):
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    kw = dict(x.oracle_kwargs(), **extra)
    o_ref, lse_ref = oracle.forward(q, k, v, x.scale, **kw)
    H.assert_o(H.host_f64(o), o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)
    refs = oracle.backward(q, k, v, do, x.scale, **kw)
    for g, r, name in zip(grads, refs, ("dQ", "dK", "dV")):
        H.assert_grad(H.host_f64(g), r, name)


@pytest.mark.parametrize("d", [64, 128])
def test_dropout_with_every_mask(H, oracle_mod, d):
    """Causal, key padding and a block mask together, with dropout."""
    import workloads as W
    rng = np.random.default_rng(90 + d)
    w = W.make("tiny", seed=91, d=d, B=2, H=2, N=700)
    mask = (rng.random((6, 6)) < 0.6).astype(np.uint8)
    np.fill_diagonal(mask, 1)
    x = H.Inputs(w, causal=True, kv_len=np.array([700, 333], np.int32), block_mask=mask)
    p, seed = 0.2, 2**35 + 11
    o, lse = H.run_fwd_dropout(x, p, seed)
    grads = H.run_bwd_dropout(x, o, lse, p, seed)
    _check_all(H, oracle_mod, x, o, lse, grads, p8=oracle_mod.drop_p8(p), seed=seed)


@pytest.mark.parametrize("d", [64, 128])
def test_empty_csr_mask(H, oracle_mod, d):
    """nnz = 0: no query row has a key; O = 0, lse = -inf, all gradients 0."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    w = W.make("tiny", seed=92, d=d, B=1, H=2, N=300)
    x = H.Inputs(w)
    B, Hh, N = x.B, x.H, x.N
    ptr = torch.zeros(4, dtype=torch.int32, device="cuda")     # nb = 3
    o = H.nan_like_bf16((B, Hh, N, d))
    lse = torch.full((B, Hh, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_csr(x.q, x.k, x.v, o, lse, B, Hh, N, d, x.scale, 0, None, ptr, None, 0, st)
    fa.fa_check(st)
    assert torch.all(o.float() == 0) and torch.all(torch.isneginf(lse))
    shape = (B, Hh, N, d)
    dq, dk, dv = (H.nan_like_bf16(shape) for _ in range(3))
    nbytes = fa.fa_bwd_csr_workspace_size(B, Hh, N, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    fa.fa_bwd_csr(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hh, N, d, x.scale, 0, None, ptr,
                  None, 0, ws, nbytes, st)
    fa.fa_check(st)
    for g in (dq, dk, dv):
        assert torch.all(g.float() == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_many_tiny_heads(H, oracle_mod, d):
    """B*H = 2048 heads of 70 rows: far more work items than SMs, each a
    single ragged tile."""
    import workloads as W
    x = H.Inputs(W.make("tiny", seed=93, d=d, B=64, H=32, N=70, causal=True))
    o, lse = H.run_fwd(x)
    grads = H.run_bwd(x, o, lse)
    _check_all(H, oracle_mod, x, o, lse, grads)


def test_two_streams_with_their_own_workspaces(H, oracle_mod):
    """Two problems enqueued on two streams at once; each backward has its own
    workspace (and so its own work counter): both match their own oracle."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    xs = [H.Inputs(W.make("tiny", seed=94 + i, B=2, H=4, N=900, causal=bool(i))) for i in range(2)]
    streams = [torch.cuda.Stream() for _ in xs]
    outs = []
    for x in xs:   # every buffer filled on the default stream before the two streams start
        shape = (x.B, x.H, x.N, x.d)
        nbytes = fa.fa_bwd_workspace_size(x.B, x.H, x.N, x.d)
        outs.append((H.nan_like_bf16(shape),
                     torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda"),
                     tuple(H.nan_like_bf16(shape) for _ in range(3)),
                     torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")))
    torch.cuda.synchronize()
    for x, st, (o, lse, (dq, dk, dv), ws) in zip(xs, streams, outs):
        fa.fa_fwd(x.q, x.k, x.v, o, lse, x.B, x.H, x.N, x.d, x.scale, x.causal, None, None, st)
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.B, x.H, x.N, x.d, x.scale, x.causal,
                  None, None, ws, ws.numel(), st)
    for st in streams:
        fa.fa_check(st)
    for x, (o, lse, grads, _) in zip(xs, outs):
        _check_all(H, oracle_mod, x, o, lse, grads)


@pytest.mark.parametrize("d", [64, 128])
def test_forwards_on_concurrent_streams_match_serial_runs(H, d):
    """The d = 64 forward hands out its units by cancelling the launch of CTAs
    of its own grid; with three forwards (hundreds of units each, more than
    the CTAs that run) enqueued on three streams at once, every unit of every
    call must still run exactly once: O and lse equal, bit for bit, those of
    the same calls run one at a time."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    specs = [dict(seed=130, B=2, H=8, N=4096, causal=True),
             dict(seed=131, B=4, H=8, N=2048, causal=False),
             dict(seed=132, B=1, H=16, N=3000, causal=True)]
    xs = [H.Inputs(W.make("tiny", d=d, **sp)) for sp in specs]

    def run(streams):
        outs = []
        for x in xs:
            shape = (x.B, x.H, x.N, x.d)
            outs.append((H.nan_like_bf16(shape),
                         torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")))
        torch.cuda.synchronize()
        for x, st, (o, lse) in zip(xs, streams, outs):
            fa.fa_fwd(x.q, x.k, x.v, o, lse, x.B, x.H, x.N, x.d, x.scale, x.causal, None, None, st)
        for st in set(streams):
            fa.fa_check(st)
        torch.cuda.synchronize()
        return outs

    ref = run([torch.cuda.current_stream()] * len(xs))
    for _ in range(3):
        got = run([torch.cuda.Stream() for _ in xs])
        for (o, lse), (o_r, lse_r) in zip(got, ref):
            assert torch.equal(o.view(torch.int16), o_r.view(torch.int16))
            assert torch.equal(lse, lse_r)


@pytest.mark.parametrize("d,masked,N", [(64, False, 2048), (64, True, 2048), (64, False, 4096),
                                        (128, False, 2048), (128, True, 2048),
                                        (128, False, 4096)])
def test_backwards_back_to_back_share_a_workspace(H, d, masked, N):
    """Three backward calls on different inputs enqueued back to back on one
    stream, with no forward and no synchronisation between them, all sharing
    one workspace.  At d = 128, and up to N = 2048 at d = 64, each call's
    zeroing of the dQ accumulators starts without waiting for the previous
    kernel (otherwise the preprocess zeroes after its wait), so it must not
    overtake the previous call's dQ conversion (or its main kernel): every
    call's dK and dV equal, bit for bit, and its dQ matches (within the
    gradient tolerance) the same call run on its own: element by element
    within two bf16 ulps (the fp32 partial sums are added in hardware order)
    plus 1e-3 of the largest magnitude, so that even one row with a lost or
    stale partial fails."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    B, Hh = 2, 8
    nb = -(-N // 128)
    xs = []
    for i in range(3):
        mask = None
        if masked:
            m = np.random.default_rng(140 + i).random((nb, nb)) < 0.3
            mask = (m | np.eye(nb, dtype=bool)).astype(np.uint8)
        xs.append(H.Inputs(W.make("tiny", seed=140 + i, d=d, B=B, H=Hh, N=N), block_mask=mask))
    fwd = [H.run_fwd(x) for x in xs]
    solo = [H.run_bwd(x, o, lse) for x, (o, lse) in zip(xs, fwd)]
    shape = (B, Hh, N, d)
    nbytes = fa.fa_bwd_workspace_size(B, Hh, N, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    outs = [tuple(H.nan_like_bf16(shape) for _ in range(3)) for _ in xs]
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    for x, (o, lse), (dq, dk, dv) in zip(xs, fwd, outs):
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hh, N, d, x.scale, x.causal,
                  x.kv_len, x.mask, ws, nbytes, st)
    fa.fa_check(st)
    for (dq, dk, dv), (dq_s, dk_s, dv_s) in zip(outs, solo):
        assert torch.equal(dk.view(torch.int16), dk_s.view(torch.int16))
        assert torch.equal(dv.view(torch.int16), dv_s.view(torch.int16))
        got, want = H.host_f64(dq), H.host_f64(dq_s)
        assert np.all(np.isfinite(got))
        bound = 2.0 ** -6 * np.abs(want) + 1e-3 * np.abs(want).max()
        bad = np.abs(got - want) > bound
        assert not bad.any(), f"dQ: {int(bad.sum())} elements differ from the call on its own"



@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [2048, 2049])
@pytest.mark.parametrize("variant", ["causal", "kv_len"])
def test_either_side_of_the_ahead_zeroing_length(H, oracle_mod, d, N, variant):
    """At d = 64 the backward zeroes its dQ accumulators ahead of its wait
    for the previous kernel up to N = 2048 and in the preprocess beyond (at
    d = 128 always ahead): both sides against the oracle (fwd and bwd run
    back to back, without a host synchronisation between them)."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    kw = {"causal": True} if variant == "causal" else {"kv_len": np.array([N - 300], np.int32)}
    x = H.Inputs(W.make("tiny", seed=160 + N + d, d=d, B=1, H=2, N=N), **kw)
    shape = (x.B, x.H, x.N, x.d)
    o = H.nan_like_bf16(shape)
    lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    grads = tuple(H.nan_like_bf16(shape) for _ in range(3))
    nbytes = fa.fa_bwd_workspace_size(x.B, x.H, x.N, x.d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd(x.q, x.k, x.v, o, lse, x.B, x.H, x.N, x.d, x.scale, x.causal, x.kv_len, None, st)
    fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, *grads, x.B, x.H, x.N, x.d, x.scale, x.causal,
              x.kv_len, None, ws, nbytes, st)
    fa.fa_check(st)
    _check_all(H, oracle_mod, x, o, lse, grads)


def test_several_head_groups_on_a_garbage_workspace(H, oracle_mod):
    """The backward's main kernel hands out its items by head group (as many
    heads as keep their Q, dO and dQ accumulators within about half of L2):
    three groups here (36 heads of N = 8192 at d = 64, 16 per group), causal
    with ragged key padding, on a workspace filled with 0x7F bytes (3.4e38
    as fp32, so an accumulator row left unzeroed gives a huge dQ): dQ on rows
    of every head against the oracle, dK and dV on sampled key tiles, and a
    second call on the same workspace bit for bit in dK and dV and within two
    bf16 ulps (plus 1e-3 of the largest magnitude) in dQ."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    B, Hh, N, d = 3, 12, 8192, 64
    x = H.Inputs(W.make("tiny", seed=171, d=d, B=B, H=Hh, N=N), causal=True,
                 kv_len=np.array([8192, 5000, 130], np.int32))
    shape = (B, Hh, N, d)
    st = torch.cuda.current_stream()
    o = H.nan_like_bf16(shape)
    lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(x.q, x.k, x.v, o, lse, B, Hh, N, d, x.scale, x.causal, x.kv_len, None, st)
    nbytes = fa.fa_bwd_workspace_size(B, Hh, N, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    runs = []
    for _ in range(2):
        grads = tuple(H.nan_like_bf16(shape) for _ in range(3))
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, *grads, B, Hh, N, d, x.scale, x.causal,
                  x.kv_len, None, ws, nbytes, st)
        fa.fa_check(st)
        runs.append(grads)
    rng = np.random.default_rng(172)
    rows = W.sample_rows(rng, B, Hh, N, 12)
    keys = W.sample_key_tiles(rng, B, Hh, N, 1)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    dq_ref, dk_ref, dv_ref = oracle_mod.backward(q, k, v, do, x.scale, q_rows=rows, k_rows=keys,
                                                 **x.oracle_kwargs())
    dq, dk, dv = runs[0]
    H.assert_grad(H.host_f64(dq).reshape(-1, d)[rows], dq_ref, "dQ")
    H.assert_grad(H.host_f64(dk).reshape(-1, d)[keys], dk_ref, "dK")
    H.assert_grad(H.host_f64(dv).reshape(-1, d)[keys], dv_ref, "dV")
    assert np.all(np.isfinite(H.host_f64(dq)))
    dq2, dk2, dv2 = runs[1]
    assert torch.equal(dk.view(torch.int16), dk2.view(torch.int16))
    assert torch.equal(dv.view(torch.int16), dv2.view(torch.int16))
    got, want = H.host_f64(dq2), H.host_f64(dq)
    bound = 2.0 ** -6 * np.abs(want) + 1e-3 * np.abs(want).max()
    assert not (np.abs(got - want) > bound).any()


@pytest.mark.parametrize("d,masked", [(64, False), (64, True), (128, False)])
def test_fwd_bwd_captured_in_a_cuda_graph(H, d, masked):
    """fa_fwd + fa_bwd captured into a CUDA graph and replayed several times
    (after one eager call on the shapes, which configures the kernels): each
    replay gives the eager call's O, lse, dK and dV bit for bit and its dQ
    within two bf16 ulps (fp32 partial sums in hardware order)."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    B, Hh, N = 2, 4, 1000
    mask = None
    if masked:
        nb = -(-N // 128)
        m = np.random.default_rng(170).random((nb, nb)) < 0.4
        mask = (m | np.eye(nb, dtype=bool)).astype(np.uint8)
    x = H.Inputs(W.make("tiny", seed=170 + d, d=d, B=B, H=Hh, N=N), block_mask=mask)
    o_ref, lse_ref = H.run_fwd(x)
    dq_ref, dk_ref, dv_ref = H.run_bwd(x, o_ref, lse_ref)
    shape = (B, Hh, N, d)
    o = H.nan_like_bf16(shape)
    lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv = (H.nan_like_bf16(shape) for _ in range(3))
    nbytes = fa.fa_bwd_workspace_size(B, Hh, N, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            st = torch.cuda.current_stream()
            fa.fa_fwd(x.q, x.k, x.v, o, lse, B, Hh, N, d, x.scale, x.causal, x.kv_len, x.mask, st)
            fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hh, N, d, x.scale, x.causal,
                      x.kv_len, x.mask, ws, nbytes, st)
    torch.cuda.synchronize()
    for _ in range(3):
        for t in (o, dq, dk, dv):
            t.view(torch.int16).fill_(-1)
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        fa.fa_check(torch.cuda.current_stream())
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)
        assert torch.equal(dk.view(torch.int16), dk_ref.view(torch.int16))
        assert torch.equal(dv.view(torch.int16), dv_ref.view(torch.int16))
        got, want = H.host_f64(dq), H.host_f64(dq_ref)
        assert np.all(np.isfinite(got))
        bound = 2.0 ** -6 * np.abs(want) + 1e-3 * np.abs(want).max()
        assert not (np.abs(got - want) > bound).any()
