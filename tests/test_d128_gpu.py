"""GPU parity of head dimension 128 (fa_fwd / fa_bwd, the dropout and CSR
variants, fa_fwd_splitkv with d = 128) against the fp64 oracle, which takes
any d.  Same tolerances as d = 64; masks, ragged tails, empty rows and the
lazy rescale under peaky keys are covered as for d = 64."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

D = 128


@pytest.fixture(scope="module")
def H(fa_lib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gpu_harness
    return gpu_harness


def _full(H, oracle, x, bwd=True):
    o, lse = H.run_fwd(x)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    o_ref, lse_ref = oracle.forward(q, k, v, x.scale, **x.oracle_kwargs())
    H.assert_o(H.host_f64(o), o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)
    if bwd:
        dq, dk, dv = H.run_bwd(x, o, lse)
        dq_ref, dk_ref, dv_ref = oracle.backward(q, k, v, do, x.scale, **x.oracle_kwargs())
        H.assert_grad(H.host_f64(dq), dq_ref, "dQ")
        H.assert_grad(H.host_f64(dk), dk_ref, "dK")
        H.assert_grad(H.host_f64(dv), dv_ref, "dV")
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_d128_tiny(H, oracle_mod, causal):
    import workloads as W
    _full(H, oracle_mod, H.Inputs(W.make("tiny", d=D, B=2, H=2, causal=causal)))


@pytest.mark.parametrize("N", [1, 2, 127, 129, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_d128_ragged(H, oracle_mod, N, causal):
    """Several tiles with a ragged tail (and N = 1, a single key)."""
    import workloads as W
    _full(H, oracle_mod, H.Inputs(W.make("tiny", seed=10 + N, d=D, B=1, H=3, N=N,
                                         causal=causal)))


def test_d128_key_padding(H, oracle_mod):
    """BERT-shaped key padding, with lengths 0 (O = 0, lse = -inf), 1 and a
    tile edge."""
    import workloads as W
    w = W.make("bert", d=D, B=4, H=2)
    x = H.Inputs(w, kv_len=np.array([0, 1, 128, 437], np.int32))
    o, lse = _full(H, oracle_mod, x)
    assert torch.all(o[0].float() == 0) and torch.all(torch.isinf(lse[0]))


def test_d128_block_sparse_with_an_empty_row(H, oracle_mod):
    import workloads as W
    w = W.make("tiny", seed=21, d=D, B=1, H=2, N=1024)
    rng = np.random.default_rng(22)
    mask = (rng.random((8, 8)) < 0.4).astype(np.uint8)
    mask[3, :] = 0                              # query tile 3 attends nothing
    np.fill_diagonal(mask[4:, 4:], 1)
    for causal in (False, True):
        x = H.Inputs(w, causal=causal, block_mask=mask)
        o, lse = _full(H, oracle_mod, x)
        assert torch.all(o[:, :, 384:512].float() == 0)


def test_d128_all_ones_mask_equals_dense(H, oracle_mod):
    import workloads as W
    w = W.make("tiny", seed=23, d=D, B=1, H=2, N=1024)
    o1, l1 = H.run_fwd(H.Inputs(w))
    o2, l2 = H.run_fwd(H.Inputs(w, block_mask=np.ones((8, 8), np.uint8)))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_d128_long_causal_peaky_sampled_rows(H, oracle_mod):
    """The long-context causal workload at d = 128 (peaky keys stress the
    lazy rescale): forward on 256 sampled query rows per head, backward on
    those rows (dQ) and on two sampled key tiles per head (dK, dV)."""
    import workloads as W
    w = W.make("gpt2_4k", d=D, B=1, H=4)
    x = H.Inputs(w)
    o, lse = H.run_fwd(x)
    dq, dk, dv = H.run_bwd(x, o, lse)
    rng = np.random.default_rng(24)
    rows = W.sample_rows(rng, 1, 4, w.spec.N, 256)
    keys = W.sample_key_tiles(rng, 1, 4, w.spec.N, 2)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    o_ref, lse_ref = oracle_mod.forward(q, k, v, x.scale, rows=rows, **x.oracle_kwargs())
    H.assert_o(H.host_f64(o).reshape(-1, D)[rows], o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64).reshape(-1)[rows], lse_ref)
    dq_ref, dk_ref, dv_ref = oracle_mod.backward(q, k, v, do, x.scale, q_rows=rows, k_rows=keys,
                                                 **x.oracle_kwargs())
    H.assert_grad(H.host_f64(dq).reshape(-1, D)[rows], dq_ref, "dQ")
    H.assert_grad(H.host_f64(dk).reshape(-1, D)[keys], dk_ref, "dK")
    H.assert_grad(H.host_f64(dv).reshape(-1, D)[keys], dv_ref, "dV")


def test_d128_backward_is_deterministic_in_dk_dv(H, oracle_mod):
    """Two runs give bitwise equal dK and dV (no atomics there); dQ, summed
    by reduce-adds in any order, agrees to fp32 rounding."""
    import workloads as W
    x = H.Inputs(W.make("tiny", seed=25, d=D, B=2, H=2, N=1000, causal=True))
    o, lse = H.run_fwd(x)
    a = H.run_bwd(x, o, lse)
    b = H.run_bwd(x, o, lse)
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    assert torch.equal(a[2].view(torch.int16), b[2].view(torch.int16))
    assert H.rel_fro(H.host_f64(a[0]), H.host_f64(b[0])) <= 1e-2


@pytest.mark.parametrize("p,seed", [(0.1, 5), (0.5, 2**33 + 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_d128_dropout(H, oracle_mod, p, seed, causal):
    import workloads as W
    x = H.Inputs(W.make("tiny", seed=30, d=D, B=2, H=2, N=300, causal=causal))
    o, lse = H.run_fwd_dropout(x, p, seed)
    dq, dk, dv = H.run_bwd_dropout(x, o, lse, p, seed)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    kw = dict(x.oracle_kwargs(), p8=oracle_mod.drop_p8(p), seed=seed)
    o_ref, lse_ref = oracle_mod.forward(q, k, v, x.scale, **kw)
    H.assert_o(H.host_f64(o), o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)
    dq_ref, dk_ref, dv_ref = oracle_mod.backward(q, k, v, do, x.scale, **kw)
    H.assert_grad(H.host_f64(dq), dq_ref, "dQ")
    H.assert_grad(H.host_f64(dk), dk_ref, "dK")
    H.assert_grad(H.host_f64(dv), dv_ref, "dV")


@pytest.mark.parametrize("Nq,Nk,S", [(1, 8192, 0), (1, 8192, 7), (16, 1000, 0), (200, 333, 3),
                                     (3, 1, 0)])
def test_d128_splitkv(H, oracle_mod, Nq, Nk, S):
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    rng = np.random.default_rng(40 + Nq)
    B, Hh = 2, 4
    q, k, v = (W.f32_to_bf16_bits(rng.standard_normal((B, Hh, n, D), dtype=np.float32))
               for n in (Nq, Nk, Nk))
    kv_len = np.array([Nk, max(0, Nk // 3)], np.int32)
    dq, dk, dv = (H.dev_bf16(t) for t in (q, k, v))
    o = H.nan_like_bf16((B, Hh, Nq, D))
    lse = torch.full((B, Hh, Nq), float("nan"), dtype=torch.float32, device="cuda")
    kl = torch.from_numpy(kv_len).cuda()
    nbytes = fa.fa_fwd_splitkv_workspace_size(B, Hh, Nq, Nk, D, S)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_splitkv(dq, dk, dv, o, lse, B, Hh, Nq, Nk, D, 0.125, kl, S, ws, nbytes, st)
    fa.fa_check(st)
    o_ref, lse_ref = oracle_mod.forward_qk(W.bf16_bits_to_f64(q), W.bf16_bits_to_f64(k),
                                           W.bf16_bits_to_f64(v), 0.125, kv_len=kv_len)
    H.assert_o(H.host_f64(o), o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)


def test_d128_bert_full(H, oracle_mod):
    """The BERT-shaped workload at d = 128, every output against the oracle."""
    import workloads as W
    _full(H, oracle_mod, H.Inputs(W.make("bert", d=D)))


def test_d128_block_sparse_64k_sampled(H, oracle_mod):
    """The 64K block-sparse workload at d = 128 (two heads), checked on sampled
    query rows (O, lse, dQ) and sampled key tiles (dK, dV)."""
    import workloads as W
    w = W.make("sparse64k", d=D, H=2)
    x = H.Inputs(w)
    o, lse = H.run_fwd(x)
    dq, dk, dv = H.run_bwd(x, o, lse)
    rng = np.random.default_rng(26)
    rows = W.sample_rows(rng, 1, 2, w.spec.N, 128)
    keys = W.sample_key_tiles(rng, 1, 2, w.spec.N, 2)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    o_ref, lse_ref = oracle_mod.forward(q, k, v, x.scale, rows=rows, **x.oracle_kwargs())
    H.assert_o(H.host_f64(o).reshape(-1, D)[rows], o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64).reshape(-1)[rows], lse_ref)
    dq_ref, dk_ref, dv_ref = oracle_mod.backward(q, k, v, do, x.scale, q_rows=rows, k_rows=keys,
                                                 **x.oracle_kwargs())
    H.assert_grad(H.host_f64(dq).reshape(-1, D)[rows], dq_ref, "dQ")
    H.assert_grad(H.host_f64(dk).reshape(-1, D)[keys], dk_ref, "dK")
    H.assert_grad(H.host_f64(dv).reshape(-1, D)[keys], dv_ref, "dV")
