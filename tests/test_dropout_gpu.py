"""GPU parity of the fused dropout path against the fp64 oracle with the same
keep mask (the counter-based hash of include/fa.h, implemented independently
on both sides, so the masks agree bit for bit and the tolerances are those of
plain attention)."""
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


def _check(H, oracle, x, p, seed, rows=None, keys=None):
    p8 = oracle.drop_p8(p)
    o, lse = H.run_fwd_dropout(x, p, seed)
    dq, dk, dv = H.run_bwd_dropout(x, o, lse, p, seed)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    kw = dict(x.oracle_kwargs(), p8=p8, seed=seed)
    d = x.d
    if rows is None:
        o_ref, lse_ref = oracle.forward(q, k, v, x.scale, **kw)
        H.assert_o(H.host_f64(o), o_ref)
        H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)
        dq_ref, dk_ref, dv_ref = oracle.backward(q, k, v, do, x.scale, **kw)
        H.assert_grad(H.host_f64(dq), dq_ref, "dQ")
        H.assert_grad(H.host_f64(dk), dk_ref, "dK")
        H.assert_grad(H.host_f64(dv), dv_ref, "dV")
    else:
        o_ref, lse_ref = oracle.forward(q, k, v, x.scale, rows=rows, **kw)
        H.assert_o(H.host_f64(o).reshape(-1, d)[rows], o_ref)
        H.assert_lse(lse.cpu().numpy().astype(np.float64).reshape(-1)[rows], lse_ref)
        dq_ref, dk_ref, dv_ref = oracle.backward(q, k, v, do, x.scale, q_rows=rows, k_rows=keys,
                                                 **kw)
        H.assert_grad(H.host_f64(dq).reshape(-1, d)[rows], dq_ref, "dQ")
        H.assert_grad(H.host_f64(dk).reshape(-1, d)[keys], dk_ref, "dK")
        H.assert_grad(H.host_f64(dv).reshape(-1, d)[keys], dv_ref, "dV")
    return o, lse


@pytest.mark.parametrize("p,seed", [(0.1, 1), (0.5, 2**40 + 7), (0.75, 3)])
def test_dropout_tiny_full(H, oracle_mod, p, seed):
    import workloads as W
    _check(H, oracle_mod, H.Inputs(W.make("tiny", B=2, H=2)), p, seed)


# N = 1 is left to the plain ragged test: with one key the exact dQ and dK are
# 0 (dS = P (Z dP / (1-p') - D) with D = Z dP / (1-p')), so a relative norm
# only measures the bf16 rounding of the stored O that D is computed from.
@pytest.mark.parametrize("N", [2, 127, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_dropout_ragged(H, oracle_mod, N, causal):
    import workloads as W
    w = W.make("tiny", seed=200 + N, B=2, H=3, N=N)
    _check(H, oracle_mod, H.Inputs(w, causal=causal), 0.2, 11 + N)


def test_dropout_bert_key_padding(H, oracle_mod):
    import workloads as W
    _check(H, oracle_mod, H.Inputs(W.make("bert", B=4)), 0.1, 12345)


def test_dropout_gpt2_causal(H, oracle_mod):
    import workloads as W
    _check(H, oracle_mod, H.Inputs(W.make("gpt2", B=2)), 0.1, 777)


def test_dropout_mask_and_kv_len(H, oracle_mod):
    import workloads as W
    w = W.make("tiny", seed=13, B=2, H=2, N=512)
    mask = np.array([[1, 0, 1, 0], [0, 1, 0, 0], [1, 1, 1, 0], [0, 0, 1, 1]], np.uint8)
    x = H.Inputs(w, causal=True, block_mask=mask, kv_len=np.array([512, 300], np.int32))
    _check(H, oracle_mod, x, 0.3, 99)


def test_dropout_gpt2_4k_sampled(H, oracle_mod):
    import workloads as W
    x = H.Inputs(W.make("gpt2_4k"))
    rng = np.random.default_rng(41)
    rows = W.sample_rows(rng, x.B, x.H, x.N, 64)
    keys = W.sample_key_tiles(rng, x.B, x.H, x.N, 1)
    _check(H, oracle_mod, x, 0.1, 4242, rows=rows, keys=keys)


def test_zero_dropout_is_bitwise_plain(H, oracle_mod):
    """p = 0 through the dropout entry points runs the plain kernels."""
    import workloads as W
    x = H.Inputs(W.make("gpt2", B=1))
    o1, l1 = H.run_fwd(x)
    o2, l2 = H.run_fwd_dropout(x, 0.0, 5)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    g2 = H.run_bwd_dropout(x, o2, l2, 0.0, 5)
    g1 = H.run_bwd(x, o1, l1)
    assert torch.equal(g1[1].view(torch.int16), g2[1].view(torch.int16))
    assert torch.equal(g1[2].view(torch.int16), g2[2].view(torch.int16))


def test_dropout_changes_with_seed_and_keeps_lse(H, oracle_mod):
    import workloads as W
    x = H.Inputs(W.make("gpt2", B=1))
    o0, l0 = H.run_fwd(x)
    o1, l1 = H.run_fwd_dropout(x, 0.25, 1)
    o2, l2 = H.run_fwd_dropout(x, 0.25, 2)
    # lse is taken before dropout
    assert torch.allclose(l0, l1, rtol=1e-6, atol=0) and torch.allclose(l0, l2, rtol=1e-6, atol=0)
    assert not torch.equal(o1, o2)
