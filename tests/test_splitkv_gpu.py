"""GPU parity of the split-KV forward (short query block against a long
key/value cache, key range split across CTAs and merged) against the fp64
oracle's forward with Nq query rows and Nk key rows."""
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


def _inputs(seed, B, Hh, Nq, Nk, d=64):
    import workloads as W
    rng = np.random.default_rng(seed)
    q = W.f32_to_bf16_bits(rng.standard_normal((B, Hh, Nq, d), dtype=np.float32))
    k = W.f32_to_bf16_bits(rng.standard_normal((B, Hh, Nk, d), dtype=np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((B, Hh, Nk, d), dtype=np.float32))
    return q, k, v


def _run(H, q, k, v, scale, kv_len=None, num_splits=0):
    import exact_io_aware_25_gb300 as fa
    B, Hh, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv = (H.dev_bf16(x) for x in (q, k, v))
    o = H.nan_like_bf16((B, Hh, Nq, d))
    lse = torch.full((B, Hh, Nq), float("nan"), dtype=torch.float32, device="cuda")
    kl = None if kv_len is None else torch.from_numpy(np.asarray(kv_len, np.int32)).cuda()
    nbytes = fa.fa_fwd_splitkv_workspace_size(B, Hh, Nq, Nk, d, num_splits)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_splitkv(dq, dk, dv, o, lse, B, Hh, Nq, Nk, d, scale, kl, num_splits, ws, nbytes, st)
    fa.fa_check(st)
    return o, lse


def _check(H, oracle, q, k, v, scale=0.125, kv_len=None, num_splits=0):
    import workloads as W
    o, lse = _run(H, q, k, v, scale, kv_len, num_splits)
    o_ref, lse_ref = oracle.forward_qk(W.bf16_bits_to_f64(q), W.bf16_bits_to_f64(k),
                                       W.bf16_bits_to_f64(v), scale, kv_len=kv_len)
    H.assert_o(H.host_f64(o), o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)
    return o, lse


@pytest.mark.parametrize("num_splits", [0, 1, 3, 64])
def test_decode_one_query(H, oracle_mod, num_splits):
    q, k, v = _inputs(1, 2, 8, 1, 8192)
    _check(H, oracle_mod, q, k, v, num_splits=num_splits)


@pytest.mark.parametrize("Nq,Nk", [(16, 1000), (128, 4096), (200, 333), (7, 129), (3, 1)])
def test_short_queries_ragged_lengths(H, oracle_mod, Nq, Nk):
    q, k, v = _inputs(2 + Nq, 2, 4, Nq, Nk)
    _check(H, oracle_mod, q, k, v, num_splits=0)
    _check(H, oracle_mod, q, k, v, num_splits=5)


def test_key_padding_including_empty_batches(H, oracle_mod):
    """kv_len per batch, with 0 (O = 0, lse = -inf), 1, a tile edge and a
    length past the last split's start."""
    q, k, v = _inputs(3, 4, 2, 4, 3000)
    o, lse = _check(H, oracle_mod, q, k, v, kv_len=np.array([0, 1, 128, 2999], np.int32),
                    num_splits=6)
    assert torch.all(o[0].float() == 0) and torch.all(torch.isinf(lse[0]))


def test_splitkv_agrees_with_the_plain_forward(H, oracle_mod):
    """Nq == Nk, no mask: the split-and-merge result equals fa_fwd's to
    rounding (different summation grouping)."""
    import workloads as W
    w = W.make("gpt2", B=1, causal=False)
    x = H.Inputs(w, causal=False)
    o1, l1 = H.run_fwd(x)
    o2, l2 = _run(H, w.q, w.k, w.v, w.spec.scale, num_splits=4)
    assert torch.allclose(l1, l2, rtol=0, atol=1e-4)
    assert (o1.float() - o2.float()).abs().max().item() < 2e-2


def test_long_cache_many_heads(H, oracle_mod):
    """A decode-shaped problem at size (B16 H16, one query, 32K keys) on
    sampled heads."""
    import workloads as W
    q, k, v = _inputs(5, 16, 16, 1, 32768)
    o, lse = _run(H, q, k, v, 0.125, num_splits=0)
    heads = [(0, 0), (3, 7), (15, 15)]
    for b, h in heads:
        o_ref, lse_ref = oracle_mod.forward_qk(W.bf16_bits_to_f64(q[b:b + 1, h:h + 1]),
                                               W.bf16_bits_to_f64(k[b:b + 1, h:h + 1]),
                                               W.bf16_bits_to_f64(v[b:b + 1, h:h + 1]), 0.125)
        H.assert_o(H.host_f64(o[b:b + 1, h:h + 1]), o_ref)
        H.assert_lse(lse[b:b + 1, h:h + 1].cpu().numpy().astype(np.float64), lse_ref)
