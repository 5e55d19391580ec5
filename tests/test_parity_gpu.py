"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.

Small and mid-size workloads are compared element by element over every
output.  The two large workloads (B=2 H=12 N=4096 causal with peaky keys, and
the 64K block-sparse one) run at full size in the launch configuration the
benchmark times, and are compared on seeded samples: 256 query rows per
(b, h) for O, lse and dQ, and two whole key tiles per (b, h) for dK and dV.
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


def _full_check(H, oracle, x, check_bwd=True):
    o, lse = H.run_fwd(x)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    o_ref, lse_ref = oracle.forward(q, k, v, x.scale, **x.oracle_kwargs())
    H.assert_o(H.host_f64(o), o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_ref)
    if not check_bwd:
        return o, lse
    dq, dk, dv = H.run_bwd(x, o, lse)
    dq_ref, dk_ref, dv_ref = oracle.backward(q, k, v, do, x.scale, **x.oracle_kwargs())
    H.assert_grad(H.host_f64(dq), dq_ref, "dQ")
    H.assert_grad(H.host_f64(dk), dk_ref, "dK")
    H.assert_grad(H.host_f64(dv), dv_ref, "dV")
    return o, lse


def _sampled_check(H, oracle, x, rows_per_head=256, key_tiles_per_head=2, seed=1234):
    import workloads as W
    rng = np.random.default_rng(seed)
    B, Hh, N, d = x.B, x.H, x.N, x.d
    o, lse = H.run_fwd(x)
    dq, dk, dv = H.run_bwd(x, o, lse)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    rows = W.sample_rows(rng, B, Hh, N, rows_per_head)
    keys = W.sample_key_tiles(rng, B, Hh, N, key_tiles_per_head)
    o_ref, lse_ref = oracle.forward(q, k, v, x.scale, rows=rows, **x.oracle_kwargs())
    H.assert_o(H.host_f64(o).reshape(-1, d)[rows], o_ref)
    H.assert_lse(lse.cpu().numpy().astype(np.float64).reshape(-1)[rows], lse_ref)
    dq_ref, dk_ref, dv_ref = oracle.backward(q, k, v, do, x.scale, q_rows=rows, k_rows=keys,
                                             **x.oracle_kwargs())
    H.assert_grad(H.host_f64(dq).reshape(-1, d)[rows], dq_ref, "dQ")
    H.assert_grad(H.host_f64(dk).reshape(-1, d)[keys], dk_ref, "dK")
    H.assert_grad(H.host_f64(dv).reshape(-1, d)[keys], dv_ref, "dV")


# ---------------------------------------------------------------- the five workloads


def test_tiny(H, oracle_mod):
    import workloads as W
    _full_check(H, oracle_mod, H.Inputs(W.make("tiny")))


def test_bert_key_padding(H, oracle_mod):
    import workloads as W
    _full_check(H, oracle_mod, H.Inputs(W.make("bert")))


def test_gpt2_causal(H, oracle_mod):
    import workloads as W
    _full_check(H, oracle_mod, H.Inputs(W.make("gpt2")))


def test_gpt2_4k_causal_peaky_sampled(H, oracle_mod):
    import workloads as W
    _sampled_check(H, oracle_mod, H.Inputs(W.make("gpt2_4k")))


def test_sparse64k_sampled(H, oracle_mod):
    import workloads as W
    _sampled_check(H, oracle_mod, H.Inputs(W.make("sparse64k")), rows_per_head=128,
                   key_tiles_per_head=2)


@pytest.mark.parametrize("N,d,density,causal,kv,empty_cols", [
    (131072, 64, 0.01, False, None, False),    # 1024 key tiles: the most a block mask may have
    (100000, 128, 0.03, True, None, True),     # 782 tiles: a partial last group of columns
    (66000, 64, 0.03, False, [40000], True),
    (33000, 128, 0.05, True, [33000], False),
])
def test_block_mask_at_large_n(H, oracle_mod, N, d, density, causal, kv, empty_cols):
    """Block masks past the 64K workload's 512 key tiles, up to the 1024-tile
    maximum, with empty key columns, causal and key padding: the per-key-tile
    query lists of the backward span several groups of columns and both rounds
    of their mask loads.  Sampled rows and key tiles against the oracle."""
    import workloads as W
    rng = np.random.default_rng(N + d)
    nb = -(-N // 128)
    mask = (rng.random((nb, nb)) < density).astype(np.uint8)
    if empty_cols:
        mask[:, rng.choice(nb, size=nb // 4, replace=False)] = 0
    w = W.make("tiny", seed=N % 1000 + d, d=d, B=1, H=1, N=N)
    x = H.Inputs(w, causal=causal, block_mask=mask,
                 kv_len=None if kv is None else np.array(kv, np.int32))
    _sampled_check(H, oracle_mod, x, rows_per_head=48, key_tiles_per_head=3, seed=N)


# ---------------------------------------------------------------- edge cases


@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(H, oracle_mod, N, causal):
    import workloads as W
    w = W.make("tiny", seed=100 + N, B=2, H=3, N=N)
    _full_check(H, oracle_mod, H.Inputs(w, causal=causal))


@pytest.mark.parametrize("kv", [[1, 300], [0, 129], [128, 77], [300, 256]])
def test_key_padding_edges(H, oracle_mod, kv):
    """kv_len of 0 (every row empty: O = 0, lse = -inf), 1, tile edges."""
    import workloads as W
    w = W.make("tiny", seed=7, B=2, H=2, N=300)
    _full_check(H, oracle_mod, H.Inputs(w, kv_len=np.array(kv, np.int32)))


def test_many_key_tiles_without_work(H, oracle_mod):
    """More (key tile, head) items than SMs, most of them with no query tile
    to visit (keys past kv_len): their dK / dV are zero and the items around
    them are unaffected."""
    import workloads as W
    w = W.make("tiny", seed=11, B=4, H=4, N=4096)
    x = H.Inputs(w, kv_len=np.array([130, 4096, 1, 300], np.int32))
    _sampled_check(H, oracle_mod, x, rows_per_head=64, key_tiles_per_head=3, seed=5)
    _, dk, dv = H.run_bwd(x, *H.run_fwd(x))
    assert torch.all(dk[0, :, 256:].float() == 0) and torch.all(dv[2, :, 128:].float() == 0)


def test_block_mask_with_empty_key_columns(H, oracle_mod):
    """A block mask whose key-tile columns are mostly empty, over more items
    than SMs, with causal on top."""
    import workloads as W
    w = W.make("tiny", seed=12, B=2, H=8, N=4096)
    rng = np.random.default_rng(12)
    mask = np.zeros((32, 32), np.uint8)
    cols = rng.choice(32, size=6, replace=False)
    mask[:, cols] = rng.integers(0, 2, size=(32, 6)).astype(np.uint8)
    x = H.Inputs(w, causal=True, block_mask=mask)
    _sampled_check(H, oracle_mod, x, rows_per_head=64, key_tiles_per_head=3, seed=6)
    _, dk, _ = H.run_bwd(x, *H.run_fwd(x))
    empty = [c for c in range(32) if c not in set(cols.tolist())]
    for c in empty[:4]:
        assert torch.all(dk[:, :, c * 128:(c + 1) * 128].float() == 0)


def test_mask_with_empty_rows_and_causal(H, oracle_mod):
    import workloads as W
    w = W.make("tiny", seed=8, B=1, H=2, N=500)
    mask = np.array([[0, 0, 0, 0], [1, 0, 1, 1], [0, 1, 0, 0], [1, 1, 1, 1]], np.uint8)
    _full_check(H, oracle_mod, H.Inputs(w, causal=True, block_mask=mask,
                                        kv_len=np.array([450], np.int32)))


def test_all_ones_mask_equals_dense_bitwise(H, oracle_mod):
    """All-ones block mask at N=4096 gives bit-identical O, lse, dK, dV to no
    mask (same tiles in the same order); dQ, accumulated with atomics, agrees
    to rounding."""
    import workloads as W
    w = W.make("sparse64k", N=4096)
    x_dense = H.Inputs(w, block_mask=None)
    x_dense.mask_np, x_dense.mask = None, None
    x_ones = H.Inputs(w, block_mask=np.ones((32, 32), np.uint8))
    o1, l1 = H.run_fwd(x_dense)
    o2, l2 = H.run_fwd(x_ones)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    g1 = H.run_bwd(x_dense, o1, l1)
    g2 = H.run_bwd(x_ones, o2, l2)
    assert torch.equal(g1[1].view(torch.int16), g2[1].view(torch.int16))
    assert torch.equal(g1[2].view(torch.int16), g2[2].view(torch.int16))
    assert H.rel_fro(H.host_f64(g2[0]), H.host_f64(g1[0])) < 1e-3
    # and the dense result itself matches the oracle on sampled rows
    rng = np.random.default_rng(3)
    rows = W.sample_rows(rng, 1, 8, 4096, 64)
    o_ref, lse_ref = oracle_mod.forward(x_dense.f64("q"), x_dense.f64("k"), x_dense.f64("v"),
                                        x_dense.scale, rows=rows)
    H.assert_o(H.host_f64(o1).reshape(-1, 64)[rows], o_ref)


def test_masked_blocks_do_not_leak(H, oracle_mod):
    """K/V values inside masked-out blocks and past kv_len never reach O or
    lse (bitwise), and the gradients of never-attended keys are exactly 0."""
    import workloads as W
    w = W.make("tiny", seed=9, B=2, H=2, N=512)
    mask = np.array([[1, 0, 1, 0], [0, 1, 0, 0], [1, 1, 1, 0], [0, 0, 1, 1]], np.uint8)
    kv_len = np.array([512, 300], np.int32)
    x = H.Inputs(w, block_mask=mask, kv_len=kv_len)
    o1, l1 = H.run_fwd(x)
    k2 = x.k.clone()
    v2 = x.v.clone()
    k2[1, :, 300:] = 77.0
    v2[1, :, 300:] = -33.0
    o2, l2 = H.run_fwd(x, k=k2, v=v2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    dq, dk, dv = H.run_bwd(x, o1, l1)
    assert torch.all(dk[1, :, 300:].float() == 0) and torch.all(dv[1, :, 300:].float() == 0)


def test_constant_values(H, oracle_mod):
    import workloads as W
    w = W.make("gpt2", B=1, H=2)
    x = H.Inputs(w)
    c = torch.linspace(-2, 2, 64, device="cuda").to(torch.bfloat16)
    v = c.expand(1, 2, 1024, 64).contiguous()
    o, _ = H.run_fwd(x, v=v)
    want = np.broadcast_to(H.host_f64(c), (1, 2, 1024, 64))
    H.assert_o(H.host_f64(o), want)


def test_timeout_path_reports_status_without_fault(H):
    """A starved producer makes the consumers' bounded waits run out: the
    kernel returns early, fa_check reports FA_ERR_TIMEOUT, and the context
    stays usable."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    x = H.Inputs(W.make("tiny"))
    fa.fa_set_wait_timeout_ns(50_000_000)
    try:
        fa.fa_debug_starve_next_fwd(True)
        shape = (x.B, x.H, x.N, x.d)
        o = H.nan_like_bf16(shape)
        lse = torch.empty((x.B, x.H, x.N), dtype=torch.float32, device="cuda")
        st = torch.cuda.current_stream()
        fa.fa_fwd(x.q, x.k, x.v, o, lse, x.B, x.H, x.N, x.d, x.scale, 0, None, None, st)
        with pytest.raises(fa.FaError) as ei:
            fa.fa_check(st)
        assert ei.value.status == fa.FA_ERR_TIMEOUT
    finally:
        fa.fa_debug_starve_next_fwd(False)
        fa.fa_set_wait_timeout_ns(0)
    # the next call works normally
    o, lse = H.run_fwd(x)
    assert torch.isfinite(o.float()).all()
