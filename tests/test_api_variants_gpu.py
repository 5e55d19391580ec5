"""GPU parity of the API variants against the fp64 oracle:

* fa_fwd_stats: the row statistics (m, l) next to O and lse;
* fa_fwd_csr / fa_bwd_csr: the block mask given as CSR (unsorted, with
  repeated entries) equals the dense mask, and bad entries are reported;
* fa_fwd_qk / fa_bwd_qk: Nq != Nk with the bottom-right causal mask.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL_M_MAXABS = 1e-3   # m is a max of fp32 scores, like lse
TOL_L_REL = 2e-3      # l: fp32 sum of ex2.approx terms


@pytest.fixture(scope="module")
def H(fa_lib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gpu_harness
    return gpu_harness


def _stats(H, x):
    import exact_io_aware_25_gb300 as fa
    shape = (x.B, x.H, x.N)
    o = H.nan_like_bf16((x.B, x.H, x.N, x.d))
    lse, m, l = (torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
                 for _ in range(3))
    st = torch.cuda.current_stream()
    fa.fa_fwd_stats(x.q, x.k, x.v, o, lse, m, l, x.B, x.H, x.N, x.d, x.scale, x.causal,
                    x.kv_len, x.mask, st)
    fa.fa_check(st)
    return o, lse, m, l


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("variant", ["plain", "causal", "kv_len", "mask"])
def test_row_statistics(H, oracle_mod, d, variant):
    import workloads as W
    w = W.make("tiny", seed=70, d=d, B=2, H=2, N=700)
    kw = {}
    if variant == "causal":
        kw["causal"] = True
    if variant == "kv_len":
        kw["kv_len"] = np.array([0, 333], np.int32)
    if variant == "mask":
        m = (np.random.default_rng(71).random((6, 6)) < 0.5).astype(np.uint8)
        m[2, :] = 0
        kw["block_mask"] = m
    x = H.Inputs(w, **kw)
    o, lse, m_g, l_g = _stats(H, x)
    o1, lse1 = H.run_fwd(x)
    assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse, lse1)
    o_r, lse_r, m_r, l_r = oracle_mod.forward_stats(x.f64("q"), x.f64("k"), x.f64("v"), x.scale,
                                                    **x.oracle_kwargs())
    H.assert_o(H.host_f64(o), o_r)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_r)
    m_g, l_g = m_g.cpu().numpy().astype(np.float64), l_g.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(m_g), np.isneginf(m_r))
    fin = np.isfinite(m_r)
    assert np.all(l_g[~fin] == 0)
    assert float(np.max(np.abs(m_g[fin] - m_r[fin]))) <= TOL_M_MAXABS
    assert float(np.max(np.abs(l_g[fin] / l_r[fin] - 1))) <= TOL_L_REL


def _csr_from_dense(mask, rng, dup=True):
    """CSR of a dense block mask with each row's entries shuffled and, when
    dup, some repeated."""
    ptr, idx = [0], []
    for r in range(mask.shape[0]):
        cols = list(np.flatnonzero(mask[r]))
        if dup and cols:
            cols += list(rng.choice(cols, size=min(3, len(cols))))
        rng.shuffle(cols)
        idx += cols
        ptr.append(len(idx))
    return np.array(ptr, np.int32), np.array(idx if idx else [0], np.int32), len(idx)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_csr_mask_equals_dense_mask(H, oracle_mod, d, causal):
    """fa_fwd_csr equals fa_fwd with the same mask bit for bit (O, lse); for
    d = 64 fa_bwd_csr equals fa_bwd (dK, dV bitwise, dQ to fp32 summation
    order); and the oracle agrees."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    rng = np.random.default_rng(72 + d)
    w = W.make("tiny", seed=73, d=d, B=2, H=2, N=1200)
    nb = 10
    mask = (rng.random((nb, nb)) < 0.35).astype(np.uint8)
    mask[4, :] = 0
    np.fill_diagonal(mask[6:, 6:], 1)
    ptr, idx, nnz = _csr_from_dense(mask, rng)
    x = H.Inputs(w, causal=causal, block_mask=mask)
    dptr, didx = torch.from_numpy(ptr).cuda(), torch.from_numpy(idx).cuda()
    o = H.nan_like_bf16((x.B, x.H, x.N, d))
    lse = torch.full((x.B, x.H, x.N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_csr(x.q, x.k, x.v, o, lse, x.B, x.H, x.N, d, x.scale, causal, None, dptr, didx,
                  nnz, st)
    fa.fa_check(st)
    o1, lse1 = H.run_fwd(x)
    assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse, lse1)
    o_r, lse_r = oracle_mod.forward(x.f64("q"), x.f64("k"), x.f64("v"), x.scale,
                                    **x.oracle_kwargs())
    H.assert_o(H.host_f64(o), o_r)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_r)
    if d != 64:
        return
    shape = (x.B, x.H, x.N, d)
    dq, dk, dv = (H.nan_like_bf16(shape) for _ in range(3))
    nbytes = fa.fa_bwd_csr_workspace_size(x.B, x.H, x.N, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    fa.fa_bwd_csr(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.B, x.H, x.N, d, x.scale, causal,
                  None, dptr, didx, nnz, ws, nbytes, st)
    fa.fa_check(st)
    dq1, dk1, dv1 = H.run_bwd(x, o1, lse1)
    assert torch.equal(dk.view(torch.int16), dk1.view(torch.int16))
    assert torch.equal(dv.view(torch.int16), dv1.view(torch.int16))
    assert H.rel_fro(H.host_f64(dq), H.host_f64(dq1)) <= 1e-2
    dq_r, dk_r, dv_r = oracle_mod.backward(x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do"),
                                           x.scale, **x.oracle_kwargs())
    H.assert_grad(H.host_f64(dq), dq_r, "dQ")
    H.assert_grad(H.host_f64(dk), dk_r, "dK")
    H.assert_grad(H.host_f64(dv), dv_r, "dV")


def test_csr_bad_entries_are_reported(H):
    """A tile index past nb and a row range past nnz are skipped by the
    kernels' own bounds checks and reported as FA_ERR_INVALID_ARG."""
    import exact_io_aware_25_gb300 as fa
    import workloads as W
    w = W.make("tiny", seed=74, B=1, H=1, N=512)
    x = H.Inputs(w)
    st = torch.cuda.current_stream()
    o = torch.empty((1, 1, 512, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 1, 512), dtype=torch.float32, device="cuda")
    bad = [
        (np.array([0, 1, 2, 3, 4], np.int32), np.array([0, 1, 9, 3], np.int32), 4),  # col 9 >= nb 4
        (np.array([0, 1, 2, 3, 6], np.int32), np.array([0, 1, 2, 3], np.int32), 4),  # end 6 > nnz
    ]
    for ptr, idx, nnz in bad:
        fa.fa_fwd_csr(x.q, x.k, x.v, o, lse, 1, 1, 512, 64, 0.125, 0, None,
                      torch.from_numpy(ptr).cuda(), torch.from_numpy(idx).cuda(), nnz, st)
        with pytest.raises(fa.FaError) as e:
            fa.fa_check(st)
        assert e.value.status == fa.FA_ERR_INVALID_ARG
    fa.fa_check(st)   # the error word was cleared


def _qk(H, q, k, v, causal, kv_len=None, scale=0.125):
    import exact_io_aware_25_gb300 as fa
    B, Hh, Nq, d = q.shape
    Nk = k.shape[2]
    dq_, dk_, dv_ = (H.dev_bf16(t) for t in (q, k, v))
    o = H.nan_like_bf16((B, Hh, Nq, d))
    lse = torch.full((B, Hh, Nq), float("nan"), dtype=torch.float32, device="cuda")
    kl = None if kv_len is None else torch.from_numpy(np.asarray(kv_len, np.int32)).cuda()
    st = torch.cuda.current_stream()
    fa.fa_fwd_qk(dq_, dk_, dv_, o, lse, B, Hh, Nq, Nk, d, scale, causal, kl, st)
    fa.fa_check(st)
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (100, 1000), (128, 4096), (300, 333), (500, 200),
                                   (257, 257)])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_qk_bottom_right_causal(H, oracle_mod, d, Nq, Nk, causal):
    import workloads as W
    rng = np.random.default_rng(80 + Nq + Nk + d)
    B, Hh = 2, 3
    q, k, v = (W.f32_to_bf16_bits(rng.standard_normal((B, Hh, n, d), dtype=np.float32))
               for n in (Nq, Nk, Nk))
    kv_len = np.array([Nk, max(1, (2 * Nk) // 3)], np.int32)
    o, lse = _qk(H, q, k, v, causal, kv_len)
    o_r, lse_r = oracle_mod.forward_qk(W.bf16_bits_to_f64(q), W.bf16_bits_to_f64(k),
                                       W.bf16_bits_to_f64(v), 0.125, kv_len=kv_len, causal=causal)
    H.assert_o(H.host_f64(o), o_r)
    H.assert_lse(lse.cpu().numpy().astype(np.float64), lse_r)


def test_fwd_qk_square_equals_fa_fwd(H):
    import workloads as W
    w = W.make("gpt2", B=1, H=2)
    x = H.Inputs(w)
    o1, l1 = H.run_fwd(x)
    o2, l2 = _qk(H, w.q, w.k, w.v, True, scale=w.spec.scale)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def _bwd_qk(H, q, k, v, do, o, lse, causal, kv_len=None, scale=0.125):
    import exact_io_aware_25_gb300 as fa
    B, Hh, Nq, d = q.shape
    Nk = k.shape[2]
    tq, tk, tv, tdo = (H.dev_bf16(t) for t in (q, k, v, do))
    dq = H.nan_like_bf16((B, Hh, Nq, d))
    dk, dv = H.nan_like_bf16((B, Hh, Nk, d)), H.nan_like_bf16((B, Hh, Nk, d))
    kl = None if kv_len is None else torch.from_numpy(np.asarray(kv_len, np.int32)).cuda()
    nbytes = fa.fa_bwd_workspace_size(B, Hh, Nq, d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_bwd_qk(tq, tk, tv, o, lse, tdo, dq, dk, dv, B, Hh, Nq, Nk, d, scale, causal, kl, ws,
                 nbytes, st)
    fa.fa_check(st)
    return dq, dk, dv


def _qk_inputs(rng, B, Hh, Nq, Nk, d):
    import workloads as W
    return tuple(W.f32_to_bf16_bits(rng.standard_normal((B, Hh, n, d), dtype=np.float32))
                 for n in (Nq, Nk, Nk, Nq))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (100, 1000), (300, 333), (500, 200), (200, 777),
                                   (128, 4096)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_qk_bottom_right_causal(H, oracle_mod, d, Nq, Nk, causal):
    """Every dQ, dK, dV of the Nq x Nk problem against the oracle's backward
    (offsets Nk - Nq that are not multiples of the 128-row tile, Nq > Nk with
    query rows that see no key, key padding)."""
    import workloads as W
    rng = np.random.default_rng(180 + Nq + Nk + d)
    B, Hh = 2, 3
    q, k, v, do = _qk_inputs(rng, B, Hh, Nq, Nk, d)
    kv_len = np.array([Nk, max(1, (2 * Nk) // 3)], np.int32)
    o, lse = _qk(H, q, k, v, causal, kv_len)
    dq, dk, dv = _bwd_qk(H, q, k, v, do, o, lse, causal, kv_len)
    f = W.bf16_bits_to_f64
    refs = oracle_mod.backward_qk(f(q), f(k), f(v), f(do), 0.125, kv_len=kv_len, causal=causal)
    for g, r, name in zip((dq, dk, dv), refs, ("dQ", "dK", "dV")):
        H.assert_grad(H.host_f64(g), r, name)
    if causal and Nq > Nk:   # rows i < Nq - Nk see no key
        assert torch.all(dq[:, :, :Nq - Nk].float() == 0)


def test_bwd_qk_square_equals_fa_bwd(H):
    """Nq == Nk: the same kernels with the same (top-left) causal rule, so dK
    and dV are bitwise those of fa_bwd; dQ, summed by reduce-adds in any
    order, agrees to fp32 rounding."""
    import workloads as W
    w = W.make("gpt2", B=1, H=2)
    x = H.Inputs(w)
    o, lse = H.run_fwd(x)
    a = H.run_bwd(x, o, lse)
    b = _bwd_qk(H, w.q, w.k, w.v, w.do, o, lse, True, scale=w.spec.scale)
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    assert torch.equal(a[2].view(torch.int16), b[2].view(torch.int16))
    assert H.rel_fro(H.host_f64(a[0]), H.host_f64(b[0])) <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_qk_long_keys_sampled(H, oracle_mod, d):
    """A 1000-query block at the end of 8192 keys (causal), checked on sampled
    query rows (dQ) and sampled keys (dK, dV)."""
    import workloads as W
    rng = np.random.default_rng(190 + d)
    B, Hh, Nq, Nk = 1, 2, 1000, 8192
    q, k, v, do = _qk_inputs(rng, B, Hh, Nq, Nk, d)
    o, lse = _qk(H, q, k, v, True)
    dq, dk, dv = _bwd_qk(H, q, k, v, do, o, lse, True)
    rows = np.sort(rng.choice(B * Hh * Nq, 96, replace=False)).astype(np.int64)
    keys = np.sort(rng.choice(B * Hh * Nk, 96, replace=False)).astype(np.int64)
    f = W.bf16_bits_to_f64
    dq_r, dk_r, dv_r = oracle_mod.backward_qk(f(q), f(k), f(v), f(do), 0.125, q_rows=rows,
                                              k_rows=keys, causal=True)
    H.assert_grad(H.host_f64(dq).reshape(-1, d)[rows], dq_r, "dQ")
    H.assert_grad(H.host_f64(dk).reshape(-1, d)[keys], dk_r, "dK")
    H.assert_grad(H.host_f64(dv).reshape(-1, d)[keys], dv_r, "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(300, 1), (1, 1), (129, 2)])
def test_bwd_qk_tiny_key_counts(H, oracle_mod, d, Nq, Nk):
    """One or two keys under bottom-right causal: only the last Nk query rows
    see any key; the others get dQ = 0.  The second batch has kv_len = 0: no
    key at all, every gradient of it is 0."""
    import workloads as W
    rng = np.random.default_rng(200 + Nq + Nk + d)
    B, Hh = 2, 2
    q, k, v, do = _qk_inputs(rng, B, Hh, Nq, Nk, d)
    kv_len = np.array([Nk, 0], np.int32)
    o, lse = _qk(H, q, k, v, True, kv_len)
    dq, dk, dv = _bwd_qk(H, q, k, v, do, o, lse, True, kv_len)
    f = W.bf16_bits_to_f64
    refs = oracle_mod.backward_qk(f(q), f(k), f(v), f(do), 0.125, kv_len=kv_len, causal=True)
    for g, r, name in zip((dq, dk, dv), refs, ("dQ", "dK", "dV")):
        H.assert_grad(H.host_f64(g)[0], r[0], name)
    if Nq > Nk:
        assert torch.all(dq[0, :, :Nq - Nk].float() == 0)
    for g in (dq, dk, dv):
        assert torch.all(g[1].float() == 0)
