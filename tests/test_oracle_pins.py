"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test pins the oracle to something other than itself: a closed form
derived by hand (tests/golden/closed_form.json), an invariant of softmax
attention, the pages' own streaming algorithm under every block split,
a special case, or central finite differences.  A plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, log2
instead of ln, an off-by-one causal mask) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def _rand(rng, B, H, N, d, scale=1.0):
    return rng.standard_normal((B, H, N, d)) * scale


def _mask_for(rng, N, blk, density=0.5):
    nb = -(-N // blk)
    m = (rng.random((nb, nb)) < density).astype(np.uint8)
    np.fill_diagonal(m, 1)
    return m


VARIANTS = [
    dict(),
    dict(causal=True),
    dict(kv_len=True),
    dict(mask=True),
    dict(causal=True, kv_len=True, mask=True),
]


def _variant_args(rng, B, N, blk, v):
    kw = {"causal": v.get("causal", False)}
    if v.get("kv_len"):
        kw["kv_len"] = rng.integers(1, N + 1, size=B).astype(np.int32)
    if v.get("mask"):
        kw["block_mask"] = _mask_for(rng, N, blk)
        kw["block"] = blk
    return kw


def _allowed_np(B, N, causal=False, kv_len=None, block_mask=None, block=128):
    """Boolean [B, N, N] allowed set, written from the mask definitions."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    out = np.ones((B, N, N), bool)
    if causal:
        out &= (j <= i)[None]
    if kv_len is not None:
        out &= (j[None] < np.minimum(np.asarray(kv_len), N)[:, None, None])
    if block_mask is not None:
        out &= block_mask[(i // block), (j // block)].astype(bool)[None]
    return out


def _evalnum(x):
    if isinstance(x, str):
        if x == "-inf":
            return -math.inf
        if "+" in x:
            return sum(_evalnum(t) for t in x.split("+"))
        if "*" in x:
            a, b = x.split("*")
            return float(a) * _evalnum(b)
        assert x.startswith("ln")
        return math.log(float(x[2:]))
    return float(x)


def _arr(nested):
    return np.array([[_evalnum(e) for e in row] for row in nested], np.float64)


# ---------------------------------------------------------------- golden


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_closed_form_golden(oracle_mod, case):
    B, H, N, d = case["B"], case["H"], case["N"], case["d"]
    q = _arr(case["q"]).reshape(B, H, N, d)
    k = _arr(case["k"]).reshape(B, H, N, d)
    v = _arr(case["v"]).reshape(B, H, N, d)
    do = _arr(case["do"]).reshape(B, H, N, d)
    kv_len = None if case["kv_len"] is None else np.array(case["kv_len"], np.int32)
    o, lse = oracle_mod.forward(q, k, v, case["scale"], causal=case["causal"], kv_len=kv_len)
    np.testing.assert_allclose(o.reshape(N, d), _arr(case["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(N), [_evalnum(x) for x in case["lse"]], rtol=0,
                               atol=1e-12)
    dq, dk, dv = oracle_mod.backward(q, k, v, do, case["scale"], causal=case["causal"],
                                     kv_len=kv_len)
    np.testing.assert_allclose(dq.reshape(N, d), _arr(case["dq"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.reshape(N, d), _arr(case["dk"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.reshape(N, d), _arr(case["dv"]), rtol=0, atol=1e-12)


GOLDEN_QK = os.path.join(os.path.dirname(GOLDEN), "closed_form_qk.json")


@pytest.mark.parametrize("case", json.load(open(GOLDEN_QK))["cases"], ids=lambda c: c["name"])
def test_closed_form_golden_short_queries(oracle_mod, case):
    """Nq != Nk with bottom-right causal: forward_qk and backward_qk against
    hand-derived values (tests/golden/closed_form_qk.json)."""
    B, H, Nq, Nk, d = case["B"], case["H"], case["Nq"], case["Nk"], case["d"]
    q = _arr(case["q"]).reshape(B, H, Nq, d)
    k = _arr(case["k"]).reshape(B, H, Nk, d)
    v = _arr(case["v"]).reshape(B, H, Nk, d)
    do = _arr(case["do"]).reshape(B, H, Nq, d)
    o, lse = oracle_mod.forward_qk(q, k, v, case["scale"], causal=True)
    np.testing.assert_allclose(o.reshape(Nq, d), _arr(case["o"]), rtol=0, atol=1e-12)
    want = np.array([_evalnum(x) for x in case["lse"]])
    got = lse.reshape(Nq)
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    fin = np.isfinite(want)
    np.testing.assert_allclose(got[fin], want[fin], rtol=0, atol=1e-12)
    dq, dk, dv = oracle_mod.backward_qk(q, k, v, do, case["scale"], causal=True)
    np.testing.assert_allclose(dq.reshape(Nq, d), _arr(case["dq"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.reshape(Nk, d), _arr(case["dk"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.reshape(Nk, d), _arr(case["dv"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- invariants


@pytest.mark.parametrize("v", VARIANTS, ids=str)
def test_probability_rows_sum_to_one_and_masked_are_zero(oracle_mod, v):
    rng = np.random.default_rng(11)
    B, H, N, d, blk = 2, 2, 23, 5, 4
    q, k = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    kw = _variant_args(rng, B, N, blk, v)
    allowed = _allowed_np(B, N, kw["causal"], kw.get("kv_len"), kw.get("block_mask"), blk)
    for bh in range(B * H):
        P = oracle_mod.probs(q, k, 0.7, bh=bh, **kw)
        al = allowed[bh // H]
        assert np.all(P[~al] == 0.0)
        assert np.all(P[al] > 0.0)
        rows = al.any(axis=1)
        np.testing.assert_allclose(P[rows].sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(P[~rows] == 0.0)


@pytest.mark.parametrize("v", VARIANTS, ids=str)
def test_constant_values_give_that_constant(oracle_mod, v):
    rng = np.random.default_rng(12)
    B, H, N, d, blk = 2, 3, 19, 4, 4
    q, k = _rand(rng, B, H, N, d, 2.0), _rand(rng, B, H, N, d, 2.0)
    c = rng.standard_normal(d)
    vv = np.broadcast_to(c, (B, H, N, d)).copy()
    kw = _variant_args(rng, B, N, blk, v)
    o, lse = oracle_mod.forward(q, k, vv, 0.3, **kw)
    allowed = _allowed_np(B, N, kw["causal"], kw.get("kv_len"), kw.get("block_mask"), blk)
    for b in range(B):
        rows = allowed[b].any(axis=1)
        np.testing.assert_allclose(o[b][:, rows], np.broadcast_to(c, o[b][:, rows].shape),
                                   rtol=0, atol=1e-13)
        assert np.all(o[b][:, ~rows] == 0.0)
        assert np.all(np.isneginf(lse[b][:, ~rows]))


@pytest.mark.parametrize("v", VARIANTS, ids=str)
def test_every_block_split_of_the_streaming_forward_equals_one_shot(oracle_mod, v):
    """The explainer's running (m, l) merge and O update, steps 1-4, give the
    one-shot softmax for every block size (query and key/value)."""
    rng = np.random.default_rng(13)
    B, H, N, d, blk = 1, 2, 9, 3, 3
    q, k, vv = (_rand(rng, B, H, N, d, 1.5) for _ in range(3))
    kw = _variant_args(rng, B, N, blk, v)
    o_ref, lse_ref = oracle_mod.forward(q, k, vv, 0.9, **kw)
    for Br in range(1, N + 1):
        for Bc in range(1, N + 1):
            o, lse = oracle_mod.forward_tiled(q, k, vv, 0.9, Br, Bc, **kw)
            np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("v", VARIANTS, ids=str)
def test_zero_queries_average_the_allowed_values(oracle_mod, v):
    """Q = 0 makes every score 0: o_i is the mean of v over A_i, lse_i = ln |A_i|."""
    rng = np.random.default_rng(14)
    B, H, N, d, blk = 2, 2, 21, 3, 4
    q = np.zeros((B, H, N, d))
    k, vv = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    kw = _variant_args(rng, B, N, blk, v)
    o, lse = oracle_mod.forward(q, k, vv, 1.3, **kw)
    allowed = _allowed_np(B, N, kw["causal"], kw.get("kv_len"), kw.get("block_mask"), blk)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                a = np.flatnonzero(allowed[b, i])
                if len(a) == 0:
                    continue
                np.testing.assert_allclose(o[b, h, i], vv[b, h, a].mean(axis=0), rtol=0,
                                           atol=1e-13)
                assert abs(lse[b, h, i] - math.log(len(a))) < 1e-13


def test_single_allowed_key_returns_its_value(oracle_mod):
    """Causal row 0 attends only to key 0 (top-left aligned mask)."""
    rng = np.random.default_rng(15)
    B, H, N, d = 1, 3, 17, 6
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    o, lse = oracle_mod.forward(q, k, vv, 0.4, causal=True)
    np.testing.assert_allclose(o[:, :, 0], vv[:, :, 0], rtol=0, atol=1e-15)
    s00 = 0.4 * np.einsum("bhc,bhc->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-14)
    # row 1 attends exactly to keys {0, 1}: two-way softmax
    s = 0.4 * np.einsum("bhc,bhjc->bhj", q[:, :, 1], k[:, :, :2])
    w = np.exp(s - s.max(-1, keepdims=True))
    w /= w.sum(-1, keepdims=True)
    np.testing.assert_allclose(o[:, :, 1], np.einsum("bhj,bhjc->bhc", w, vv[:, :, :2]),
                               rtol=0, atol=1e-14)


@pytest.mark.parametrize("v", VARIANTS, ids=str)
def test_key_shift_moves_lse_by_scaled_query_dot(oracle_mod, v):
    """K + 1 c^T adds scale*<q_i, c> to every score of row i: O unchanged,
    lse_i shifted by exactly that amount (pins where the scale is applied)."""
    rng = np.random.default_rng(16)
    B, H, N, d, blk = 2, 2, 15, 4, 4
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    c = rng.standard_normal(d)
    kw = _variant_args(rng, B, N, blk, v)
    o1, l1 = oracle_mod.forward(q, k, vv, 0.6, **kw)
    o2, l2 = oracle_mod.forward(q, k + c, vv, 0.6, **kw)
    fin = np.isfinite(l1)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    shift = 0.6 * np.einsum("bhic,c->bhi", q, c)
    np.testing.assert_allclose((l2 - l1)[fin], shift[fin], rtol=0, atol=1e-12)


def test_joint_key_value_permutation_leaves_output_unchanged(oracle_mod):
    rng = np.random.default_rng(17)
    B, H, N, d = 2, 2, 25, 5
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    perm = rng.permutation(N)
    o1, l1 = oracle_mod.forward(q, k, vv, 0.5)
    o2, l2 = oracle_mod.forward(q, k[:, :, perm], vv[:, :, perm], 0.5)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


def test_all_ones_block_mask_equals_no_mask(oracle_mod):
    rng = np.random.default_rng(18)
    B, H, N, d, blk = 1, 2, 30, 4, 8
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    ones = np.ones((4, 4), np.uint8)
    o1, l1 = oracle_mod.forward(q, k, vv, 0.5, causal=True)
    o2, l2 = oracle_mod.forward(q, k, vv, 0.5, causal=True, block_mask=ones, block=blk)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    g1 = oracle_mod.backward(q, k, vv, do, 0.5, causal=True)
    g2 = oracle_mod.backward(q, k, vv, do, 0.5, causal=True, block_mask=ones, block=blk)
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)


def test_masked_blocks_and_padded_keys_contribute_nothing(oracle_mod):
    """Values in masked-out blocks or past kv_len never reach O, lse, dQ; the
    gradients of keys no query attends to are exactly zero."""
    rng = np.random.default_rng(19)
    B, H, N, d, blk = 2, 2, 24, 4, 8
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    mask = np.array([[1, 0, 1], [0, 1, 0], [1, 0, 0]], np.uint8)
    kv_len = np.array([20, 13], np.int32)
    kw = dict(block_mask=mask, block=blk, kv_len=kv_len)
    allowed = _allowed_np(B, N, False, kv_len, mask, blk)
    k2, v2 = k.copy(), vv.copy()
    for b in range(B):
        dead = ~allowed[b].any(axis=0)   # keys no query row attends to
        k2[b, :, dead] += 100.0
        v2[b, :, dead] -= 50.0
    o1, l1 = oracle_mod.forward(q, k, vv, 0.5, **kw)
    o2, l2 = oracle_mod.forward(q, k2, v2, 0.5, **kw)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    dq, dk, dv = oracle_mod.backward(q, k, vv, do, 0.5, **kw)
    for b in range(B):
        dead = ~allowed[b].any(axis=0)
        assert np.all(dk[b][:, dead] == 0.0) and np.all(dv[b][:, dead] == 0.0)
        empty = ~allowed[b].any(axis=1)
        assert np.all(dq[b][:, empty] == 0.0)


# ---------------------------------------------------------------- backward


@pytest.mark.parametrize("v", VARIANTS, ids=str)
def test_backward_matches_central_finite_differences(oracle_mod, v):
    """dQ, dK, dV of L = sum(dO o O) against central differences of the forward."""
    rng = np.random.default_rng(20)
    B, H, N, d, blk, scale, h = 2, 1, 9, 3, 4, 0.8, 1e-6
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    kw = _variant_args(rng, B, N, blk, v)

    def loss(q_, k_, v_):
        o, _ = oracle_mod.forward(q_, k_, v_, scale, **kw)
        return float(np.sum(do * o))

    dq, dk, dv = oracle_mod.backward(q, k, vv, do, scale, **kw)
    for which, grad in (("q", dq), ("k", dk), ("v", dv)):
        num = np.zeros_like(grad)
        base = {"q": q, "k": k, "v": vv}
        for idx in np.ndindex(*grad.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[which][idx] += h
            minus[which][idx] -= h
            num[idx] = (loss(plus["q"], plus["k"], plus["v"])
                        - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert err < 1e-6, (which, err)


def test_row_selection_matches_full_results(oracle_mod):
    rng = np.random.default_rng(21)
    B, H, N, d, blk = 2, 2, 20, 4, 8
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    kw = dict(causal=True, kv_len=np.array([17, 9], np.int32),
              block_mask=np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]], np.uint8), block=blk)
    o, lse = oracle_mod.forward(q, k, vv, 0.5, **kw)
    dq, dk, dv = oracle_mod.backward(q, k, vv, do, 0.5, **kw)
    rows = np.array([0, 5, 19, 20 + 3, 40 + 11, 79], np.int64)
    o_r, l_r = oracle_mod.forward(q, k, vv, 0.5, rows=rows, **kw)
    np.testing.assert_array_equal(o_r, o.reshape(-1, d)[rows])
    np.testing.assert_array_equal(l_r, lse.reshape(-1)[rows])
    keys = np.array([1, 8, 16, 33, 61, 70], np.int64)
    dq_r, dk_r, dv_r = oracle_mod.backward(q, k, vv, do, 0.5, q_rows=rows, k_rows=keys, **kw)
    np.testing.assert_array_equal(dq_r, dq.reshape(-1, d)[rows])
    np.testing.assert_array_equal(dk_r, dk.reshape(-1, d)[keys])
    np.testing.assert_array_equal(dv_r, dv.reshape(-1, d)[keys])


def test_cross_check_with_numpy_definition(oracle_mod):
    """Independent numpy restatement (matrix form) on tiny masked cases."""
    rng = np.random.default_rng(22)
    B, H, N, d, blk, scale = 2, 2, 13, 4, 4, 0.7
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    kv_len = np.array([13, 6], np.int32)
    mask = np.array([[1, 1, 0, 1], [0, 1, 1, 0], [1, 0, 1, 1], [1, 1, 1, 1]], np.uint8)
    allowed = _allowed_np(B, N, True, kv_len, mask, blk)
    o, lse = oracle_mod.forward(q, k, vv, scale, causal=True, kv_len=kv_len, block_mask=mask,
                                block=blk)
    dq, dk, dv = oracle_mod.backward(q, k, vv, do, scale, causal=True, kv_len=kv_len,
                                     block_mask=mask, block=blk)
    for b in range(B):
        for h in range(H):
            S = scale * q[b, h] @ k[b, h].T
            S = np.where(allowed[b], S, -np.inf)
            rows = allowed[b].any(1)
            m = np.where(rows, S.max(1), 0.0)
            E = np.exp(S - m[:, None])
            P = E / np.where(rows, E.sum(1), 1.0)[:, None]
            O = P @ vv[b, h]
            np.testing.assert_allclose(o[b, h], O, rtol=0, atol=1e-12)
            L = np.where(rows, m + np.log(np.where(rows, E.sum(1), 1.0)), -np.inf)
            np.testing.assert_allclose(lse[b, h], L, rtol=0, atol=1e-12)
            dV = P.T @ do[b, h]
            dP = do[b, h] @ vv[b, h].T
            Dv = (do[b, h] * O).sum(1)
            dS = P * (dP - Dv[:, None])
            np.testing.assert_allclose(dv[b, h], dV, rtol=0, atol=1e-12)
            np.testing.assert_allclose(dq[b, h], scale * dS @ k[b, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(dk[b, h], scale * dS.T @ q[b, h], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- dropout
#
# Dropout is fused into the kernels ([EXPL] "Key ideas", kernel fusion); the
# keep mask comes from a counter-based hash both sides implement from its
# published definition.  These pins tie the oracle's dropout to the
# definition O = (P o Z) V / (1 - p') through paths that do not use it.


def test_dropout_with_zero_threshold_is_the_plain_definition(oracle_mod):
    rng = np.random.default_rng(30)
    B, H, N, d = 2, 2, 19, 4
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    o1, l1 = oracle_mod.forward(q, k, vv, 0.7, causal=True)
    o2, l2 = oracle_mod.forward(q, k, vv, 0.7, causal=True, p8=0, seed=1234)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    g1 = oracle_mod.backward(q, k, vv, do, 0.7, causal=True)
    g2 = oracle_mod.backward(q, k, vv, do, 0.7, causal=True, p8=0, seed=99)
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)


def _keep_grid(oracle_mod, seed, p8, bh, n):
    return np.array([[oracle_mod.keep(seed, p8, bh, i, j) for j in range(n)] for i in range(n)])


@pytest.mark.parametrize("p8", [26, 128, 230])
def test_dropout_keep_rate_and_nested_thresholds(oracle_mod, p8):
    """The kept fraction is 1 - p8/256 within 5 binomial sigmas, and a higher
    threshold keeps a subset of what a lower one keeps (keep iff byte >= p8)."""
    n = 96
    z = np.concatenate([_keep_grid(oracle_mod, 7, p8, bh, n).ravel() for bh in (0, 5)])
    p_keep = 1 - p8 / 256
    sigma = math.sqrt(p_keep * (1 - p_keep) / z.size)
    assert abs(z.mean() - p_keep) < 5 * sigma
    z_hi = _keep_grid(oracle_mod, 7, min(p8 + 20, 255), 0, n)
    assert np.all(z_hi <= _keep_grid(oracle_mod, 7, p8, 0, n))


def test_dropout_bytes_are_uniform_and_depend_on_seed_and_head(oracle_mod):
    """Recover each element's byte (the largest threshold that still keeps it)
    and check it is uniform over 0..255 (chi-square, 255 degrees of freedom);
    other seeds and heads give different masks."""
    n = 48

    def byte(seed, bh, i, j):
        lo, hi = 0, 255                      # keep(0) always holds
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if oracle_mod.keep(seed, mid, bh, i, j):
                lo = mid
            else:
                hi = mid - 1
        return lo

    u = np.array([byte(3, bh, i, j) for bh in (0, 1) for i in range(n) for j in range(n)])
    counts = np.bincount(u, minlength=256)
    expected = u.size / 256
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)
    a = _keep_grid(oracle_mod, 3, 128, 0, n)
    assert (a != _keep_grid(oracle_mod, 4, 128, 0, n)).mean() > 0.3
    assert (a != _keep_grid(oracle_mod, 3, 128, 1, n)).mean() > 0.3
    assert (a != _keep_grid(oracle_mod, 3 + (1 << 32), 128, 0, n)).mean() > 0.3


def test_dropout_forward_equals_masked_probabilities_times_values(oracle_mod):
    """o_i = sum_j P_ij Z_ij v_j * 256/(256-p8) with P from the plain
    probabilities and Z from the keep mask, for every mask variant."""
    rng = np.random.default_rng(31)
    B, H, N, d, blk, scale, p8, seed = 2, 2, 21, 5, 4, 0.9, 77, 2024
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    kw = _variant_args(rng, B, N, blk, dict(causal=True, kv_len=True, mask=True))
    o, lse = oracle_mod.forward(q, k, vv, scale, p8=p8, seed=seed, **kw)
    _, lse0 = oracle_mod.forward(q, k, vv, scale, **kw)
    np.testing.assert_array_equal(lse, lse0)          # lse is taken before dropout
    for b in range(B):
        for h in range(H):
            bh = b * H + h
            P = oracle_mod.probs(q, k, scale, bh=bh, **kw)
            Z = _keep_grid(oracle_mod, seed, p8, bh, N)
            want = (P * Z) @ vv[b, h] * (256.0 / (256 - p8))
            np.testing.assert_allclose(o[b, h], want, rtol=0, atol=1e-12)


def test_dropout_backward_matches_central_finite_differences(oracle_mod):
    """With the keep mask fixed, the dropout forward is smooth in q, k, v:
    its dQ, dK, dV against central differences of sum(dO o O)."""
    rng = np.random.default_rng(32)
    B, H, N, d, blk, scale, h, p8, seed = 1, 2, 10, 3, 4, 0.8, 1e-6, 90, 5
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    kw = _variant_args(rng, B, N, blk, dict(causal=True, kv_len=True))

    def loss(q_, k_, v_):
        o, _ = oracle_mod.forward(q_, k_, v_, scale, p8=p8, seed=seed, **kw)
        return float(np.sum(do * o))

    dq, dk, dv = oracle_mod.backward(q, k, vv, do, scale, p8=p8, seed=seed, **kw)
    for which, grad in (("q", dq), ("k", dk), ("v", dv)):
        num = np.zeros_like(grad)
        base = {"q": q, "k": k, "v": vv}
        for idx in np.ndindex(*grad.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[which][idx] += h
            minus[which][idx] -= h
            num[idx] = (loss(plus["q"], plus["k"], plus["v"])
                        - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert err < 1e-6, (which, err)


def test_dropout_output_is_unbiased_over_seeds(oracle_mod):
    """The keep scale makes the dropped-out output an unbiased estimate of the
    plain one: the mean over 400 seeds is within a few standard errors."""
    rng = np.random.default_rng(33)
    B, H, N, d, scale, p8 = 1, 1, 12, 4, 0.5, 64
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    o0, _ = oracle_mod.forward(q, k, vv, scale)
    runs = np.stack([oracle_mod.forward(q, k, vv, scale, p8=p8, seed=s)[0] for s in range(400)])
    se = runs.std(axis=0) / math.sqrt(runs.shape[0])
    z = np.abs(runs.mean(axis=0) - o0) / np.maximum(se, 1e-12)
    assert np.mean(z < 4) > 0.98 and np.max(z) < 6


def test_dropout_threshold_rounding(oracle_mod):
    assert oracle_mod.drop_p8(0.0) == 0
    assert oracle_mod.drop_p8(0.1) == 26          # 25.6 -> 26
    assert oracle_mod.drop_p8(0.5) == 128
    assert oracle_mod.drop_p8(0.998) == 255       # 255.49 -> 255
    assert oracle_mod.drop_p8(0.9999) == 255      # 255.97 rounds to 256, capped
    assert oracle_mod.drop_p8(1.5 / 256) == 2     # tie 1.5 -> even
    assert oracle_mod.drop_p8(2.5 / 256) == 2     # tie 2.5 -> even


# ---------------------------------------------------------------- Nq != Nk (split-KV forward)


def test_short_queries_equal_the_same_rows_of_a_square_problem(oracle_mod):
    """Query rows are independent: the rows of a short Q against Nk keys equal
    the same rows of the square problem whose Q is extended to Nk rows."""
    rng = np.random.default_rng(40)
    B, H, Nq, Nk, d, scale = 2, 3, 5, 37, 6, 0.6
    q = _rand(rng, B, H, Nq, d)
    k, vv = _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nk, d)
    kv_len = np.array([37, 11], np.int32)
    o, lse = oracle_mod.forward_qk(q, k, vv, scale, kv_len=kv_len)
    q_sq = np.concatenate([q, _rand(rng, B, H, Nk - Nq, d)], axis=2)
    o_sq, lse_sq = oracle_mod.forward(q_sq, k, vv, scale, kv_len=kv_len)
    np.testing.assert_array_equal(o, o_sq[:, :, :Nq])
    np.testing.assert_array_equal(lse, lse_sq[:, :, :Nq])


def test_short_queries_special_cases(oracle_mod):
    rng = np.random.default_rng(41)
    B, H, Nq, Nk, d = 1, 2, 3, 50, 4
    q = _rand(rng, B, H, Nq, d)
    k = _rand(rng, B, H, Nk, d)
    c = np.array([0.5, -1.0, 2.0, 0.25])
    o, lse = oracle_mod.forward_qk(q, k, np.broadcast_to(c, (B, H, Nk, d)), 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-14)
    # one key: the output is its value and lse its score
    vv = _rand(rng, B, H, Nk, d)
    o1, l1 = oracle_mod.forward_qk(q, k, vv, 0.3, kv_len=np.array([1], np.int32))
    np.testing.assert_allclose(o1, np.broadcast_to(vv[:, :, :1], o1.shape), rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, 0.3 * np.einsum("bhic,bhc->bhi", q, k[:, :, 0]), rtol=0,
                               atol=1e-13)
    # zero queries: the mean of the values and lse = ln Nk
    o0, l0 = oracle_mod.forward_qk(np.zeros_like(q), k, vv, 0.3)
    np.testing.assert_allclose(o0, np.broadcast_to(vv.mean(axis=2, keepdims=True), o0.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(l0, np.log(Nk), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- Nq != Nk with a causal mask


def test_bottom_right_causal_square_case_is_the_top_left_rule(oracle_mod):
    """Nq == Nk: the bottom-right alignment (j <= i + Nk - Nq) is j <= i,
    the causal rule of the square forward."""
    rng = np.random.default_rng(50)
    B, H, N, d = 2, 2, 19, 5
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    kv_len = np.array([19, 7], np.int32)
    o, lse = oracle_mod.forward_qk(q, k, vv, 0.4, kv_len=kv_len, causal=True)
    o2, lse2 = oracle_mod.forward(q, k, vv, 0.4, causal=True, kv_len=kv_len)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


@pytest.mark.parametrize("Nq,Nk", [(1, 9), (4, 9), (9, 9), (12, 9)])
def test_bottom_right_causal_closed_form(oracle_mod, Nq, Nk):
    """Q = 0: every allowed key has score 0, so o_i is the mean of v_j over
    j <= i + Nk - Nq and lse_i = ln(i + Nk - Nq + 1); rows with no key
    (i < Nq - Nk) get o = 0 and lse = -inf.  The last query sees all keys."""
    rng = np.random.default_rng(51)
    B, H, d = 1, 2, 3
    k, vv = _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nk, d)
    o, lse = oracle_mod.forward_qk(np.zeros((B, H, Nq, d)), k, vv, 0.7, causal=True)
    for i in range(Nq):
        n_allowed = min(Nk, max(0, i + Nk - Nq + 1))
        if n_allowed == 0:
            assert np.all(o[:, :, i] == 0) and np.all(np.isneginf(lse[:, :, i]))
            continue
        np.testing.assert_allclose(o[:, :, i], vv[:, :, :n_allowed].mean(axis=2), rtol=0,
                                   atol=1e-14)
        np.testing.assert_allclose(lse[:, :, i], math.log(n_allowed), rtol=0, atol=1e-14)


def test_bottom_right_causal_against_numpy_softmax(oracle_mod):
    """Brute force with numpy on a tiny case: the mask j <= i + Nk - Nq
    written out, softmax and product by V."""
    rng = np.random.default_rng(52)
    B, H, Nq, Nk, d, scale = 1, 2, 6, 11, 4, 0.5
    q, k, vv = _rand(rng, B, H, Nq, d), _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nk, d)
    o, lse = oracle_mod.forward_qk(q, k, vv, scale, causal=True)
    s = scale * np.einsum("bhic,bhjc->bhij", q, k)
    allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    s = np.where(allowed, s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    e = np.exp(s - mx)
    np.testing.assert_allclose(o, np.einsum("bhij,bhjc->bhic", e / e.sum(-1, keepdims=True), vv),
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, (mx + np.log(e.sum(-1, keepdims=True)))[..., 0], rtol=1e-12,
                               atol=1e-13)


# ---------------------------------------------------------------- Nq != Nk backward


def test_short_query_backward_square_case_is_the_square_backward(oracle_mod):
    """Nq == Nk: backward_qk is the square backward (bottom-right causal is
    then the top-left rule)."""
    rng = np.random.default_rng(53)
    B, H, N, d = 2, 2, 13, 4
    q, k, vv, do = (_rand(rng, B, H, N, d) for _ in range(4))
    kv_len = np.array([13, 6], np.int32)
    for causal in (False, True):
        a = oracle_mod.backward_qk(q, k, vv, do, 0.6, kv_len=kv_len, causal=causal)
        b = oracle_mod.backward(q, k, vv, do, 0.6, kv_len=kv_len, causal=causal)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("Nq,Nk,causal", [(3, 8, True), (8, 5, True), (4, 7, False)])
def test_short_query_backward_matches_central_finite_differences(oracle_mod, Nq, Nk, causal):
    """dQ, dK, dV of L = sum(dO o O) for the Nq x Nk forward, against
    central differences of forward_qk (with key padding; with Nq > Nk the
    first Nq - Nk causal rows have no key and give nothing)."""
    rng = np.random.default_rng(54 + Nq)
    B, H, d, scale, h = 2, 1, 3, 0.7, 1e-6
    q, do = _rand(rng, B, H, Nq, d), _rand(rng, B, H, Nq, d)
    k, vv = _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nk, d)
    kv_len = np.array([Nk, Nk - 2], np.int32)

    def loss(q_, k_, v_):
        o, _ = oracle_mod.forward_qk(q_, k_, v_, scale, kv_len=kv_len, causal=causal)
        return float(np.sum(do * o))

    grads = oracle_mod.backward_qk(q, k, vv, do, scale, kv_len=kv_len, causal=causal)
    base = {"q": q, "k": k, "v": vv}
    for which, grad in zip(("q", "k", "v"), grads):
        assert grad.shape == base[which].shape
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[which][idx] += h
            minus[which][idx] -= h
            num[idx] = (loss(plus["q"], plus["k"], plus["v"])
                        - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert err < 1e-6, (which, err)


def test_short_query_backward_closed_form_at_zero_queries(oracle_mod):
    """Q = 0 under bottom-right causal: P_ij = 1/n_i on the n_i = i + Nk - Nq + 1
    allowed keys, so dV_j = sum over rows i that see j of dO_i / n_i, and
    dK = scale * dS^T Q = 0."""
    rng = np.random.default_rng(57)
    B, H, Nq, Nk, d = 1, 2, 4, 9, 3
    k, vv, do = _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nq, d)
    _, dk, dv = oracle_mod.backward_qk(np.zeros((B, H, Nq, d)), k, vv, do, 0.9, causal=True)
    want = np.zeros_like(dv)
    for i in range(Nq):
        n = i + Nk - Nq + 1
        want[:, :, :n] += do[:, :, i:i + 1] / n
    np.testing.assert_allclose(dv, want, rtol=0, atol=1e-14)
    assert np.all(dk == 0.0)


def test_short_query_backward_row_selection(oracle_mod):
    rng = np.random.default_rng(58)
    B, H, Nq, Nk, d = 2, 2, 5, 17, 3
    q, do = _rand(rng, B, H, Nq, d), _rand(rng, B, H, Nq, d)
    k, vv = _rand(rng, B, H, Nk, d), _rand(rng, B, H, Nk, d)
    kw = dict(kv_len=np.array([17, 10], np.int32), causal=True)
    dq, dk, dv = oracle_mod.backward_qk(q, k, vv, do, 0.5, **kw)
    rows = np.array([0, 4, 7, 19], np.int64)
    keys = np.array([0, 16, 20, 50, 67], np.int64)
    dq_r, dk_r, dv_r = oracle_mod.backward_qk(q, k, vv, do, 0.5, q_rows=rows, k_rows=keys, **kw)
    np.testing.assert_array_equal(dq_r, dq.reshape(-1, d)[rows])
    np.testing.assert_array_equal(dk_r, dk.reshape(-1, d)[keys])
    np.testing.assert_array_equal(dv_r, dv.reshape(-1, d)[keys])


# ---------------------------------------------------------------- row statistics (m, l)


@pytest.mark.parametrize("v", VARIANTS)
def test_row_statistics_against_numpy(oracle_mod, v):
    """m_i = max over the allowed keys of s_ij and l_i = sum exp(s_ij - m_i),
    recomputed with numpy from a mask written out here; the forward's o and
    lse are unchanged by asking for them."""
    rng = np.random.default_rng(60)
    B, H, N, d, scale, blk = 2, 2, 23, 4, 0.45, 8
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    causal = v.get("causal", False)
    kv_len = np.array([23, 9], np.int32) if v.get("kv_len") else None
    mask = _mask_for(rng, N, blk) if v.get("mask") else None
    o, lse, m, l = oracle_mod.forward_stats(q, k, vv, scale, causal=causal, kv_len=kv_len,
                                            block_mask=mask, block=blk)
    o2, lse2 = oracle_mod.forward(q, k, vv, scale, causal=causal, kv_len=kv_len,
                                  block_mask=mask, block=blk)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    s = scale * np.einsum("bhic,bhjc->bhij", q, k)
    i, j = np.arange(N)[:, None], np.arange(N)[None, :]
    for b in range(B):
        allowed = np.ones((N, N), bool)
        if causal:
            allowed &= j <= i
        if kv_len is not None:
            allowed &= j < kv_len[b]
        if mask is not None:
            allowed &= mask[i // blk, j // blk] != 0
        sb = np.where(allowed, s[b], -np.inf)
        m_ref = sb.max(axis=-1)
        for h in range(H):
            for r in range(N):
                if not np.isfinite(m_ref[h, r]):
                    assert np.isneginf(m[b, h, r]) and l[b, h, r] == 0
                    continue
                # same scores up to the summation order of the dot products
                np.testing.assert_allclose(m[b, h, r], m_ref[h, r], rtol=1e-14, atol=1e-15)
                np.testing.assert_allclose(l[b, h, r], np.exp(sb[h, r] - m_ref[h, r]).sum(),
                                           rtol=1e-12)
    fin = np.isfinite(m)
    np.testing.assert_allclose(lse[fin], m[fin] + np.log(l[fin]), rtol=0, atol=1e-13)


def test_row_statistics_special_cases(oracle_mod):
    """Causal row 0 has one key: m = s_00, l = 1.  Q = 0: m = 0, l = |A_i|."""
    rng = np.random.default_rng(61)
    B, H, N, d = 1, 1, 10, 3
    q, k, vv = (_rand(rng, B, H, N, d) for _ in range(3))
    _, _, m, l = oracle_mod.forward_stats(q, k, vv, 0.8, causal=True)
    assert math.isclose(m[0, 0, 0], 0.8 * float(q[0, 0, 0] @ k[0, 0, 0]), rel_tol=1e-14)
    assert l[0, 0, 0] == 1.0
    _, _, m0, l0 = oracle_mod.forward_stats(np.zeros_like(q), k, vv, 0.8, causal=True)
    assert np.all(m0 == 0)
    np.testing.assert_array_equal(l0[0, 0], np.arange(1, N + 1))
