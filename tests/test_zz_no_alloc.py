"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).  Checked through
the C ABI against fa_bwd with a caller-provided workspace, on two calls in a
row, within the parity tolerance the other GPU tests use.  Kept in a file
that pytest collects last."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _run(fa, W, H, use_noalloc, x, o, lse):
    shape = (x.B, x.H, x.N, x.d)
    dq, dk, dv = H.nan_like_bf16(shape), H.nan_like_bf16(shape), H.nan_like_bf16(shape)
    st = torch.cuda.current_stream()
    if use_noalloc:
        fa.fa_bwd_noalloc(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.B, x.H, x.N, x.d, x.scale,
                          x.causal, x.kv_len, x.mask, st)
    else:
        nbytes = fa.fa_bwd_workspace_size(x.B, x.H, x.N, x.d)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.B, x.H, x.N, x.d, x.scale,
                  x.causal, x.kv_len, x.mask, ws, nbytes, st)
    fa.fa_check(st)
    return dq, dk, dv


def test_noalloc_backward_matches_workspace_backward_twice(fa_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_25_gb300 as fa
    import gpu_harness as H
    import workloads as W
    # two different problems back to back: the second call must not see the
    # first call's scratch contents
    cases = [H.Inputs(W.make("bert")), H.Inputs(W.make("gpt2", B=2), )]
    for x in cases:
        o, lse = H.run_fwd(x)
        ref = _run(fa, W, H, False, x, o, lse)
        for _ in range(2):
            got = _run(fa, W, H, True, x, o, lse)
            for g, r, name in zip(got, ref, ("dQ", "dK", "dV")):
                H.assert_grad(H.host_f64(g), H.host_f64(r), name)
            # dK, dV use no atomics: identical to the workspace path bit for bit
            assert torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16))
            assert torch.equal(got[2].view(torch.int16), ref[2].view(torch.int16))


def test_noalloc_block_mask_matches_workspace_backward(fa_lib):
    """A block-sparse mask through the fixed scratch: the per-key-tile query
    lists the backward builds live in that array too.  A 4 x 4 mask with an
    empty key column (its dK, dV must be 0) and an empty query row."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_25_gb300 as fa
    import gpu_harness as H
    import workloads as W
    mask = np.array([[1, 0, 1, 0],
                     [0, 1, 1, 0],
                     [0, 0, 0, 0],
                     [1, 1, 0, 0]], np.uint8)
    x = H.Inputs(W.make("tiny", seed=97, B=2, H=3, N=512), block_mask=mask)
    o, lse = H.run_fwd(x)
    ref = _run(fa, W, H, False, x, o, lse)
    for _ in range(2):
        got = _run(fa, W, H, True, x, o, lse)
        H.assert_grad(H.host_f64(got[0]), H.host_f64(ref[0]), "dQ")
        assert torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(got[2].view(torch.int16), ref[2].view(torch.int16))
        # key tile 3 is attended by no query tile
        assert torch.all(got[1][:, :, 384:].float() == 0) and torch.all(got[2][:, :, 384:].float() == 0)


def test_noalloc_rejects_problems_beyond_its_scratch(fa_lib):
    import exact_io_aware_25_gb300 as fa
    limit = fa.fa_bwd_noalloc_max_scratch_bytes()
    assert limit == 64 << 20
    # B=1 H=8 N=65536 needs 8 * 65536 * 264 bytes > 64 MiB; rejected before any launch
    assert fa.fa_bwd_workspace_size(1, 8, 65536, 64) > limit
    with pytest.raises(fa.FaError) as ei:
        fa.fa_bwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 8, 65536, 64, 0.125)
    assert ei.value.status == fa.FA_ERR_WORKSPACE


def test_noalloc_backward_at_d128(fa_lib, oracle_mod):
    """The d = 128 backward through the fixed scratch, against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_25_gb300 as fa
    import gpu_harness as H
    import workloads as W
    x = H.Inputs(W.make("tiny", seed=96, d=128, B=2, H=2, N=500, causal=True))
    o, lse = H.run_fwd(x)
    shape = (x.B, x.H, x.N, 128)
    dq, dk, dv = (H.nan_like_bf16(shape) for _ in range(3))
    st = torch.cuda.current_stream()
    fa.fa_bwd_noalloc(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.B, x.H, x.N, 128, x.scale,
                      x.causal, None, None, st)
    fa.fa_check(st)
    q, k, v, do = x.f64("q"), x.f64("k"), x.f64("v"), x.f64("do")
    refs = oracle_mod.backward(q, k, v, do, x.scale, **x.oracle_kwargs())
    for g, r, name in zip((dq, dk, dv), refs, ("dQ", "dK", "dV")):
        H.assert_grad(H.host_f64(g), r, name)
