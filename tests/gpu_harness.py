"""Helpers shared by the GPU parity tests: device upload of the seeded bf16
inputs, calls through the C ABI (via the thin binding), and the comparison
metrics with the tolerances the parity bar states."""
from __future__ import annotations

import numpy as np
import torch

import exact_io_aware_25_gb300 as fa
import workloads as W

# Tolerances (floating point; the GPU computes in bf16 with fp32 accumulation,
# the oracle in fp64 on the same bf16-rounded inputs).
TOL_O_MAXABS = 2e-2
TOL_O_RELFRO = 5e-3
TOL_LSE_MAXABS = 1e-3
TOL_GRAD_RELFRO = 1e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    bits = t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return W.bf16_bits_to_f64(bits)


def nan_like_bf16(shape) -> torch.Tensor:
    # 0xFFFF is a bf16 NaN: any element the kernel fails to write fails parity
    return torch.full(shape, -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)


class Inputs:
    """Device copies of one workload plus its masks."""

    def __init__(self, w: W.Workload, causal=None, scale=None, kv_len=None, block_mask=None):
        self.w = w
        s = w.spec
        self.B, self.H, self.N, self.d = s.B, s.H, s.N, s.d
        self.causal = s.causal if causal is None else causal
        self.scale = s.scale if scale is None else scale
        self.kv_len_np = w.kv_len if kv_len is None else kv_len
        self.mask_np = w.block_mask if block_mask is None else block_mask
        self.q, self.k, self.v, self.do = (dev_bf16(getattr(w, n)) for n in ("q", "k", "v", "do"))
        self.kv_len = (None if self.kv_len_np is None
                       else torch.from_numpy(np.asarray(self.kv_len_np, np.int32)).cuda())
        self.mask = (None if self.mask_np is None
                     else torch.from_numpy(np.ascontiguousarray(self.mask_np, np.uint8)).cuda())

    def oracle_kwargs(self):
        return dict(causal=self.causal, kv_len=self.kv_len_np, block_mask=self.mask_np)

    def f64(self, name):
        return self.w.f64(name)


def run_fwd(x: Inputs, q=None, k=None, v=None):
    shape = (x.B, x.H, x.N, x.d)
    o = nan_like_bf16(shape)
    lse = torch.full((x.B, x.H, x.N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd(q if q is not None else x.q, k if k is not None else x.k,
              v if v is not None else x.v, o, lse, x.B, x.H, x.N, x.d, x.scale, x.causal,
              x.kv_len, x.mask, st)
    fa.fa_check(st)
    return o, lse


def run_bwd(x: Inputs, o, lse, q=None, k=None, v=None, do=None):
    shape = (x.B, x.H, x.N, x.d)
    dq, dk, dv = nan_like_bf16(shape), nan_like_bf16(shape), nan_like_bf16(shape)
    nbytes = fa.fa_bwd_workspace_size(x.B, x.H, x.N, x.d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")  # garbage on entry
    st = torch.cuda.current_stream()
    fa.fa_bwd(q if q is not None else x.q, k if k is not None else x.k,
              v if v is not None else x.v, o, lse, do if do is not None else x.do, dq, dk, dv,
              x.B, x.H, x.N, x.d, x.scale, x.causal, x.kv_len, x.mask, ws, nbytes, st)
    fa.fa_check(st)
    return dq, dk, dv


def rel_fro(got: np.ndarray, want: np.ndarray) -> float:
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    return float(num / den) if den > 0 else float(num)


def assert_o(got, want, what="O", maxabs_scale=1.0):
    """O within the parity tolerances; maxabs_scale widens the absolute bound
    for outputs scaled up on purpose (dropout's 1/(1-p'): every kept term of
    O, and its bf16 rounding, is multiplied by it; the relative bound holds as is)."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ma = float(np.max(np.abs(got - want))) if got.size else 0.0
    rf = rel_fro(got, want)
    assert ma <= TOL_O_MAXABS * maxabs_scale and rf <= TOL_O_RELFRO, \
        f"{what}: max-abs {ma:.3e}, rel-fro {rf:.3e}"
    return ma, rf


def assert_lse(got, want):
    fin = np.isfinite(want)
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), "lse: -inf pattern differs"
    if fin.any():
        ma = float(np.max(np.abs(got[fin] - want[fin])))
        assert ma <= TOL_LSE_MAXABS, f"lse: max-abs {ma:.3e}"


def assert_grad(got, want, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rf = rel_fro(got, want)
    assert rf <= TOL_GRAD_RELFRO, f"{what}: rel-fro {rf:.3e}"
    return rf


def run_fwd_dropout(x: Inputs, p, seed):
    shape = (x.B, x.H, x.N, x.d)
    o = nan_like_bf16(shape)
    lse = torch.full((x.B, x.H, x.N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    fa.fa_fwd_dropout(x.q, x.k, x.v, o, lse, x.B, x.H, x.N, x.d, x.scale, x.causal, x.kv_len,
                      x.mask, p, seed, st)
    fa.fa_check(st)
    return o, lse


def run_bwd_dropout(x: Inputs, o, lse, p, seed):
    shape = (x.B, x.H, x.N, x.d)
    dq, dk, dv = nan_like_bf16(shape), nan_like_bf16(shape), nan_like_bf16(shape)
    nbytes = fa.fa_bwd_workspace_size(x.B, x.H, x.N, x.d)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")  # garbage on entry
    st = torch.cuda.current_stream()
    fa.fa_bwd_dropout(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.B, x.H, x.N, x.d, x.scale,
                      x.causal, x.kv_len, x.mask, p, seed, ws, nbytes, st)
    fa.fa_check(st)
    return dq, dk, dv
