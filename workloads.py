"""Seeded synthetic attention workloads (inputs only).

This module draws the inputs that both the CUDA path and the CPU oracle
consume.  It holds none of the attention arithmetic: it draws normal
variates, rounds them to bf16, and builds the masks and lengths.  Nothing
here imports the oracle or the CUDA library.

Shapes follow the pages' workloads (FlashAttention explainer, "Results"):
BERT-large (sequence 512), GPT-2 (1K and 4K contexts) and block-sparse
attention at 64K (Path-256); only the shapes are used, never a dataset.

Recipe per workload (numpy ``default_rng(seed)``, PCG64; draw order Q, K, V,
dO as float32 standard normals, then the workload-specific draws; cast to
bf16 with round-to-nearest-even):

* ``tiny``    B=1 H=1 N=128 d=64, no mask, scale 1/8.
* ``bert``    B=16 H=16 N=512 d=64; Q, K, V scaled by 0.5 before the cast;
              kv_len[b] uniform integer in [256, 512]; scale 1/8.
* ``gpt2``    B=8 H=12 N=1024 d=64, causal, scale 1/8.
* ``gpt2_4k`` B=2 H=12 N=4096 d=64, causal, scale 1/8; per (b, h) round(0.01 N)
              = 41 key rows chosen without replacement are multiplied by 8
              in float32 before the cast (exact in bf16).
* ``sparse64k`` B=1 H=8 N=65536 d=64, non-causal, scale 1/8; 128x128 block
              mask of 512x512 entries: the band |i - j| <= 1 (1534 blocks)
              plus off-band blocks drawn uniformly without replacement until
              nnz = round(0.05 * 512 * 512) = 13107.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    scale: float
    qkv_scale: float = 1.0
    kv_len: tuple | None = None       # ("uniform", lo, hi)
    peaky_frac: float = 0.0           # fraction of key rows scaled by peaky_mul
    peaky_mul: float = 8.0
    sparse_nnz_frac: float = 0.0      # block-sparse density (0 = dense)
    band: int = 1                     # |i - j| <= band blocks always kept


SPECS = {
    "tiny": Spec("tiny", 1, 1, 128, 64, False, 1.0 / 8.0),
    "bert": Spec("bert", 16, 16, 512, 64, False, 1.0 / 8.0, qkv_scale=0.5,
                 kv_len=("uniform", 256, 512)),
    "gpt2": Spec("gpt2", 8, 12, 1024, 64, True, 1.0 / 8.0),
    "gpt2_4k": Spec("gpt2_4k", 2, 12, 4096, 64, True, 1.0 / 8.0, peaky_frac=0.01),
    "sparse64k": Spec("sparse64k", 1, 8, 65536, 64, False, 1.0 / 8.0, sparse_nnz_frac=0.05),
}
# seed = position of the workload in the list of five configurations (1-based)
SEEDS = {"tiny": 1, "bert": 2, "gpt2": 3, "gpt2_4k": 4, "sparse64k": 5}


@dataclasses.dataclass
class Workload:
    spec: Spec
    q: np.ndarray            # uint16 bf16 bit patterns [B, H, N, d]
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    kv_len: np.ndarray | None    # int32 [B]
    block_mask: np.ndarray | None  # uint8 [nb, nb]

    @property
    def shape(self):
        s = self.spec
        return s.B, s.H, s.N, s.d

    def f64(self, name: str) -> np.ndarray:
        """The bf16 values of tensor ``name`` widened exactly to float64."""
        return bf16_bits_to_f64(getattr(self, name))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round-to-nearest-even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def make_block_mask(rng: np.random.Generator, nb: int, nnz_frac: float, band: int) -> np.ndarray:
    """Band |i - j| <= band plus uniformly drawn off-band blocks up to the target count."""
    i = np.arange(nb)[:, None]
    j = np.arange(nb)[None, :]
    mask = (np.abs(i - j) <= band).astype(np.uint8)
    target = int(round(nnz_frac * nb * nb))
    have = int(mask.sum())
    if target > have:
        off = np.flatnonzero(mask.reshape(-1) == 0)
        pick = rng.choice(off, size=target - have, replace=False)
        mask.reshape(-1)[pick] = 1
    return mask


def make(name: str, seed: int | None = None, **over) -> Workload:
    """Draw the workload ``name`` (see module docstring), optionally with
    fields of its Spec overridden (e.g. ``N=4096`` or ``B=1``)."""
    spec = dataclasses.replace(SPECS[name], **over) if over else SPECS[name]
    if seed is None:
        seed = SEEDS.get(name, 0)
    return generate(spec, seed)


def generate(spec: Spec, seed: int) -> Workload:
    rng = np.random.default_rng(seed)
    shape = (spec.B, spec.H, spec.N, spec.d)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    do = rng.standard_normal(shape, dtype=np.float32)
    if spec.qkv_scale != 1.0:
        s = np.float32(spec.qkv_scale)
        q *= s
        k *= s
        v *= s
    kv_len = None
    if spec.kv_len is not None:
        _, lo, hi = spec.kv_len
        kv_len = rng.integers(lo, hi + 1, size=spec.B).astype(np.int32)
    if spec.peaky_frac > 0:
        n_peaky = int(round(spec.peaky_frac * spec.N))
        for b in range(spec.B):
            for h in range(spec.H):
                rows = rng.choice(spec.N, size=n_peaky, replace=False)
                k[b, h, rows, :] *= np.float32(spec.peaky_mul)
    block_mask = None
    if spec.sparse_nnz_frac > 0:
        nb = math.ceil(spec.N / BLOCK)
        block_mask = make_block_mask(rng, nb, spec.sparse_nnz_frac, spec.band)
    return Workload(spec, f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v),
                    f32_to_bf16_bits(do), kv_len, block_mask)


def sample_rows(rng: np.random.Generator, B: int, H: int, N: int, per_head: int) -> np.ndarray:
    """Global row ids (bh * N + i): ``per_head`` distinct rows of every (b, h), sorted."""
    out = []
    for bh in range(B * H):
        n = min(per_head, N)
        rows = np.sort(rng.choice(N, size=n, replace=False))
        out.append(bh * N + rows)
    return np.concatenate(out).astype(np.int64)


def sample_key_tiles(rng: np.random.Generator, B: int, H: int, N: int, tiles_per_head: int,
                     tile: int = BLOCK) -> np.ndarray:
    """Global key-row ids covering ``tiles_per_head`` whole key tiles per (b, h)."""
    nt = math.ceil(N / tile)
    out = []
    for bh in range(B * H):
        for t in np.sort(rng.choice(nt, size=min(tiles_per_head, nt), replace=False)):
            rows = np.arange(t * tile, min((t + 1) * tile, N))
            out.append(bh * N + rows)
    return np.concatenate(out).astype(np.int64)
