"""Seeded synthetic inputs for deterministic gradient reduction.

This module only draws random data: it holds none of the method's arithmetic,
so both the CPU oracle (through the tests) and the GPU library (through the
tests and the benchmark) can take their inputs from it. Every generator uses
one ``torch.Generator('cpu')`` seeded per workload and draws in a fixed order;
fp32 draws are narrowed to bf16 with torch's round-to-nearest-even. All
tensors are CPU tensors; ``bits()`` gives the raw bf16 bit patterns as a numpy
uint16 array for the oracle.

The five workloads (shapes, distributions and draw order):
  colsum_small   x bf16 [2048, 16] ~ U(-1, 1)                                 seed 1
  index_add      src fp32 [262144, 128] ~ N(0, 1); idx int32 ~ U[0, 16384),
                 then floor(0.1 N) positions (a random permutation's prefix)
                 set to -1; out fp32 [16385, 128] zeros                      seed 2
  dprob          dY, Y bf16 [65536, 4096] ~ N(0, 1)                          seed 3
  colsum_strided base bf16 [4, 2048, 128] ~ N(0, 0.02^2); the view
                 base[..., :64] (token stride 128); base[..., 64:] is then
                 overwritten with bf16 NaN as a poison                        seed 4
  colsum_large   x bf16 [8388608, 64] ~ N(0, 0.02^2), drawn after the
                 strided base from the same generator                        seed 4
  wgrad          expert of each of 32768 tokens ~ multinomial(uniform over 8),
                 counts -> offsets; G bf16 [32768, 4096], X bf16 [32768, 2048]
                 ~ N(0, 1), rows grouped by expert; main_grad fp32
                 [8, 4096, 2048] ~ N(0, 1e-3^2)                              seed 5
  dbias          expert of each of 65536 rows ~ multinomial(uniform over 8),
                 counts -> offsets; dY bf16 [65536, 2048] ~ N(0, 1), rows
                 grouped by expert (the cuDNN-frontend dsReLU example's
                 valid_m 64k, n 2048); dbias fp32 [8, 2048] zeros             seed 6
  topk           65536 rows of 128 slots: one id a slot, unique in the row
                 (slot k's id in [k*512, (k+1)*512) of 65536 keys), slots
                 shuffled per row; 10 % of the slots then padding (-1) and
                 every 64th row all padding; logits ~ N(0, 3^2) fp32          seed 7
  aux loss       router probs fp32 [65536, 128] = softmax over the experts of
                 N(0, 1) logits; tokens_per_expert int32 [128] = counts of a
                 top-8 routing (8 experts drawn per token without
                 replacement); scale = 1e-2 * E / (topk * N^2)               seed 8
  dsrelu dprob   expert of each of 16384 tokens ~ multinomial(uniform over 8),
                 counts -> offsets; A bf16 [16384, 2048] ~ N(0, 1), B bf16
                 [8, 2048, 4096] ~ N(0, 1/2048) (so C ~ N(0, 1)), dY bf16
                 [16384, 4096] ~ N(0, 1); dprob fp32 [16384] zeros           seed 9
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (shares memory)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    assert t.dtype == torch.float32
    return t.contiguous().numpy()


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return g


def _draw(shape, dist: str, g: torch.Generator, scale: float = 1.0) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=g) * scale
    if dist == "ternary":
        return torch.randint(-1, 2, shape, generator=g).to(torch.float32)
    raise ValueError(dist)


# --------------------------------------------------------------------------
# column sum
# --------------------------------------------------------------------------

@dataclass
class ColsumInput:
    base: torch.Tensor      # contiguous storage the view lives in
    B: int
    S: int
    H: int
    stride_b: int           # elements
    stride_s: int           # elements
    offset: int = 0         # element offset of x[0][0][0] inside base


def colsum_input(B: int, S: int, H: int, *, seed: int, dist: str = "normal", scale: float = 1.0,
                 dtype: torch.dtype = torch.bfloat16, token_stride: int | None = None,
                 poison: bool = True) -> ColsumInput:
    """x [B, S, H]; with token_stride > H the rows live in a wider base and the
    unused columns hold NaN (bf16) or NaN (fp32) so a stray read shows."""
    g = _gen(seed)
    ts = H if token_stride is None else token_stride
    assert ts >= H
    base = _draw((B, S, ts), dist, g, scale).to(dtype)
    if ts > H and poison:
        base[..., H:] = float("nan")
    return ColsumInput(base.reshape(-1), B, S, H, S * ts, ts)


def colsum_small() -> ColsumInput:
    return colsum_input(1, 2048, 16, seed=1, dist="uniform")


def _strided_and_large():
    g = _gen(4)
    base = (torch.randn((4, 2048, 128), generator=g) * 0.02).to(torch.bfloat16)
    base[..., 64:] = float("nan")
    strided = ColsumInput(base.reshape(-1), 4, 2048, 64, 2048 * 128, 128)
    return strided, g


def colsum_strided() -> ColsumInput:
    return _strided_and_large()[0]


def colsum_large() -> ColsumInput:
    _, g = _strided_and_large()
    x = (torch.randn((8388608, 64), generator=g) * 0.02).to(torch.bfloat16)
    return ColsumInput(x.reshape(-1), 1, 8388608, 64, 8388608 * 64, 64)


# --------------------------------------------------------------------------
# dprob
# --------------------------------------------------------------------------

@dataclass
class DprobInput:
    dY: torch.Tensor  # [M, ld] (only the first N columns are read)
    Y: torch.Tensor
    M: int
    N: int


def dprob_input(M: int, N: int, *, seed: int, dist: str = "normal",
                dtype: torch.dtype = torch.bfloat16, ld: int | None = None) -> DprobInput:
    g = _gen(seed)
    ldv = N if ld is None else ld
    dY = _draw((M, ldv), dist, g).to(dtype)
    Y = _draw((M, ldv), dist, g).to(dtype)
    if ldv > N:
        dY[:, N:] = float("nan")
        Y[:, N:] = float("nan")
    return DprobInput(dY, Y, M, N)


def dprob_full() -> DprobInput:
    return dprob_input(65536, 4096, seed=3)


# --------------------------------------------------------------------------
# index_add
# --------------------------------------------------------------------------

@dataclass
class IndexAddInput:
    src: torch.Tensor   # fp32 [N, D]
    idx: torch.Tensor   # int32 [N]
    out: torch.Tensor   # fp32 [R+1, D]
    R: int


def index_add_input(N: int, D: int, R: int, *, seed: int, pad_frac: float = 0.1,
                    dist: str = "normal", out_init: str = "zeros") -> IndexAddInput:
    g = _gen(seed)
    src = _draw((N, D), dist, g).to(torch.float32)
    idx = torch.randint(0, max(R, 1), (N,), generator=g, dtype=torch.int64).to(torch.int32)
    n_pad = int(pad_frac * N)
    if n_pad:
        pos = torch.randperm(N, generator=g)[:n_pad]
        idx[pos] = -1
    if R == 0:
        idx[:] = -1
    if out_init == "zeros":
        out = torch.zeros((R + 1, D), dtype=torch.float32)
    else:
        out = _draw((R + 1, D), dist, g).to(torch.float32)
    return IndexAddInput(src, idx, out, R)


def index_add_full() -> IndexAddInput:
    return index_add_input(262144, 128, 16384, seed=2)


# --------------------------------------------------------------------------
# grouped wgrad
# --------------------------------------------------------------------------

@dataclass
class WgradInput:
    G: torch.Tensor          # bf16 [T, N]
    X: torch.Tensor          # bf16 [T, K]
    offs: torch.Tensor       # int64 [E+1]
    main_grad: torch.Tensor  # fp32 [E, N, K]
    E: int


def wgrad_input(E: int, T: int, N: int, K: int, *, seed: int, dist: str = "normal",
                counts: list[int] | None = None, mg_scale: float = 1e-3) -> WgradInput:
    g = _gen(seed)
    if counts is None:
        ex = torch.multinomial(torch.ones(E), T, replacement=True, generator=g)
        cnt = torch.bincount(ex, minlength=E)
    else:
        assert len(counts) == E and sum(counts) == T
        cnt = torch.tensor(counts, dtype=torch.int64)
    offs = torch.zeros(E + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(cnt, 0)
    G = _draw((T, N), dist, g).to(torch.bfloat16)
    X = _draw((T, K), dist, g).to(torch.bfloat16)
    if dist == "ternary":
        mg = torch.randint(-4, 5, (E, N, K), generator=g).to(torch.float32)
    else:
        mg = torch.randn((E, N, K), generator=g) * mg_scale
    return WgradInput(G, X, offs, mg.to(torch.float32), E)


def wgrad_full() -> WgradInput:
    return wgrad_input(8, 32768, 4096, 2048, seed=5)


# --------------------------------------------------------------------------
# one tensor-core K16 step (inputs for the hardware check of the step model)
# --------------------------------------------------------------------------

@dataclass
class TcStepInput:
    A: np.ndarray   # bf16 bits [n, 128, 16]
    B: np.ndarray   # bf16 bits [n, 16, 256]
    C: np.ndarray   # fp32 [n, 128, 256]
    accumulate: int


def _bf16_bits_np(x: np.ndarray) -> np.ndarray:
    return bits(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16))


def _wide(rng, shape, lo, hi):
    s = rng.choice([-1.0, 1.0], shape)
    return (s * (1 + rng.random(shape)) * np.exp2(rng.integers(lo, hi, shape))).astype(np.float32)


def tc_step_input(kind: str, n: int, seed: int) -> TcStepInput:
    """kind: 'normal' (N(0,1) operands and accumulator), 'normal_noacc' (no
    accumulator input), 'wide' (magnitudes 2^-12..2^12, accumulator 2^-20..2^20),
    'designed' (B = 1: rows of A are 16-term patterns - one large term among
    tiny ones, cancelling pairs, equal magnitudes, spread powers of two - added
    to accumulators from 2^-40 to 2^30)."""
    rng = np.random.default_rng(seed)
    acc = 0 if kind == "normal_noacc" else 1
    if kind in ("normal", "normal_noacc"):
        A = rng.standard_normal((n, 128, 16)).astype(np.float32)
        B = rng.standard_normal((n, 16, 256)).astype(np.float32)
        C = rng.standard_normal((n, 128, 256)).astype(np.float32)
    elif kind == "wide":
        A = _wide(rng, (n, 128, 16), -12, 12)
        B = _wide(rng, (n, 16, 256), -12, 12)
        C = _wide(rng, (n, 128, 256), -20, 20)
    elif kind == "designed":
        A = np.zeros((n, 128, 16), np.float32)
        C = np.zeros((n, 128, 256), np.float32)
        for p in range(n):
            for m in range(128):
                k = rng.integers(0, 6)
                if k == 0:
                    A[p, m] = _wide(rng, (16,), -30, -10)
                    A[p, m, rng.integers(16)] = _wide(rng, (1,), 0, 4)[0]
                elif k == 1:
                    A[p, m] = _wide(rng, (16,), -26, -14)
                    i, j = rng.choice(16, 2, replace=False)
                    big = _wide(rng, (1,), 2, 10)[0]
                    A[p, m, i], A[p, m, j] = big, -big
                elif k == 2:
                    A[p, m] = rng.choice([-1, 1], 16) * np.exp2(rng.integers(-30, 0))
                elif k == 3:
                    A[p, m] = rng.choice([-1, 1], 16) * np.exp2(rng.integers(-40, 5, 16))
                elif k == 4:
                    A[p, m, rng.integers(16)] = _wide(rng, (1,), -10, 10)[0]
                else:
                    A[p, m] = _wide(rng, (16,), -8, 8)
                c = rng.integers(0, 4)
                C[p, m] = (_wide(rng, (256,), -6, 6) if c == 0 else _wide(rng, (256,), 10, 30) if c == 1 else
                           np.exp2(rng.integers(-30, 30, 256)) * rng.choice([-1, 1], 256) if c == 2 else
                           _wide(rng, (256,), -40, -20)).astype(np.float32)
        B = np.ones((n, 16, 256), np.float32)
    else:
        raise ValueError(kind)
    return TcStepInput(_bf16_bits_np(A), _bf16_bits_np(B), C, acc)


# --------------------------------------------------------------------------
# grouped dbias
# --------------------------------------------------------------------------

@dataclass
class DbiasInput:
    dY: torch.Tensor         # [T, ld] storage; the rows' first H columns are the data
    offs: torch.Tensor       # int64 [E+1]
    out: torch.Tensor        # fp32 [E, H]
    T: int
    H: int
    ld: int
    E: int


def dbias_input(T: int, H: int, E: int, *, seed: int, dist: str = "normal", dtype: torch.dtype = torch.bfloat16,
                counts: list[int] | None = None, ld: int | None = None, out_init: str = "zeros") -> DbiasInput:
    """Rows grouped by expert: counts from a multinomial over E experts (or
    given); with ld > H the unused columns hold NaN so a stray read shows."""
    g = _gen(seed)
    if counts is None:
        ex = torch.multinomial(torch.ones(E), T, replacement=True, generator=g)
        cnt = torch.bincount(ex, minlength=E)
    else:
        assert len(counts) == E and sum(counts) == T
        cnt = torch.tensor(counts, dtype=torch.int64)
    offs = torch.zeros(E + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(cnt, 0)
    ld = H if ld is None else ld
    assert ld >= H
    dY = _draw((T, ld), dist, g).to(dtype)
    if ld > H:
        dY[:, H:] = float("nan")
    if out_init == "zeros":
        out = torch.zeros((E, H), dtype=torch.float32)
    else:
        out = _draw((E, H), dist, g).to(torch.float32)
    return DbiasInput(dY, offs, out, T, H, ld, E)


def dbias_full() -> DbiasInput:
    return dbias_input(65536, 2048, 8, seed=6)


# --------------------------------------------------------------------------
# canonical compact top-K
# --------------------------------------------------------------------------

@dataclass
class TopkInput:
    ids: torch.Tensor     # int32 [R, K], padding -1
    logits: torch.Tensor  # fp32 [R, K]


def topk_input(R: int, K: int, *, seed: int, n_keys: int = 65536, pad_frac: float = 0.1,
               pad_row_every: int = 64, scale: float = 3.0) -> TopkInput:
    """Ids unique within a row (slot k draws from its own block of n_keys / K keys), in a
    shuffled slot order; then padding slots and all-padding rows."""
    g = _gen(seed)
    width = max(1, n_keys // K)
    ids = torch.randint(0, width, (R, K), generator=g) + torch.arange(K) * width
    order = torch.argsort(torch.rand((R, K), generator=g), dim=1)
    ids = torch.gather(ids, 1, order)
    pad = torch.rand((R, K), generator=g) < pad_frac
    ids[pad] = -1
    if pad_row_every:
        ids[::pad_row_every] = -1
    logits = torch.randn((R, K), generator=g) * scale
    return TopkInput(ids.to(torch.int32), logits.to(torch.float32))


def topk_full() -> TopkInput:
    return topk_input(65536, 128, seed=7)


# --------------------------------------------------------------------------
# aux-loss scalar
# --------------------------------------------------------------------------

@dataclass
class AuxInput:
    probs: torch.Tensor   # fp32 [N, E]
    tpe: torch.Tensor     # int32 [E]
    scale: float


def aux_input(N: int, E: int, *, seed: int, topk: int = 8, dist: str = "softmax", coeff: float = 1e-2) -> AuxInput:
    g = _gen(seed)
    if dist == "softmax":
        probs = torch.softmax(torch.randn((N, E), generator=g), dim=1)
    else:
        probs = _draw((N, E), dist, g)
    k = min(topk, E)
    picks = torch.argsort(torch.rand((max(N, 1), E), generator=g), dim=1)[:N, :k]
    tpe = torch.bincount(picks.reshape(-1), minlength=E)
    scale = coeff * E / (k * max(N, 1) ** 2)
    return AuxInput(probs.to(torch.float32), tpe.to(torch.int32), scale)


def aux_full() -> AuxInput:
    return aux_input(65536, 128, seed=8)


# --------------------------------------------------------------------------
# dprob fused into the grouped dsReLU GEMM
# --------------------------------------------------------------------------

@dataclass
class DsreluInput:
    A: torch.Tensor      # bf16 [T, K], rows grouped by expert
    B: torch.Tensor      # bf16 [E, K, N]
    dY: torch.Tensor     # bf16 [T, N]
    offs: torch.Tensor   # int64 [E + 1]
    dprob: torch.Tensor  # fp32 [T]


def dsrelu_input(E: int, T: int, K: int, N: int, *, seed: int, dist: str = "normal",
                 counts: list[int] | None = None, out_init: str = "zeros") -> DsreluInput:
    g = _gen(seed)
    if counts is None:
        ex = torch.multinomial(torch.ones(E), T, replacement=True, generator=g)
        cnt = torch.bincount(ex, minlength=E)
    else:
        assert len(counts) == E and sum(counts) == T
        cnt = torch.tensor(counts, dtype=torch.int64)
    offs = torch.zeros(E + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(cnt, 0)
    A = _draw((T, K), dist, g).to(torch.bfloat16)
    Bs = 1.0 if dist == "ternary" else K ** -0.5
    B = (_draw((E, K, N), dist, g) * Bs).to(torch.bfloat16)
    dY = _draw((T, N), dist, g).to(torch.bfloat16)
    dprob = torch.zeros(T, dtype=torch.float32) if out_init == "zeros" else _draw((T,), "normal", g)
    return DsreluInput(A, B, dY, offs, dprob.to(torch.float32))


def dsrelu_full() -> DsreluInput:
    return dsrelu_input(8, 16384, 2048, 4096, seed=9)
