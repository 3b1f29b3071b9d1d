"""Helpers shared by the tests: bit comparisons, fp64 references and bounds.

The fp64 references here are plain numpy sums (no canonical order); they pin
the oracle's magnitudes and completeness, never its bits.
"""
from __future__ import annotations

import os

import numpy as np

U32 = 2.0 ** -24  # unit roundoff of binary32


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def assert_bits_equal(got, want, what: str = "") -> None:
    g, w = f32_bits(got), f32_bits(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.flatnonzero(g.reshape(-1) != w.reshape(-1))
    if bad.size:
        i = bad[0]
        gv = g.reshape(-1)[i:i + 1].view(np.float32)[0]
        wv = w.reshape(-1)[i:i + 1].view(np.float32)[0]
        raise AssertionError(f"{what}: {bad.size} of {g.size} outputs differ; first at flat {i}: "
                             f"got {gv!r} ({g.reshape(-1)[i]:#010x}) want {wv!r} ({w.reshape(-1)[i]:#010x})")


def gamma(k: int) -> float:
    return k * U32 / (1.0 - k * U32)


def rel_l2(got, exact) -> float:
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    den = np.linalg.norm(exact)
    return float(np.linalg.norm(got - exact) / (den if den > 0 else 1.0))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_hand_cases():
    cases = []
    with open(os.path.join(GOLDEN, "hand_cases.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, width, values, expected, passage = [f.strip() for f in line.split("|")]
            vals = np.array([float(v) for v in values.split(",")], np.float32)
            cases.append((kind, int(width), vals, np.float32(float(expected)), passage))
    return cases
