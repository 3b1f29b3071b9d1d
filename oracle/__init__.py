"""CPU oracle for deterministic gradient reduction (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The GPU library never loads it and
shares no code with it: ``dgr_oracle.c`` is compiled here, with gcc, into its
own shared library, and called through ctypes on numpy arrays.

Every function takes host (numpy) arrays of the same bytes that the GPU path
receives and returns what the canonical order defines:
tile partials by a fixed-width pairwise tree, folded in ascending tile order,
FP32 throughout (see the comments in ``dgr_oracle.c`` for the page passages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_dgr.so")

# No FMA contraction, no fast-math: every operation is one IEEE binary32 RN.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fno-unsafe-math-optimizations",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/liboracle_dgr.so (if stale)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class TcModel(ctypes.Structure):
    """Parameters of the tensor-core K16 step model (see dgr_oracle.c)."""
    _fields_ = [("group", ctypes.c_int32), ("frac_bits", ctypes.c_int32),
                ("acc_in_sum", ctypes.c_int32), ("final_rn", ctypes.c_int32),
                ("ref_from_fields", ctypes.c_int32)]

    def __repr__(self) -> str:
        return (f"TcModel(group={self.group}, frac_bits={self.frac_bits}, acc_in_sum={self.acc_in_sum}, "
                f"final_rn={self.final_rn}, ref_from_fields={self.ref_from_fields})")


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.dgro_pairwise.argtypes = [P, I64, I64]
        L.dgro_pairwise.restype = F32
        L.dgro_fold.argtypes = [P, I64]
        L.dgro_fold.restype = F32
        L.dgro_ordered_colsum.argtypes = [P, I32, I64, I64, I64, I64, I64, I64, P, I32, P]
        L.dgro_ordered_colsum.restype = I32
        L.dgro_ordered_rowdot_dprob.argtypes = [P, P, I32, I64, I64, I64, I64, I64, P, I32, P]
        L.dgro_ordered_rowdot_dprob.restype = I32
        L.dgro_det_index_add.argtypes = [P, I64, I64, I64, P, I64, P, I64, I64, P, P, P]
        L.dgro_det_index_add.restype = I32
        L.dgro_tc_default_model.argtypes = [P]
        L.dgro_tc_default_model.restype = None
        L.dgro_tc_k16_batch.argtypes = [I64, P, P, P, P, P, P]
        L.dgro_tc_k16_batch.restype = None
        L.dgro_grouped_wgrad_accumulate.argtypes = [P, P, P, I64, I64, I64, P, I64, I32, P]
        L.dgro_grouped_wgrad_accumulate.restype = I32
        L.dgro_wgrad_elements.argtypes = [P, P, P, I64, I64, P, I64, I64, P, P, P, P, P]
        L.dgro_wgrad_elements.restype = I32
        L.dgro_grouped_dbias.argtypes = [P, I32, I64, I64, I64, P, I64, I64, P, I64, I32]
        L.dgro_grouped_dbias.restype = I32
        L.dgro_topk_canonicalize.argtypes = [P, I64, P, I64, I64, I64, P, P, P, I64]
        L.dgro_topk_canonicalize.restype = I32
        L.dgro_exp_tang_array.argtypes = [P, P, I64]
        L.dgro_exp_tang_array.restype = None
        L.dgro_exp_tang_constants.argtypes = [P, P]
        L.dgro_exp_tang_constants.restype = None
        L.dgro_aux_loss.argtypes = [P, I64, I64, I64, P, F32, P]
        L.dgro_aux_loss.restype = I32
        L.dgro_dsrelu_dprob.argtypes = [P, P, P, I64, I64, I64, I64, P, P, I32, P, I64, P]
        L.dgro_dsrelu_dprob.restype = I32
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {name} failed with code {rc}")


DTYPE_F32, DTYPE_BF16 = 0, 1


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return DTYPE_F32
    if a.dtype == np.uint16:  # bf16 bit patterns
        return DTYPE_BF16
    raise TypeError(f"oracle takes float32 or bf16 bits (uint16), got {a.dtype}")


def pairwise(leaves: np.ndarray, width: int) -> np.float32:
    """Tile partial of `leaves` (len <= width) by the fixed-width pairwise tree."""
    v = np.ascontiguousarray(leaves, dtype=np.float32)
    assert 1 <= v.size <= width
    return np.float32(lib().dgro_pairwise(_ptr(v), v.size, width))


def fold(partials: np.ndarray) -> np.float32:
    """Ascending fold F = P0; F = F + Pj."""
    v = np.ascontiguousarray(partials, dtype=np.float32)
    assert v.size >= 1
    return np.float32(lib().dgro_fold(_ptr(v), v.size))


def ordered_colsum(x: np.ndarray, B: int, S: int, H: int, stride_b: int, stride_s: int,
                   out: np.ndarray, *, accumulate: bool = False, tile_rows: int = 128,
                   return_slots: bool = False):
    """Column sum over tokens t = b*S + s of the flat buffer `x` (elements)."""
    assert x.ndim == 1 and out.dtype == np.float32 and out.size == H
    n_tiles = -(-B * S // tile_rows)
    slots = np.empty((max(n_tiles, 1), H), np.float32) if return_slots else None
    rc = lib().dgro_ordered_colsum(_ptr(x), _dtype_code(x), B, S, H, stride_b, stride_s, tile_rows,
                                   _ptr(out), int(accumulate), _ptr(slots) if slots is not None else None)
    _check(rc, "ordered_colsum")
    return slots[:n_tiles] if return_slots else None


def ordered_rowdot_dprob(dY: np.ndarray, Y: np.ndarray, M: int, N: int, ld_dy: int, ld_y: int,
                         dprob: np.ndarray, *, accumulate: bool = False, tile_n: int = 128,
                         return_slots: bool = False):
    """dprob[m] = fold over N-tiles of the pairwise tree of dY*Y (flat buffers)."""
    assert dY.dtype == Y.dtype and dprob.dtype == np.float32 and dprob.size == M
    n_tiles = -(-N // tile_n)
    slots = np.empty((max(M, 1), max(n_tiles, 1)), np.float32) if return_slots else None
    rc = lib().dgro_ordered_rowdot_dprob(_ptr(dY), _ptr(Y), _dtype_code(dY), M, N, ld_dy, ld_y,
                                         tile_n, _ptr(dprob), int(accumulate),
                                         _ptr(slots) if slots is not None else None)
    _check(rc, "ordered_rowdot_dprob")
    return slots[:M, :n_tiles] if return_slots else None


def det_index_add(out: np.ndarray, R: int, D: int, ld_out: int, src: np.ndarray, ld_src: int,
                  idx: np.ndarray, N: int, *, seg_tile: int = 128):
    """In-place deterministic index_add into out[R+1, D]; returns (bad, perm, seg_start)."""
    assert out.dtype == np.float32 and src.dtype == np.float32 and idx.dtype == np.int32
    bad = np.zeros(1, np.int64)
    perm = np.empty(max(N, 1), np.int32)
    seg = np.empty(R + 2, np.int32)
    rc = lib().dgro_det_index_add(_ptr(out), R, D, ld_out, _ptr(src), ld_src, _ptr(idx), N, seg_tile,
                                  _ptr(bad), _ptr(perm), _ptr(seg))
    _check(rc, "det_index_add")
    return int(bad[0]), perm[:N], seg


def default_tc_model() -> TcModel:
    m = TcModel()
    lib().dgro_tc_default_model(ctypes.byref(m))
    return m


def tc_k16_batch(acc: np.ndarray, has_acc: np.ndarray, a_bits: np.ndarray, b_bits: np.ndarray,
                 model: TcModel | None = None) -> np.ndarray:
    """Model of one K16 tensor-core step for n elements; a_bits, b_bits are [n, 16] bf16 bits."""
    m = model if model is not None else default_tc_model()
    acc = np.ascontiguousarray(acc, np.float32)
    has = np.ascontiguousarray(has_acc, np.int32)
    a = np.ascontiguousarray(a_bits, np.uint16)
    b = np.ascontiguousarray(b_bits, np.uint16)
    n = acc.size
    assert has.size == n and a.shape == (n, 16) and b.shape == (n, 16)
    res = np.empty(n, np.float32)
    lib().dgro_tc_k16_batch(n, _ptr(acc), _ptr(has), _ptr(a), _ptr(b), ctypes.byref(m), _ptr(res))
    return res


def grouped_wgrad_accumulate(G_bits: np.ndarray, X_bits: np.ndarray, offs: np.ndarray, E: int,
                             N: int, K: int, main_grad: np.ndarray, *, chunk_tokens: int = 512,
                             sequential_into_out: bool = False, model: TcModel | None = None):
    """In place: main_grad[e] = main_grad[e] + fold_c p_c (full, for small shapes)."""
    m = model if model is not None else default_tc_model()
    assert G_bits.dtype == np.uint16 and X_bits.dtype == np.uint16 and offs.dtype == np.int64
    assert main_grad.dtype == np.float32 and main_grad.flags.c_contiguous
    rc = lib().dgro_grouped_wgrad_accumulate(_ptr(G_bits), _ptr(X_bits), _ptr(offs), E, N, K,
                                             _ptr(main_grad), chunk_tokens, int(sequential_into_out),
                                             ctypes.byref(m))
    _check(rc, "grouped_wgrad_accumulate")


def wgrad_elements(G_bits: np.ndarray, X_bits: np.ndarray, offs: np.ndarray, N: int, K: int,
                   e_idx: np.ndarray, n_idx: np.ndarray, k_idx: np.ndarray,
                   main_grad_in: np.ndarray, *, chunk_tokens: int = 512,
                   model: TcModel | None = None) -> np.ndarray:
    """Updated main_grad values at the listed (e, n, k), given their old values."""
    m = model if model is not None else default_tc_model()
    e = np.ascontiguousarray(e_idx, np.int64)
    n = np.ascontiguousarray(n_idx, np.int64)
    k = np.ascontiguousarray(k_idx, np.int64)
    mg = np.ascontiguousarray(main_grad_in, np.float32)
    res = np.empty(e.size, np.float32)
    rc = lib().dgro_wgrad_elements(_ptr(G_bits), _ptr(X_bits), _ptr(offs), N, K, _ptr(mg),
                                   chunk_tokens, e.size, _ptr(e), _ptr(n), _ptr(k),
                                   ctypes.byref(m), _ptr(res))
    _check(rc, "wgrad_elements")
    return res


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))


def grouped_dbias(dY: np.ndarray, T: int, H: int, ld: int, offs: np.ndarray, out: np.ndarray, *,
                  ld_out: int | None = None, accumulate: bool = False, tile_rows: int = 128) -> None:
    """out[e][h] (+)= ordered column sum of dY over expert e's rows offs[e] .. offs[e+1]-1
    (flat buffers, elements; tiles counted from each expert's first row)."""
    o = np.ascontiguousarray(offs, dtype=np.int64)
    E = o.size - 1
    ld_out = H if ld_out is None else ld_out
    assert dY.ndim == 1 and out.dtype == np.float32 and out.ndim == 1 and out.flags.c_contiguous
    assert E >= 1 and (E == 0 or out.size >= (E - 1) * ld_out + H)
    rc = lib().dgro_grouped_dbias(_ptr(dY), _dtype_code(dY), T, H, ld, _ptr(o), E, tile_rows, _ptr(out),
                                  ld_out, int(accumulate))
    _check(rc, "grouped_dbias")


def exp_tang(x: np.ndarray) -> np.ndarray:
    """The top-K softmax's binary32 exponential (Tang's table-driven method), elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib().dgro_exp_tang_array(_ptr(x), _ptr(out), x.size)
    return out


def exp_tang_constants() -> tuple[np.ndarray, np.ndarray]:
    """The method's table: S_lead[j] and S_trail[j], 2^(j/32) split in two binary32 parts."""
    lead = np.empty(32, np.float32)
    trail = np.empty(32, np.float32)
    lib().dgro_exp_tang_constants(_ptr(lead), _ptr(trail))
    return lead, trail


def topk_canonicalize(ids: np.ndarray, logits: np.ndarray):
    """Per row: slots stably sorted by id (padding, id < 0, last), logits permuted alike, and the
    softmax of the valid slots recomputed in that order. Returns (ids, logits, probs)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    R, K = ids.shape
    assert logits.shape == (R, K)
    oi = np.empty_like(ids)
    ol = np.empty_like(logits)
    pr = np.empty_like(logits)
    rc = lib().dgro_topk_canonicalize(_ptr(ids), K, _ptr(logits), K, R, K, _ptr(oi), _ptr(ol), _ptr(pr), K)
    _check(rc, "topk_canonicalize")
    return oi, ol, pr


def aux_loss(probs: np.ndarray, tokens_per_expert: np.ndarray, scale: float) -> np.float32:
    """RN(scale * S): S = the canonical sum over tokens (tiles of 128) of each token's canonical
    row dot of probs[t] with tokens_per_expert (expert tiles of 128)."""
    p = np.ascontiguousarray(probs, dtype=np.float32)
    tpe = np.ascontiguousarray(tokens_per_expert, dtype=np.int32)
    N, E = p.shape
    assert tpe.shape == (E,)
    out = np.zeros(1, np.float32)
    rc = lib().dgro_aux_loss(_ptr(p), N, E, E, _ptr(tpe), np.float32(scale), _ptr(out))
    _check(rc, "aux_loss")
    return out[0]


def dsrelu_dprob(A_bits: np.ndarray, B_bits: np.ndarray, offs: np.ndarray, dY_bits: np.ndarray, dprob: np.ndarray,
                 *, accumulate: bool = False, rows: np.ndarray | None = None, model: TcModel | None = None):
    """dprob[m] (+)= fold over N-tiles of pw_128(RN(dY * RN(relu(C)^2))), C = A_e B_e by K16
    tensor-core steps. A [T, K], B [E, K, N], dY [T, N] bf16 bits; with `rows`, dprob[i] is row rows[i]."""
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_bits, dtype=np.uint16)
    dY = np.ascontiguousarray(dY_bits, dtype=np.uint16)
    o = np.ascontiguousarray(offs, dtype=np.int64)
    T, K = A.shape
    E, K2, N = B.shape
    assert K2 == K and dY.shape == (T, N) and o.size == E + 1 and dprob.dtype == np.float32
    m = model or default_tc_model()
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    rc = lib().dgro_dsrelu_dprob(_ptr(A), _ptr(B), _ptr(o), E, T, K, N, _ptr(dY), _ptr(dprob), int(accumulate),
                                 _ptr(r) if r is not None else None, 0 if r is None else r.size, ctypes.byref(m))
    _check(rc, "dsrelu_dprob")
