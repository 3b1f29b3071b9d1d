"""Deterministic, atomic-free gradient reduction for GB300 (sm_103a).

A thin ctypes binding over ``libdgr.so`` (the C ABI declared in
``include/dgr.h``). Every function here only marshals arguments - tensor data
pointers, sizes, strides and the current CUDA stream - and calls the library;
all arithmetic runs in the library's CUDA kernels. There is no fallback: if
the library is missing or the device is not sm_103a, the call raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from contextlib import nullcontext as _nullcontext

import torch

from ._build import LIB as _LIB_PATH, build  # noqa: F401  (build is re-exported)

__all__ = [
    "DgrError", "lib", "build", "ordered_colsum", "ordered_rowdot_dprob", "det_index_add",
    "grouped_wgrad_accumulate", "colsum_workspace_bytes", "rowdot_workspace_bytes",
    "index_add_workspace_bytes", "wgrad_workspace_bytes", "workspace", "read_device_status",
    "ordered_colsum_noalloc", "colsum_noalloc_read_status",
]

DTYPE_F32, DTYPE_BF16 = 0, 1
STATUS = {0: "DGR_OK", 1: "DGR_ERR_INVALID_ARG", 2: "DGR_ERR_UNSUPPORTED", 3: "DGR_ERR_WORKSPACE_TOO_SMALL",
          4: "DGR_ERR_ALIAS", 5: "DGR_ERR_MISALIGNED", 6: "DGR_ERR_CUDA", 7: "DGR_ERR_TIMEOUT"}


class DgrError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdgr.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build the CUDA library first "
                              "(deterministic_gradient_reduction_gb300.build())")
        L = ctypes.CDLL(_LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "dgr_status_string": ([I32], ctypes.c_char_p),
            "dgr_version": ([], I32),
            "dgr_device_supported": ([I32], I32),
            "dgr_read_device_status": ([P, I32, P, P], I32),
            "dgr_query_device_status": ([P, P], I32),
            "dgr_colsum_workspace_bytes": ([I64, I64, I32], SZ),
            "dgr_ordered_colsum": ([P, I32, I64, I64, I64, I64, I64, P, I32, I32, P, SZ, P], I32),
            "dgr_rowdot_workspace_bytes": ([I64, I64, I32], SZ),
            "dgr_ordered_rowdot_dprob": ([P, P, I32, I64, I64, I64, I64, P, I32, I32, P, P, SZ, P], I32),
            "dgr_index_add_workspace_bytes": ([I64, I64, I64], SZ),
            "dgr_det_index_add": ([P, I64, I64, I64, P, I64, P, I64, I32, P, P, SZ, P], I32),
            "dgr_wgrad_workspace_bytes": ([I32, I64, I64], SZ),
            "dgr_grouped_wgrad_accumulate": ([P, P, P, I32, I64, I64, I64, P, I32, P, SZ, P], I32),
            "dgr_dbias_workspace_bytes": ([I64, I64, I32, I32], SZ),
            "dgr_grouped_dbias": ([P, I32, I64, I64, I64, P, I32, P, I64, I32, I32, P, SZ, P], I32),
            "dgr_topk_canonicalize": ([P, I64, P, I64, I64, I32, P, P, P, I64, P], I32),
            "dgr_aux_loss_workspace_bytes": ([I64], SZ),
            "dgr_aux_loss": ([P, I64, I32, I64, P, ctypes.c_float, P, P, SZ, P], I32),
            "dgr_dsrelu_dprob_workspace_bytes": ([I64, I64], SZ),
            "dgr_dsrelu_dprob": ([P, P, P, I32, I64, I64, I64, P, P, I32, P, SZ, P], I32),
            "dgr_diag_wait_timeout": ([I32, I32, P, SZ, P], I32),
            "dgr_diag_wgrad_stall": ([P, P, P, I32, I64, I64, I64, P, P, SZ, I32, I32, I32, P], I32),
            "dgr_diag_packed_ops": ([P, P, I64, P, P, P], I32),
            "dgr_diag_packed_chain": ([P, P, P, I64, P, P], I32),
            "dgr_diag_dsrelu_stall": ([P, P, P, I32, I64, I64, I64, P, P, P, SZ, I32, I32, I32, P], I32),
            "dgr_ordered_colsum_noalloc": ([P, I32, I64, I64, I64, I64, I64, P, I32, I32, P], I32),
            "dgr_colsum_noalloc_read_status": ([I32, P, P], I32),
            "dgr_diag_noalloc_wait_timeout": ([I32, I32, P], I32),
            "dgr_diag_set_schedule": ([I32, ctypes.c_uint32, I32], I32),
            "dgr_diag_colsum_plan": ([I64, I64, I32, I32, I32, I32, I32, I32, P], I32),
            "dgr_diag_atomic_colsum": ([P, I64, I32, P, P], I32),
            "dgr_diag_atomic_rowdot": ([P, P, I64, I32, P, P], I32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise DgrError(fn, rc)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"bf16 or fp32 expected, got {t.dtype}")


def workspace(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """A zeroed, 256-byte aligned device workspace of at least nbytes. With a stream, it is
    allocated and zeroed on that stream (the stream the call that uses it runs on), so the
    zeroing is ordered before the call whatever torch's current stream is doing."""
    if stream is None:
        return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")
    with torch.cuda.stream(stream):
        return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def read_device_status(ws: torch.Tensor, clear: bool = False, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check("dgr_read_device_status", lib().dgr_read_device_status(ws.data_ptr(), int(clear),
                                                                  ctypes.byref(st), _stream(stream)))
    return st.value


def query_device_status(ws: torch.Tensor, stream=None) -> int:
    """The status recorded in the workspace (0 when none; a code of STATUS), after synchronising
    the stream; the word is left as it is."""
    return int(lib().dgr_query_device_status(ws.data_ptr(), _stream(stream)))


def colsum_workspace_bytes(T: int, H: int, tile_rows: int = 128) -> int:
    return int(lib().dgr_colsum_workspace_bytes(T, H, tile_rows))


def ordered_colsum(x: torch.Tensor, out: torch.Tensor, *, accumulate: bool = False, tile_rows: int = 128,
                   ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[h] (+)= ordered column sum of x over its leading dims.

    x is [B, S, H] (or [T, H]) with a contiguous last dimension and any
    leading strides; out is fp32 [H].
    """
    if x.dim() == 2:
        x = x.unsqueeze(0)
    B, S, H = x.shape
    if H > 0 and x.stride(2) != 1:
        raise ValueError("the last dimension of x must be contiguous")
    if ws is None:
        ws = workspace(colsum_workspace_bytes(B * S, H, tile_rows), x.device, stream)
    _check("dgr_ordered_colsum", lib().dgr_ordered_colsum(
        _ptr(x), _dtype(x), B, S, H, x.stride(0), x.stride(1), _ptr(out), int(accumulate), tile_rows,
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def ordered_colsum_noalloc(x: torch.Tensor, out: torch.Tensor, *, accumulate: bool = False, tile_rows: int = 128,
                           stream=None) -> torch.Tensor:
    """ordered_colsum without a workspace: the library's static scratch array serves as one (calls
    needing more than it holds are refused; calls that overlap on the GPU race on it)."""
    if x.dim() == 2:
        x = x.unsqueeze(0)
    B, S, H = x.shape
    if H > 0 and x.stride(2) != 1:
        raise ValueError("the last dimension of x must be contiguous")
    _check("dgr_ordered_colsum_noalloc", lib().dgr_ordered_colsum_noalloc(
        _ptr(x), _dtype(x), B, S, H, x.stride(0), x.stride(1), _ptr(out), int(accumulate), tile_rows,
        _stream(stream)))
    return out


def colsum_noalloc_read_status(clear: bool = False, stream=None) -> int:
    """The status word of the no-alloc column sum's scratch (0 when no device-side error was recorded)."""
    st = ctypes.c_int32(0)
    _check("dgr_colsum_noalloc_read_status", lib().dgr_colsum_noalloc_read_status(int(clear), ctypes.byref(st),
                                                                                  _stream(stream)))
    return st.value


def rowdot_workspace_bytes(M: int, N: int, tile_n: int = 128) -> int:
    return int(lib().dgr_rowdot_workspace_bytes(M, N, tile_n))


def ordered_rowdot_dprob(dY: torch.Tensor, Y: torch.Tensor, dprob: torch.Tensor, *, accumulate: bool = False,
                         tile_n: int = 128, slots: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """dprob[m] (+)= ordered sum over n of dY[m, n] * Y[m, n] (rows may be strided)."""
    M, N = dY.shape
    if Y.shape != dY.shape or Y.dtype != dY.dtype:
        raise ValueError("dY and Y must have the same shape and dtype")
    if N > 0 and (dY.stride(1) != 1 or Y.stride(1) != 1):
        raise ValueError("rows of dY and Y must be contiguous")
    _check("dgr_ordered_rowdot_dprob", lib().dgr_ordered_rowdot_dprob(
        _ptr(dY), _ptr(Y), _dtype(dY), M, N, dY.stride(0), Y.stride(0), _ptr(dprob), int(accumulate), tile_n,
        _ptr(slots), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return dprob


def index_add_workspace_bytes(N: int, R: int, D: int) -> int:
    return int(lib().dgr_index_add_workspace_bytes(N, R, D))


def det_index_add(out: torch.Tensor, src: torch.Tensor, idx: torch.Tensor, *, seg_tile: int = 128,
                  bad_count: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """out[idx[i]] += src[i] in the canonical order; idx -1 (and out-of-range) go to out[R] (R = rows-1)."""
    R = out.shape[0] - 1
    N, D = src.shape
    if out.shape[1] != D or idx.shape != (N,) or idx.dtype != torch.int32:
        raise ValueError("out [R+1, D], src [N, D], idx int32 [N] expected")
    if ws is None:
        ws = workspace(index_add_workspace_bytes(N, R, D), out.device, stream)
    _check("dgr_det_index_add", lib().dgr_det_index_add(
        _ptr(out), R, D, out.stride(0), _ptr(src), src.stride(0), _ptr(idx), N, seg_tile, _ptr(bad_count),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def wgrad_workspace_bytes(E: int, N: int, K: int) -> int:
    return int(lib().dgr_wgrad_workspace_bytes(E, N, K))


def grouped_wgrad_accumulate(G: torch.Tensor, X: torch.Tensor, offs: torch.Tensor, main_grad: torch.Tensor, *,
                             chunk_tokens: int = 512, ws: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """main_grad[e] += G_e^T X_e with a fixed 512-token split order (offs: int64 device [E+1])."""
    T, N = G.shape
    K = X.shape[1]
    E = offs.numel() - 1
    if ws is None:
        ws = workspace(wgrad_workspace_bytes(E, N, K), G.device, stream)
    _check("dgr_grouped_wgrad_accumulate", lib().dgr_grouped_wgrad_accumulate(
        _ptr(G), _ptr(X), _ptr(offs), E, T, N, K, _ptr(main_grad), chunk_tokens, _ptr(ws), ws.numel(),
        _stream(stream)))
    return main_grad


def dbias_workspace_bytes(T: int, H: int, E: int, tile_rows: int = 128) -> int:
    return int(lib().dgr_dbias_workspace_bytes(T, H, E, tile_rows))


def grouped_dbias(dY: torch.Tensor, offs: torch.Tensor, out: torch.Tensor, *, accumulate: bool = False,
                  tile_rows: int = 128, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[e] (+)= ordered column sum of dY over expert e's rows offs[e] .. offs[e+1]-1
    (offs: int64 device [E+1]; out: fp32 [E, H])."""
    T, H = dY.shape
    E = offs.numel() - 1
    if out.dim() != 2 or out.shape != (E, H) or out.dtype != torch.float32 or offs.dtype != torch.int64:
        raise ValueError("dY [T, H], offs int64 [E+1], out fp32 [E, H] expected")
    if ws is None:
        ws = workspace(dbias_workspace_bytes(T, H, E, tile_rows), dY.device, stream)
    _check("dgr_grouped_dbias", lib().dgr_grouped_dbias(
        _ptr(dY), _dtype(dY), T, H, dY.stride(0), _ptr(offs), E, _ptr(out), out.stride(0), int(accumulate),
        tile_rows, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def topk_canonicalize(ids: torch.Tensor, logits: torch.Tensor, out_ids: torch.Tensor | None = None,
                      out_logits: torch.Tensor | None = None, probs: torch.Tensor | None = None, *,
                      stream=None):
    """Per row: slots sorted stably by id (padding, id < 0, last), logits permuted alike, softmax of
    the valid slots recomputed in that order. ids int32 [R, K], logits fp32 [R, K]."""
    if ids.dim() != 2 or ids.dtype != torch.int32 or logits.shape != ids.shape or logits.dtype != torch.float32:
        raise ValueError("ids int32 [R, K] and logits fp32 [R, K] expected")
    R, K = ids.shape
    with torch.cuda.stream(stream) if stream is not None else _nullcontext():  # outputs live on the call's stream
        out_ids = torch.empty_like(ids) if out_ids is None else out_ids
        out_logits = torch.empty_like(logits) if out_logits is None else out_logits
        probs = torch.empty_like(logits) if probs is None else probs
    if R == 0:  # no rows: nothing is read or written, and an empty tensor's strides say nothing
        _check("dgr_topk_canonicalize", lib().dgr_topk_canonicalize(
            _ptr(ids), K, _ptr(logits), K, 0, K, _ptr(out_ids), _ptr(out_logits), _ptr(probs), K,
            _stream(stream)))
        return out_ids, out_logits, probs
    ld = out_ids.stride(0)
    if out_logits.stride(0) != ld or probs.stride(0) != ld or any(t.stride(1) != 1 for t in
                                                                  (ids, logits, out_ids, out_logits, probs)):
        raise ValueError("outputs must share one row stride; rows contiguous")
    _check("dgr_topk_canonicalize", lib().dgr_topk_canonicalize(
        _ptr(ids), ids.stride(0), _ptr(logits), logits.stride(0), R, K, _ptr(out_ids), _ptr(out_logits),
        _ptr(probs), ld, _stream(stream)))
    return out_ids, out_logits, probs


def aux_loss_workspace_bytes(N: int) -> int:
    return int(lib().dgr_aux_loss_workspace_bytes(N))


def aux_loss(probs: torch.Tensor, tokens_per_expert: torch.Tensor, scale: float, out: torch.Tensor | None = None, *,
             ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[0] = RN(scale * S), S the canonical sum of probs * tokens_per_expert (each token's row dot,
    then the column sum over tokens). probs fp32 [N, E]; tokens_per_expert int32 [E] on the device."""
    if probs.dim() != 2 or probs.dtype != torch.float32 or tokens_per_expert.dtype != torch.int32:
        raise ValueError("probs fp32 [N, E] and tokens_per_expert int32 [E] expected")
    N, E = probs.shape
    if tokens_per_expert.shape != (E,) or probs.stride(1) != 1:
        raise ValueError("tokens_per_expert [E] and rows of probs contiguous expected")
    if out is None:
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():  # on the call's stream
            out = torch.empty(1, dtype=torch.float32, device=probs.device)
    if ws is None:
        ws = workspace(aux_loss_workspace_bytes(N), probs.device, stream)
    _check("dgr_aux_loss", lib().dgr_aux_loss(
        _ptr(probs), N, E, probs.stride(0), _ptr(tokens_per_expert), float(scale), _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def dsrelu_dprob_workspace_bytes(T: int, N: int) -> int:
    return int(lib().dgr_dsrelu_dprob_workspace_bytes(T, N))


def dsrelu_dprob(A: torch.Tensor, B: torch.Tensor, offs: torch.Tensor, dY: torch.Tensor, dprob: torch.Tensor, *,
                 accumulate: bool = False, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dprob[m] (+)= fold over N-tiles of pw_128(RN(dY * RN(relu(C)^2))), C = A_e B_e on the tensor
    cores (never written). A bf16 [T, K], B bf16 [E, K, N], offs int64 device [E+1], dY bf16 [T, N]."""
    T, K = A.shape
    E, K2, N = B.shape
    if (A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or dY.dtype != torch.bfloat16 or K2 != K or
            dY.shape != (T, N) or offs.shape != (E + 1,) or dprob.shape != (T,) or dprob.dtype != torch.float32):
        raise ValueError("A [T, K], B [E, K, N], dY [T, N] bf16, offs int64 [E+1], dprob fp32 [T] expected")
    if not (A.is_contiguous() and B.is_contiguous() and dY.is_contiguous()):
        raise ValueError("A, B and dY must be contiguous")
    if ws is None:
        ws = workspace(dsrelu_dprob_workspace_bytes(T, N), A.device, stream)
    _check("dgr_dsrelu_dprob", lib().dgr_dsrelu_dprob(
        _ptr(A), _ptr(B), _ptr(offs), E, T, K, N, _ptr(dY), _ptr(dprob), int(accumulate), _ptr(ws), ws.numel(),
        _stream(stream)))
    return dprob
