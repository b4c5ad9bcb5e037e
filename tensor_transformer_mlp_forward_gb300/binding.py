"""ctypes binding of ``libtpmlp.so`` (declared in include/tpmlp.h).

Argument marshalling only: each function checks that the tensors are
contiguous CUDA bfloat16 (or float32) tensors of the right shape, allocates
the outputs the caller did not pass, and calls the C entry point of the same
name on the current CUDA stream.  Every step of the computation runs in the
library's kernels; there is no other code path.  A missing library raises.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtpmlp.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "tpmlp.h")

TPMLP_OK = 0
TPMLP_ERR_NULL = 1
TPMLP_ERR_SHAPE = 2
TPMLP_ERR_ALIGN = 3
TPMLP_ERR_WORKSPACE = 4
TPMLP_ERR_LAUNCH = 5
TPMLP_ERR_DEVICE_TIMEOUT = 6
TPMLP_ERR_UNSUPPORTED = 7


class TpMlpError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed: status {status} ({message})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_S = ctypes.c_size_t
_D = ctypes.c_double
_U64 = ctypes.c_uint64

_SIGNATURES = {
    "tp_mlp_split_workspace_bytes": ([_I] * 4, _S),
    "tp_mlp_forward_workspace_bytes": ([_I] * 4, _S),
    "tp_mlp_forward": ([_P] * 6 + [_I] * 4 + [_P] * 3 + [_P, _S, _P], _I),
    "tp_mlp_backward_workspace_bytes": ([_I] * 4, _S),
    "tp_mlp_backward": ([_P] * 6 + [_I] * 4 + [_P] * 6 + [_S, _P], _I),
    "tp_mlp_column_gelu": ([_P] * 3 + [_I] * 4 + [_P] * 2 + [_P], _I),
    "tp_mlp_row_sum": ([_P] * 4 + [_I] * 4 + [_P] + [_P, _S, _P], _I),
    "tp_mlp_bias_grad_workspace_floats": ([_I, _I], _S),
    "tp_mlp_bias_grad": ([_P, _I, _I, _P, _P, _P], _I),
    "tp_mlp_bias_grad_noalloc": ([_P, _I, _I, _P, _P], _I),
    "tp_mlp_bias_grad_noalloc_max_floats": ([], _S),
    "tp_mlp_dgelu_partial_floats": ([_I, _I], _S),
    "tp_mlp_dgelu": ([_P] * 3 + [_I] * 4 + [_P] * 3 + [_P], _I),
    "tp_mlp_dx": ([_P] * 2 + [_I] * 4 + [_P] + [_P, _S, _P], _I),
    "tp_mlp_dA": ([_P] * 2 + [_I] * 4 + [_P] + [_P], _I),
    "tp_mlp_dB": ([_P] * 2 + [_I] * 4 + [_P] + [_P], _I),
    "tp_weight_grad_kmajor": ([_I, _I], _I),
    "tp_weight_grad_workspace_bytes": ([_I, _I, _I], _S),
    "tp_mlp_dA_ws": ([_P] * 2 + [_I] * 4 + [_P] + [_P, _S, _P], _I),
    "tp_mlp_dB_ws": ([_P] * 2 + [_I] * 4 + [_P] + [_P, _S, _P], _I),
    "tp_transpose": ([_P, _I, _I, _P, _I, _P], _I),
    "tp_mlp_dA_kmajor": ([_P] * 2 + [_I] * 5 + [_P] + [_P], _I),
    "tp_mlp_dB_kmajor": ([_P] * 2 + [_I] * 5 + [_P] + [_P], _I),
    "tp_mlp_forward_recompute_workspace_bytes": ([_I] * 4, _S),
    "tp_mlp_forward_recompute": ([_P] * 6 + [_I] * 4 + [_P] + [_P, _S, _P], _I),
    "tp_mlp_backward_recompute_workspace_bytes": ([_I] * 4, _S),
    "tp_mlp_backward_recompute": ([_P] * 5 + [_I] * 4 + [_P] * 6 + [_S, _P], _I),
    "tp_mlp_row_sum_dropout": ([_P] * 4 + [_I] * 4 + [_D, _U64, _U64] + [_P] + [_P, _S, _P], _I),
    "tp_mlp_forward_dropout": ([_P] * 6 + [_I] * 4 + [_D, _U64, _U64] + [_P] * 3 + [_P, _S, _P],
                               _I),
    "tp_mlp_dropout_grad": ([_P, _I, _I, _D, _U64, _U64, _P, _P], _I),
    "tp_mlp_backward_dropout_workspace_bytes": ([_I] * 4, _S),
    "tp_mlp_backward_dropout": ([_P] * 6 + [_I] * 4 + [_D, _U64, _U64] + [_P] * 6 + [_S, _P],
                                _I),
    "tp_ln_residual_forward": ([_P] * 4 + [_I, _I, ctypes.c_float] + [_P] * 4 + [_P], _I),
    "tp_ln_residual_backward_workspace_floats": ([_I, _I], _S),
    "tp_ln_residual_backward": ([_P] * 7 + [_I, _I] + [_P] * 4 + [_P], _I),
    "tp_attn_qkv": ([_P] * 3 + [_I] * 2 + [_P, _P], _I),
    "tp_attn_core_workspace_bytes": ([_I] * 4, _S),
    "tp_attn_core_forward": ([_P] + [_I] * 4 + [_P] * 2 + [_P, _S, _P], _I),
    "tp_attn_core_backward": ([_P] * 4 + [_I] * 4 + [_P] * 2 + [_P, _S, _P], _I),
    "tp_attn_forward_workspace_bytes": ([_I] * 5, _S),
    "tp_attn_forward": ([_P] * 6 + [_I] * 5 + [_P] * 4 + [_P, _S, _P], _I),
    "tp_attn_backward_workspace_bytes": ([_I] * 5, _S),
    "tp_attn_backward": ([_P] * 7 + [_I] * 5 + [_P] * 5 + [_P, _S, _P], _I),
    "tp_mlp_status_string": ([_I], ctypes.c_char_p),
    "tpmlp_status_string": ([_I], ctypes.c_char_p),
    "tpmlp_last_cuda_error": ([], _I),
    "tpmlp_device_status": ([], _I),
    "tpmlp_device_wait_site": ([], _I),
    "tpmlp_last_launch_count": ([], _I),
    "tpmlp_selftest_bounded_wait": ([_I, _P], _I),
    "tpmlp_set_cta_pair_mode": ([_I], _I),
    "tpmlp_set_epilogue_warps": ([_I], _I),
    "tpmlp_set_dependent_launch": ([_I], _I),
    "tpmlp_set_tile_scheduler": ([_I], _I),
    "tpmlp_set_wide_tiles": ([_I], _I),
}


def declared_functions(header: str = HEADER):
    """Names of the functions include/tpmlp.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(t\w+)\s*\(", text, flags=re.M)))


def lib(path: str = LIB_PATH):
    """The loaded library (loads on first use; raises if it was not built)."""
    global _lib
    if _lib is None or path != LIB_PATH:
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        if path != LIB_PATH:
            return L
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().tp_mlp_status_string(status).decode()


def _check(fn: str, status: int):
    if status != TPMLP_OK:
        msg = status_string(status)
        if status == TPMLP_ERR_LAUNCH:
            msg += f"; CUDA error {lib().tpmlp_last_cuda_error()}"
        raise TpMlpError(fn, status, msg)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(x: Optional[torch.Tensor], name: str, shape=None, dtype=torch.bfloat16):
    if x is None:
        raise ValueError(f"{name} is required")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")
    return x.data_ptr()


def _out(x, shape, like: torch.Tensor, dtype=torch.bfloat16):
    if x is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return x


def last_launch_count() -> int:
    return int(lib().tpmlp_last_launch_count())


def set_cta_pair_mode(mode: int) -> int:
    """0 single-CTA GEMMs, 1 CTA pairs from 32 output tiles of 256 x 256 up
    (default), 2 CTA pairs always.  Returns the previous mode."""
    prev = int(lib().tpmlp_set_cta_pair_mode(mode))
    if prev < 0:
        raise ValueError(f"invalid mode {mode}")
    return prev


def set_epilogue_warps(mode: int) -> int:
    """0 by the reduction's length (default), 4 or 8 epilogue warps always.
    Returns the previous mode."""
    prev = int(lib().tpmlp_set_epilogue_warps(mode))
    if prev < 0:
        raise ValueError(f"invalid mode {mode}")
    return prev


def set_dependent_launch(mode: int) -> int:
    """Which kernels start as programmatic dependents of the kernel before
    them: bit 0 the GEMMs, bit 1 the others (3, the default: both; 0: plain
    stream order).  Returns the previous mode."""
    prev = int(lib().tpmlp_set_dependent_launch(mode))
    if prev < 0:
        raise ValueError(f"invalid mode {mode}")
    return prev


def set_wide_tiles(mode: int) -> int:
    """0: 256 x 256 GEMM tiles per CTA pair (default); 1: 256 x 512 for the
    K-major plain-store GEMMs whose reduction is not split.  Returns the
    previous mode."""
    prev = int(lib().tpmlp_set_wide_tiles(mode))
    if prev < 0:
        raise ValueError(f"invalid mode {mode}")
    return prev


def set_tile_scheduler(mode: int) -> int:
    """0: persistent GEMM grids with a static tile assignment; 1: dynamic
    tiles through cluster launch control; 2 (default): dynamic for long
    reductions only.  Returns the previous mode."""
    prev = int(lib().tpmlp_set_tile_scheduler(mode))
    if prev < 0:
        raise ValueError(f"invalid mode {mode}")
    return prev


def device_status() -> int:
    return int(lib().tpmlp_device_status())


def device_wait_site() -> int:
    """Site code of the first device wait that gave up since the last read."""
    return int(lib().tpmlp_device_wait_site())


def tp_mlp_column_gelu(X, A, b1, t: int, Z=None, H=None, stream=None, want_z=True):
    """Z, H of step a2; with want_z=False only H is written (Z is None)."""
    T, h = X.shape
    F = A.shape[1]
    Z = _out(Z, (T, F), X) if want_z else None
    H = _out(H, (T, F), X)
    _check("tp_mlp_column_gelu", lib().tp_mlp_column_gelu(
        _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)), _ptr(b1, "b1", (F,)), T, h, F, t,
        _ptr(Z, "Z", (T, F)) if want_z else None, _ptr(H, "H", (T, F)), _stream(stream)))
    return Z, H


def split_workspace_bytes(T: int, h: int, F: int, t: int) -> int:
    return int(lib().tp_mlp_split_workspace_bytes(T, h, F, t))


def _workspace(ws, need: int, like: torch.Tensor):
    """The caller's workspace, or a fresh one of `need` bytes (None if 0)."""
    if ws is None and need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device=like.device)
    if ws is None:
        return None, 0
    return _ptr(ws, "workspace", None, torch.uint8), ws.numel()


def tp_mlp_row_sum(H, B, b2, residual, t: int, Y=None, workspace=None, stream=None):
    T, F = H.shape
    h = B.shape[1]
    Y = _out(Y, (T, h), H)
    wp, wn = _workspace(workspace, split_workspace_bytes(T, h, F, t), H)
    _check("tp_mlp_row_sum", lib().tp_mlp_row_sum(
        _ptr(H, "H", (T, F)), _ptr(B, "B", (F, h)), _ptr(b2, "b2", (h,)),
        _ptr(residual, "residual", (T, h)), T, h, F, t, _ptr(Y, "Y", (T, h)), wp, wn,
        _stream(stream)))
    return Y


def tp_mlp_forward(X, A, b1, B, b2, residual, t: int, Y=None, Z=None, H=None, workspace=None,
                   stream=None):
    """Y, Z, H of the block (Z, H saved for the backward pass)."""
    T, h = X.shape
    F = A.shape[1]
    Y = _out(Y, (T, h), X)
    Z = _out(Z, (T, F), X)
    H = _out(H, (T, F), X)
    wp, wn = _workspace(workspace, int(lib().tp_mlp_forward_workspace_bytes(T, h, F, t)), X)
    _check("tp_mlp_forward", lib().tp_mlp_forward(
        _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)), _ptr(b1, "b1", (F,)), _ptr(B, "B", (F, h)),
        _ptr(b2, "b2", (h,)), _ptr(residual, "residual", (T, h)), T, h, F, t,
        _ptr(Y, "Y", (T, h)), _ptr(Z, "Z", (T, F)), _ptr(H, "H", (T, F)), wp, wn,
        _stream(stream)))
    return Y, Z, H


def tp_mlp_backward_workspace_bytes(T: int, h: int, F: int, t: int) -> int:
    return int(lib().tp_mlp_backward_workspace_bytes(T, h, F, t))


def tp_mlp_backward(dY, X, A, B, Z, H, t: int, dX=None, dA=None, dB=None, db1=None, db2=None,
                    workspace=None, stream=None):
    """dX, dA, dB (bf16) and db1, db2 (float32) of the block."""
    T, h = X.shape
    F = A.shape[1]
    dX = _out(dX, (T, h), X)
    dA = _out(dA, (h, F), X)
    dB = _out(dB, (F, h), X)
    db1 = _out(db1, (F,), X, torch.float32)
    db2 = _out(db2, (h,), X, torch.float32)
    need = tp_mlp_backward_workspace_bytes(T, h, F, t)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    _check("tp_mlp_backward", lib().tp_mlp_backward(
        _ptr(dY, "dY", (T, h)), _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)), _ptr(B, "B", (F, h)),
        _ptr(Z, "Z", (T, F)), _ptr(H, "H", (T, F)), T, h, F, t,
        _ptr(dX, "dX", (T, h)), _ptr(dA, "dA", (h, F)), _ptr(dB, "dB", (F, h)),
        _ptr(db1, "db1", (F,), torch.float32), _ptr(db2, "db2", (h,), torch.float32),
        _ptr(workspace, "workspace", None, torch.uint8), workspace.numel(), _stream(stream)))
    return dX, dA, dB, db1, db2


def tp_mlp_forward_recompute(X, A, b1, B, b2, residual, t: int, Y=None, workspace=None,
                             stream=None):
    """Y of the block; nothing is saved for the backward pass but X."""
    T, h = X.shape
    F = A.shape[1]
    Y = _out(Y, (T, h), X)
    need = int(lib().tp_mlp_forward_recompute_workspace_bytes(T, h, F, t))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    _check("tp_mlp_forward_recompute", lib().tp_mlp_forward_recompute(
        _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)), _ptr(b1, "b1", (F,)), _ptr(B, "B", (F, h)),
        _ptr(b2, "b2", (h,)), _ptr(residual, "residual", (T, h)), T, h, F, t,
        _ptr(Y, "Y", (T, h)), _ptr(workspace, "workspace", None, torch.uint8),
        workspace.numel(), _stream(stream)))
    return Y


def tp_mlp_backward_recompute(dY, X, A, b1, B, t: int, dX=None, dA=None, dB=None, db1=None,
                              db2=None, workspace=None, stream=None):
    """Gradients of the block from its input X (Z and H recomputed)."""
    T, h = X.shape
    F = A.shape[1]
    dX = _out(dX, (T, h), X)
    dA = _out(dA, (h, F), X)
    dB = _out(dB, (F, h), X)
    db1 = _out(db1, (F,), X, torch.float32)
    db2 = _out(db2, (h,), X, torch.float32)
    need = int(lib().tp_mlp_backward_recompute_workspace_bytes(T, h, F, t))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    _check("tp_mlp_backward_recompute", lib().tp_mlp_backward_recompute(
        _ptr(dY, "dY", (T, h)), _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)),
        _ptr(b1, "b1", (F,)), _ptr(B, "B", (F, h)), T, h, F, t,
        _ptr(dX, "dX", (T, h)), _ptr(dA, "dA", (h, F)), _ptr(dB, "dB", (F, h)),
        _ptr(db1, "db1", (F,), torch.float32), _ptr(db2, "db2", (h,), torch.float32),
        _ptr(workspace, "workspace", None, torch.uint8), workspace.numel(), _stream(stream)))
    return dX, dA, dB, db1, db2


def tp_mlp_row_sum_dropout(H, B, b2, residual, t: int, p: float, seed: int, offset: int = 0,
                           Y=None, workspace=None, stream=None):
    """a3 with dropout before the residual add (keep drawn from seed, offset)."""
    T, F = H.shape
    h = B.shape[1]
    Y = _out(Y, (T, h), H)
    wp, wn = _workspace(workspace, split_workspace_bytes(T, h, F, t), H)
    _check("tp_mlp_row_sum_dropout", lib().tp_mlp_row_sum_dropout(
        _ptr(H, "H", (T, F)), _ptr(B, "B", (F, h)), _ptr(b2, "b2", (h,)),
        _ptr(residual, "residual", (T, h)), T, h, F, t, float(p), int(seed), int(offset),
        _ptr(Y, "Y", (T, h)), wp, wn, _stream(stream)))
    return Y


def tp_mlp_forward_dropout(X, A, b1, B, b2, residual, t: int, p: float, seed: int,
                           offset: int = 0, Y=None, Z=None, H=None, workspace=None, stream=None):
    """Y, Z, H of the block with dropout before the residual add."""
    T, h = X.shape
    F = A.shape[1]
    Y = _out(Y, (T, h), X)
    Z = _out(Z, (T, F), X)
    H = _out(H, (T, F), X)
    wp, wn = _workspace(workspace, int(lib().tp_mlp_forward_workspace_bytes(T, h, F, t)), X)
    _check("tp_mlp_forward_dropout", lib().tp_mlp_forward_dropout(
        _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)), _ptr(b1, "b1", (F,)), _ptr(B, "B", (F, h)),
        _ptr(b2, "b2", (h,)), _ptr(residual, "residual", (T, h)), T, h, F, t, float(p),
        int(seed), int(offset), _ptr(Y, "Y", (T, h)), _ptr(Z, "Z", (T, F)),
        _ptr(H, "H", (T, F)), wp, wn, _stream(stream)))
    return Y, Z, H


def tp_mlp_dropout_grad(dY, p: float, seed: int, offset: int = 0, dP=None, stream=None):
    """dP = keep * dY / (1 - p) (bf16)."""
    T, h = dY.shape
    dP = _out(dP, (T, h), dY)
    _check("tp_mlp_dropout_grad", lib().tp_mlp_dropout_grad(
        _ptr(dY, "dY", (T, h)), T, h, float(p), int(seed), int(offset), _ptr(dP, "dP", (T, h)),
        _stream(stream)))
    return dP


def tp_mlp_backward_dropout_workspace_bytes(T: int, h: int, F: int, t: int) -> int:
    return int(lib().tp_mlp_backward_dropout_workspace_bytes(T, h, F, t))


def tp_mlp_backward_dropout(dY, X, A, B, Z, H, t: int, p: float, seed: int, offset: int = 0,
                            dX=None, dA=None, dB=None, db1=None, db2=None, workspace=None,
                            stream=None):
    """dX, dA, dB (bf16) and db1, db2 (float32) of the block with dropout."""
    T, h = X.shape
    F = A.shape[1]
    dX = _out(dX, (T, h), X)
    dA = _out(dA, (h, F), X)
    dB = _out(dB, (F, h), X)
    db1 = _out(db1, (F,), X, torch.float32)
    db2 = _out(db2, (h,), X, torch.float32)
    need = tp_mlp_backward_dropout_workspace_bytes(T, h, F, t)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    _check("tp_mlp_backward_dropout", lib().tp_mlp_backward_dropout(
        _ptr(dY, "dY", (T, h)), _ptr(X, "X", (T, h)), _ptr(A, "A", (h, F)), _ptr(B, "B", (F, h)),
        _ptr(Z, "Z", (T, F)), _ptr(H, "H", (T, F)), T, h, F, t, float(p), int(seed),
        int(offset), _ptr(dX, "dX", (T, h)), _ptr(dA, "dA", (h, F)), _ptr(dB, "dB", (F, h)),
        _ptr(db1, "db1", (F,), torch.float32), _ptr(db2, "db2", (h,), torch.float32),
        _ptr(workspace, "workspace", None, torch.uint8), workspace.numel(), _stream(stream)))
    return dX, dA, dB, db1, db2


def tp_mlp_bias_grad(G, db=None, partial=None, stream=None):
    T, n = G.shape
    db = _out(db, (n,), G, torch.float32)
    need = max(1, int(lib().tp_mlp_bias_grad_workspace_floats(T, n)))
    if partial is None:
        partial = torch.empty(need, dtype=torch.float32, device=G.device)
    if partial.numel() < need:
        raise ValueError(f"partial holds {partial.numel()} floats, {need} needed")
    _check("tp_mlp_bias_grad", lib().tp_mlp_bias_grad(
        _ptr(G, "G", (T, n)), T, n, _ptr(db, "db", (n,), torch.float32),
        _ptr(partial, "partial", None, torch.float32), _stream(stream)))
    return db


def tp_mlp_bias_grad_noalloc(G, db=None, stream=None):
    """Column sums of G [T, n] with the partial sums in the library's own
    fixed device array, for callers that cannot allocate scratch memory
    (only `db` is allocated here, and only when the caller did not pass it)."""
    T, n = G.shape
    db = _out(db, (n,), G, torch.float32)
    _check("tp_mlp_bias_grad_noalloc", lib().tp_mlp_bias_grad_noalloc(
        _ptr(G, "G", (T, n)) if T else None, T, n, _ptr(db, "db", (n,), torch.float32),
        _stream(stream)))
    return db


def tp_mlp_dgelu(dY, B, Z, t: int, dZ=None, db1=None, partial=None, stream=None):
    T, h = dY.shape
    F = B.shape[0]
    dZ = _out(dZ, (T, F), dY)
    db1 = _out(db1, (F,), dY, torch.float32)
    if partial is None:
        partial = torch.empty(max(1, int(lib().tp_mlp_dgelu_partial_floats(T, F))),
                              dtype=torch.float32, device=dY.device)
    _check("tp_mlp_dgelu", lib().tp_mlp_dgelu(
        _ptr(dY, "dY", (T, h)), _ptr(B, "B", (F, h)), _ptr(Z, "Z", (T, F)), T, h, F, t,
        _ptr(dZ, "dZ", (T, F)), _ptr(db1, "db1", (F,), torch.float32),
        _ptr(partial, "partial", None, torch.float32), _stream(stream)))
    return dZ, db1


def tp_mlp_dx(dZ, A, t: int, dX=None, workspace=None, stream=None):
    T, F = dZ.shape
    h = A.shape[0]
    dX = _out(dX, (T, h), dZ)
    wp, wn = _workspace(workspace, split_workspace_bytes(T, h, F, t), dZ)
    _check("tp_mlp_dx", lib().tp_mlp_dx(
        _ptr(dZ, "dZ", (T, F)), _ptr(A, "A", (h, F)), T, h, F, t, _ptr(dX, "dX", (T, h)), wp, wn,
        _stream(stream)))
    return dX


def tp_mlp_dA(X, dZ, t: int, dA=None, stream=None):
    T, h = X.shape
    F = dZ.shape[1]
    dA = _out(dA, (h, F), X)
    _check("tp_mlp_dA", lib().tp_mlp_dA(
        _ptr(X, "X", (T, h)), _ptr(dZ, "dZ", (T, F)), T, h, F, t, _ptr(dA, "dA", (h, F)),
        _stream(stream)))
    return dA


def tp_mlp_dB(H, dY, t: int, dB=None, stream=None):
    T, F = H.shape
    h = dY.shape[1]
    dB = _out(dB, (F, h), H)
    _check("tp_mlp_dB", lib().tp_mlp_dB(
        _ptr(H, "H", (T, F)), _ptr(dY, "dY", (T, h)), T, h, F, t, _ptr(dB, "dB", (F, h)),
        _stream(stream)))
    return dB


def weight_grad_workspace_bytes(T: int, M: int, N: int) -> int:
    """Workspace that lets an M x N weight gradient split its T-token
    reduction over idle SM pairs (0: it is computed whole)."""
    return int(lib().tp_weight_grad_workspace_bytes(T, M, N))


def tp_mlp_dA_ws(X, dZ, t: int, dA=None, workspace=None, stream=None):
    """tp_mlp_dA with a workspace for the split reduction (allocated here
    when None and the shape takes a split)."""
    T, h = X.shape
    F = dZ.shape[1]
    dA = _out(dA, (h, F), X)
    wp, wn = _workspace(workspace, weight_grad_workspace_bytes(T, h, F) if t == 1 else 0, X)
    _check("tp_mlp_dA_ws", lib().tp_mlp_dA_ws(
        _ptr(X, "X", (T, h)), _ptr(dZ, "dZ", (T, F)), T, h, F, t, _ptr(dA, "dA", (h, F)),
        wp, wn, _stream(stream)))
    return dA


def tp_mlp_dB_ws(H, dY, t: int, dB=None, workspace=None, stream=None):
    """tp_mlp_dB with a workspace for the split reduction (allocated here
    when None and the shape takes a split)."""
    T, F = H.shape
    h = dY.shape[1]
    dB = _out(dB, (F, h), H)
    wp, wn = _workspace(workspace, weight_grad_workspace_bytes(T, F, h) if t == 1 else 0, H)
    _check("tp_mlp_dB_ws", lib().tp_mlp_dB_ws(
        _ptr(H, "H", (T, F)), _ptr(dY, "dY", (T, h)), T, h, F, t, _ptr(dB, "dB", (F, h)),
        wp, wn, _stream(stream)))
    return dB


def pitch(rows: int) -> int:
    """Row pitch tp_transpose needs at least: rows rounded up to 8."""
    return (rows + 7) // 8 * 8


def weight_grad_kmajor(M: int, N: int) -> bool:
    """Whether the composite backward calls compute an M x N weight gradient
    from transposed operands (tp_transpose + tp_mlp_dA_kmajor/_dB_kmajor)."""
    return bool(lib().tp_weight_grad_kmajor(M, N))


def tp_transpose(x, ld: Optional[int] = None, out=None, stream=None):
    """out[c, r] = x[r, c] for x [rows, cols]; out is [cols, ld] (ld defaults to
    pitch(rows)); columns rows .. pitch(rows) - 1 of out are zeroed."""
    rows, cols = x.shape
    ld = pitch(rows) if ld is None else ld
    out = _out(out, (cols, ld), x)
    _check("tp_transpose", lib().tp_transpose(
        _ptr(x, "x", (rows, cols)), rows, cols, _ptr(out, "out", (cols, ld)), ld, _stream(stream)))
    return out


def tp_mlp_dA_kmajor(Xt, dZt, T: int, t: int, dA=None, stream=None):
    """dA from Xt = X^T [h, ldT] and dZt = dZ^T [F, ldT] (tp_transpose's output)."""
    h, ldT = Xt.shape
    F = dZt.shape[0]
    dA = _out(dA, (h, F), Xt)
    _check("tp_mlp_dA_kmajor", lib().tp_mlp_dA_kmajor(
        _ptr(Xt, "Xt", (h, ldT)), _ptr(dZt, "dZt", (F, ldT)), T, ldT, h, F, t,
        _ptr(dA, "dA", (h, F)), _stream(stream)))
    return dA


def tp_mlp_dB_kmajor(Ht, dYt, T: int, t: int, dB=None, stream=None):
    """dB from Ht = H^T [F, ldT] and dYt = dY^T [h, ldT] (tp_transpose's output)."""
    F, ldT = Ht.shape
    h = dYt.shape[0]
    dB = _out(dB, (F, h), Ht)
    _check("tp_mlp_dB_kmajor", lib().tp_mlp_dB_kmajor(
        _ptr(Ht, "Ht", (F, ldT)), _ptr(dYt, "dYt", (h, ldT)), T, ldT, h, F, t,
        _ptr(dB, "dB", (F, h)), _stream(stream)))
    return dB


def tp_ln_residual_forward(a, r, gamma, beta, eps: float = 1e-5, X=None, s=None, mean=None,
                           rstd=None, want_s: bool = True, stream=None):
    """X, s, mean, rstd of s = a + r, X = LayerNorm(s) * gamma + beta."""
    T, h = a.shape
    X = _out(X, (T, h), a)
    if want_s:
        s = _out(s, (T, h), a)
    mean = _out(mean, (T,), a, torch.float32)
    rstd = _out(rstd, (T,), a, torch.float32)
    _check("tp_ln_residual_forward", lib().tp_ln_residual_forward(
        _ptr(a, "a", (T, h)), _ptr(r, "r", (T, h)), _ptr(gamma, "gamma", (h,)),
        _ptr(beta, "beta", (h,)), T, h, eps, _ptr(X, "X", (T, h)),
        _ptr(s, "s", (T, h)) if s is not None else None, _ptr(mean, "mean", (T,), torch.float32),
        _ptr(rstd, "rstd", (T,), torch.float32), _stream(stream)))
    return X, s, mean, rstd


def tp_ln_residual_backward(dX, dres, a, r, gamma, mean, rstd, ds=None, dgamma=None, dbeta=None,
                            partial=None, stream=None):
    """ds (= d a = d r), dgamma, dbeta of the residual add + LayerNorm."""
    T, h = a.shape
    ds = _out(ds, (T, h), a)
    dgamma = _out(dgamma, (h,), a, torch.float32)
    dbeta = _out(dbeta, (h,), a, torch.float32)
    if partial is None:
        partial = torch.empty(max(1, int(lib().tp_ln_residual_backward_workspace_floats(T, h))),
                              dtype=torch.float32, device=a.device)
    _check("tp_ln_residual_backward", lib().tp_ln_residual_backward(
        _ptr(dX, "dX", (T, h)), _ptr(dres, "dres", (T, h)) if dres is not None else None,
        _ptr(a, "a", (T, h)), _ptr(r, "r", (T, h)), _ptr(gamma, "gamma", (h,)),
        _ptr(mean, "mean", (T,), torch.float32), _ptr(rstd, "rstd", (T,), torch.float32), T, h,
        _ptr(ds, "ds", (T, h)), _ptr(dgamma, "dgamma", (h,), torch.float32),
        _ptr(dbeta, "dbeta", (h,), torch.float32), _ptr(partial, "partial", None, torch.float32),
        _stream(stream)))
    return ds, dgamma, dbeta


def selftest_bounded_wait(timeout_us: int, stream=None) -> int:
    """Runs the bounded-wait self-test kernel and returns the device status."""
    _check("tpmlp_selftest_bounded_wait",
           lib().tpmlp_selftest_bounded_wait(timeout_us, _stream(stream)))
    return device_status()


# ------------------------------------------------------------ attention block

def tp_attn_qkv(X, Wqkv, bqkv, QKV=None, stream=None):
    """QKV = X Wqkv + bqkv: [T, 3h] with columns [Q | K | V]."""
    T, h = X.shape
    QKV = _out(QKV, (T, 3 * h), X)
    _check("tp_attn_qkv", lib().tp_attn_qkv(
        _ptr(X, "X", (T, h)) if T else None, _ptr(Wqkv, "Wqkv", (h, 3 * h)),
        _ptr(bqkv, "bqkv", (3 * h,)), T, h, _ptr(QKV, "QKV", (T, 3 * h)) if T else None,
        _stream(stream)))
    return QKV


def tp_attn_core_forward(QKV, nb: int, nh: int, O=None, lse=None, workspace=None, stream=None):
    """O [T, h] (bf16) and lse [nh, T] (float32, log2 domain) of causal
    attention over nb sequences of T / nb tokens."""
    T, h3 = QKV.shape
    h = h3 // 3
    s = T // nb if nb else 1
    O = _out(O, (T, h), QKV)
    lse = _out(lse, (nh, T), QKV, torch.float32)
    wp, wn = _workspace(workspace, int(lib().tp_attn_core_workspace_bytes(nb, s, h, nh)), QKV)
    _check("tp_attn_core_forward", lib().tp_attn_core_forward(
        _ptr(QKV, "QKV", (T, 3 * h)) if T else None, nb, s, h, nh,
        _ptr(O, "O", (T, h)) if T else None, _ptr(lse, "lse", (nh, T), torch.float32) if T else None,
        wp, wn, _stream(stream)))
    return O, lse


def tp_attn_core_backward(QKV, O, lse, dO, nb: int, nh: int, dQKV=None, delta=None,
                          workspace=None, stream=None):
    """dQKV [T, 3h] of causal attention given dO; delta [nh, T] is scratch."""
    T, h3 = QKV.shape
    h = h3 // 3
    s = T // nb if nb else 1
    dQKV = _out(dQKV, (T, 3 * h), QKV)
    delta = _out(delta, (nh, T), QKV, torch.float32)
    wp, wn = _workspace(workspace, int(lib().tp_attn_core_workspace_bytes(nb, s, h, nh)), QKV)
    _check("tp_attn_core_backward", lib().tp_attn_core_backward(
        _ptr(QKV, "QKV", (T, 3 * h)), _ptr(O, "O", (T, h)),
        _ptr(lse, "lse", (nh, T), torch.float32), _ptr(dO, "dO", (T, h)), nb, s, h, nh,
        _ptr(dQKV, "dQKV", (T, 3 * h)), _ptr(delta, "delta", (nh, T), torch.float32),
        wp, wn, _stream(stream)))
    return dQKV


def tp_attn_forward(X, Wqkv, bqkv, Wo, bo, residual, nb: int, nh: int, t: int, Y=None, QKV=None,
                    O=None, lse=None, workspace=None, stream=None):
    """Y of the head-parallel attention block, with QKV, O, lse saved for the
    backward pass."""
    T, h = X.shape
    s = T // nb if nb else 1
    Y = _out(Y, (T, h), X)
    QKV = _out(QKV, (T, 3 * h), X)
    O = _out(O, (T, h), X)
    lse = _out(lse, (nh, T), X, torch.float32)
    wp, wn = _workspace(workspace, int(lib().tp_attn_forward_workspace_bytes(nb, s, h, nh, t)), X)
    nz = T > 0
    _check("tp_attn_forward", lib().tp_attn_forward(
        _ptr(X, "X", (T, h)) if nz else None, _ptr(Wqkv, "Wqkv", (h, 3 * h)),
        _ptr(bqkv, "bqkv", (3 * h,)), _ptr(Wo, "Wo", (h, h)), _ptr(bo, "bo", (h,)),
        _ptr(residual, "residual", (T, h)) if nz else None, nb, s, h, nh, t,
        _ptr(Y, "Y", (T, h)) if nz else None, _ptr(QKV, "QKV", (T, 3 * h)) if nz else None,
        _ptr(O, "O", (T, h)) if nz else None,
        _ptr(lse, "lse", (nh, T), torch.float32) if nz else None, wp, wn, _stream(stream)))
    return Y, QKV, O, lse


def tp_attn_backward_workspace_bytes(nb: int, s: int, h: int, nh: int, t: int) -> int:
    return int(lib().tp_attn_backward_workspace_bytes(nb, s, h, nh, t))


def tp_attn_backward(dY, X, Wqkv, Wo, QKV, O, lse, nb: int, nh: int, t: int, dX=None, dWqkv=None,
                     dbqkv=None, dWo=None, dbo=None, workspace=None, stream=None):
    """dX, dWqkv, dWo (bf16) and dbqkv, dbo (float32) of the attention block
    (dX is the gradient through the block; the residual's is dY)."""
    T, h = X.shape
    s = T // nb if nb else 1
    dX = _out(dX, (T, h), X)
    dWqkv = _out(dWqkv, (h, 3 * h), X)
    dbqkv = _out(dbqkv, (3 * h,), X, torch.float32)
    dWo = _out(dWo, (h, h), X)
    dbo = _out(dbo, (h,), X, torch.float32)
    need = tp_attn_backward_workspace_bytes(nb, s, h, nh, t)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    nz = T > 0
    _check("tp_attn_backward", lib().tp_attn_backward(
        _ptr(dY, "dY", (T, h)) if nz else None, _ptr(X, "X", (T, h)) if nz else None,
        _ptr(Wqkv, "Wqkv", (h, 3 * h)), _ptr(Wo, "Wo", (h, h)),
        _ptr(QKV, "QKV", (T, 3 * h)) if nz else None, _ptr(O, "O", (T, h)) if nz else None,
        _ptr(lse, "lse", (nh, T), torch.float32) if nz else None, nb, s, h, nh, t,
        _ptr(dX, "dX", (T, h)) if nz else None, _ptr(dWqkv, "dWqkv", (h, 3 * h)),
        _ptr(dbqkv, "dbqkv", (3 * h,), torch.float32), _ptr(dWo, "dWo", (h, h)),
        _ptr(dbo, "dbo", (h,), torch.float32),
        _ptr(workspace, "workspace", None, torch.uint8), workspace.numel(), _stream(stream)))
    return dX, dWqkv, dbqkv, dWo, dbo
