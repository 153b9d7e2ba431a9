"""ctypes wrapper around the plain-C CPU oracle (``oracle/oracle.c``).

Test infrastructure: only the test suite, the package smoke check and the
benchmark's CPU-baseline leg import this package.  The CUDA library never
does, and this package imports nothing from it.

Arrays are numpy; fp16 data is passed as ``np.float16`` (binary16 bits).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, F64 = 0, 1, 2
FLAG_HASH = 1
STATUS_OOB = 1
SKIP_KEY = 0xFFFFFFFF

_P = ctypes.c_void_p
_lib = None
_override = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C99, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load(path: str):
    """Load an oracle shared object and declare its signatures."""
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def use(L) -> None:
    """Route the wrappers below to ``L`` (None restores the committed oracle)."""
    global _override
    _override = L


def lib():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        build()
        _lib = load(_LIB)
    return _lib


def _declare(L) -> None:
    L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_f64.restype = ctypes.c_double
    L.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    L.oracle_f64_to_f16.restype = ctypes.c_uint16
    L.oracle_emb_fwd.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 _P, _P, ctypes.c_int64, _P, ctypes.c_uint, _P]
    L.oracle_gram.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    L.oracle_interact_fwd.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, _P, ctypes.c_int]
    L.oracle_interact_bwd.argtypes = [_P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, _P, _P]
    L.oracle_round_f16.argtypes = [_P, _P, ctypes.c_int64]
    L.oracle_round_f16.restype = None
    L.oracle_mlp_fwd.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P, _P, ctypes.c_int, _P]
    L.oracle_emb_bwd_sgd.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P,
                                     ctypes.c_int64, _P, ctypes.c_float, ctypes.c_uint, _P,
                                     _P, _P]
    for f in ("oracle_emb_fwd", "oracle_gram", "oracle_interact_fwd", "oracle_interact_bwd",
              "oracle_emb_bwd_sgd"):
        getattr(L, f).restype = ctypes.c_int


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float16:
        return F16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def f16_to_f64(bits: int) -> float:
    return lib().oracle_f16_to_f64(int(bits))


def f64_to_f16(x: float) -> int:
    return int(lib().oracle_f64_to_f16(float(x)))


def emb_fwd(tables, row_base, F, D, B, indices, offsets, flags=0):
    """Pooled embeddings [B][F][D] in the table dtype, and the status word."""
    tables = _c(tables)
    row_base = _c(row_base, np.int64)
    indices = _c(indices, np.int32)
    offsets = _c(offsets, np.int32)
    pooled = np.zeros((B, F, D), dtype=tables.dtype)
    status = np.zeros(1, dtype=np.uint32)
    rc = lib().oracle_emb_fwd(_ptr(tables), _dt(tables), _ptr(row_base), F, D, B, _ptr(indices),
                              _ptr(offsets), indices.size, _ptr(pooled), flags, _ptr(status))
    if rc:
        raise ValueError("oracle_emb_fwd rejected its arguments")
    return pooled, int(status[0])


def gram(dense, pooled, b):
    dense, pooled = _c(dense), _c(pooled)
    B, F, D = pooled.shape
    g = np.zeros((F + 1, F + 1), dtype=np.float64)
    lib().oracle_gram(_ptr(dense), _ptr(pooled), _dt(pooled), F, D, b, _ptr(g))
    return g


def interact_fwd(dense, pooled, out_cols):
    dense, pooled = _c(dense), _c(pooled)
    B, F, D = pooled.shape
    assert dense.dtype == pooled.dtype and dense.shape == (B, D)
    out = np.zeros((B, out_cols), dtype=pooled.dtype)
    rc = lib().oracle_interact_fwd(_ptr(dense), _ptr(pooled), _dt(pooled), F, D, B, _ptr(out),
                                   out_cols)
    if rc:
        raise ValueError("oracle_interact_fwd rejected its arguments")
    return out


def interact_bwd(grad_out, dense, pooled):
    dense, pooled = _c(dense), _c(pooled)
    B, F, D = pooled.shape
    gdt = np.float64 if pooled.dtype == np.float64 else np.float32
    grad_out = _c(grad_out, gdt)
    out_cols = grad_out.shape[1]
    gd = np.zeros((B, D), dtype=gdt)
    gp = np.zeros((B, F, D), dtype=gdt)
    rc = lib().oracle_interact_bwd(_ptr(grad_out), _ptr(dense), _ptr(pooled), _dt(pooled), F, D, B,
                                   out_cols, _ptr(gd), _ptr(gp))
    if rc:
        raise ValueError("oracle_interact_bwd rejected its arguments")
    return gd, gp


def emb_bwd_sgd(tables, row_base, F, D, B, indices, offsets, grad_pooled, lr, flags=0):
    """Returns (updated tables copy, status, sorted keys, sorted vals)."""
    tables = np.array(tables, dtype=np.float32, copy=True, order="C")
    row_base = _c(row_base, np.int64)
    indices = _c(indices, np.int32)
    offsets = _c(offsets, np.int32)
    grad_pooled = _c(grad_pooled, np.float32)
    nnz = indices.size
    status = np.zeros(1, dtype=np.uint32)
    sk = np.zeros(max(nnz, 1), dtype=np.uint32)
    sv = np.zeros(max(nnz, 1), dtype=np.uint32)
    rc = lib().oracle_emb_bwd_sgd(_ptr(tables), _ptr(row_base), F, D, B, _ptr(indices),
                                  _ptr(offsets), nnz, _ptr(grad_pooled), float(lr), flags,
                                  _ptr(status), _ptr(sk), _ptr(sv))
    if rc:
        raise ValueError("oracle_emb_bwd_sgd rejected its arguments")
    return tables, int(status[0]), sk[:nnz], sv[:nnz]


def mlp_fwd(x, weights, biases, half_io=False):
    """Bottom MLP: relu(W h + b) per layer, double accumulation (see oracle.c).

    x: [B][K0] float32; weights[l]: [N_l][K_l]; biases[l]: [N_l].  Returns
    float64 [B][N_last] (binary16 values when half_io)."""
    x = _c(x, np.float32)
    B = x.shape[0]
    dims = [x.shape[1]] + [int(w.shape[0]) for w in weights]
    for l, w in enumerate(weights):
        assert w.shape == (dims[l + 1], dims[l]) and biases[l].shape == (dims[l + 1],)
    W = _c(np.concatenate([np.asarray(w, np.float32).reshape(-1) for w in weights]))
    bb = _c(np.concatenate([np.asarray(b, np.float32) for b in biases]))
    d = _c(np.array(dims, dtype=np.int32))
    out = np.zeros((B, dims[-1]), dtype=np.float64)
    rc = lib().oracle_mlp_fwd(_ptr(x), B, len(weights), _ptr(d), _ptr(W), _ptr(bb), int(bool(half_io)), _ptr(out))
    assert rc == 0, rc
    return out


# ------------------------------------------------------ mixed precision (AMP)
# "DLRM For PyTorch", §Mixed precision training: fp16 tensors for the
# interaction, fp32 master tables, static loss scaling.  Each result below is
# the exact (double) value of the definition, rounded once to binary16.

def round_f16(x):
    """Doubles rounded to binary16 (ties to even), as np.float16."""
    x = _c(x, np.float64)
    bits = np.zeros(x.shape, dtype=np.uint16)
    lib().oracle_round_f16(_ptr(x), _ptr(bits), x.size)
    return bits.view(np.float16)


def emb_fwd_f16out(tables, row_base, F, D, B, indices, offsets, flags=0):
    """Pooling of fp32 master rows, delivered as fp16 (summed in double, rounded once)."""
    pooled, status = emb_fwd(np.asarray(tables, np.float64), row_base, F, D, B, indices, offsets, flags)
    return round_f16(pooled), status


def interact_bwd_f16(grad_out, dense, pooled):
    """Interaction backward of fp16 tensors: exact sums, gradients rounded once to fp16."""
    gd, gp = interact_bwd(np.asarray(grad_out, np.float64), np.asarray(dense, np.float64),
                          np.asarray(pooled, np.float64))
    return round_f16(gd), round_f16(gp)
