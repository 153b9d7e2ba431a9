"""Python binding of the GB300 DLRM embedding + dot-interaction library.

Thin argument marshalling over the C ABI in ``include/dlrm.h``: every
function below has the name of the C entry point it calls, takes CUDA torch
tensors where the C call takes device pointers, and passes the current torch
stream unless one is given.  All computation happens in the CUDA kernels of
``libdlrm_gb300.so``; there is no fallback.  If the library has not been
built, ``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdlrm_gb300.so")

DLRM_OK = 0
DLRM_ERR_INVALID_ARG = 1
DLRM_ERR_UNSUPPORTED = 2
DLRM_ERR_CUDA = 3
DLRM_ERR_WORKSPACE = 4
DLRM_ERR_NO_FIT = 5
DLRM_FLAG_POOLED_F16 = 2
DLRM_FLAG_GRAD_F16 = 4
DLRM_F32 = 0
DLRM_F16 = 1
DLRM_FLAG_HASH_INDICES = 1
DLRM_STATUS_OOB_INDEX = 1
DLRM_STATUS_TIMEOUT = 2
DLRM_STATUS_BAD_OFFSETS = 4
DLRM_MAX_NNZ = 2**31 - 65
DLRM_NOALLOC_SCRATCH_BYTES = 16 << 20

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_lib = None


class DlrmError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library (build it first with ``build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(p)
    L.dlrm_emb_fwd.argtypes = [_P, _I, _P, _I, _I, _I, _P, _P, _I64, _P, ctypes.c_uint, _P, _P]
    L.dlrm_interact_fwd.argtypes = [_P, _P, _I, _I, _I, _I, _P, _I, _P, _P]
    L.dlrm_interact_fwd_cuda_core.argtypes = [_P, _P, _I, _I, _I, _I, _P, _I, _P]
    L.dlrm_emb_interact_fwd.argtypes = [_P, _I, _P, _I, _I, _I, _P, _P, _I64, _P, _P, _I, ctypes.c_uint, _P, _P]
    L.dlrm_emb_interact_bwd.argtypes = [_P, _I, _P, _I, _I, _I, _P, _P, _I64, _P, _P, _I, _P, _P, ctypes.c_uint, _P,
                                        _P]
    L.dlrm_emb_interact_fwd_train.argtypes = [_P, _I, _P, _I, _I, _I, _P, _P, _I64, _P, _P, _P, _I, ctypes.c_uint,
                                              _P, _P]
    L.dlrm_interact_bwd.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]
    L.dlrm_interact_bwd_f16.argtypes = [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P]
    L.dlrm_interact_bwd_f16.restype = _I
    L.dlrm_emb_bwd_sgd_workspace_size.argtypes = [_I64, _I, _I64]
    L.dlrm_emb_bwd_sgd_workspace_size.restype = ctypes.c_size_t
    L.dlrm_emb_bwd_sgd.argtypes = [_P, _P, _I64, _I, _I, _I, _P, _P, _I64, _P, ctypes.c_float, _P,
                                   ctypes.c_size_t, ctypes.c_uint, _P, _P]
    L.dlrm_emb_bwd_sgd_noalloc.argtypes = [_P, _P, _I64, _I, _I, _I, _P, _P, _I64, _P, ctypes.c_float,
                                           ctypes.c_uint, _P, _P]
    L.dlrm_set_wait_limit.argtypes = [_I64]
    L.dlrm_set_wait_limit.restype = _I64
    L.dlrm_ws_align.argtypes = [ctypes.c_size_t]
    L.dlrm_ws_align.restype = ctypes.c_size_t
    L.dlrm_last_error.argtypes = []
    L.dlrm_last_error.restype = ctypes.c_char_p
    L.dlrm_synth_fill_uniform.argtypes = [_P, _I, ctypes.c_uint64, _I64, _I64, ctypes.c_double, _P]
    L.dlrm_plan_tables.argtypes = [_I, _P, _I, _P, _P]
    L.dlrm_batch_shard.argtypes = [_I64, _I, _I, _P, _P]
    L.dlrm_a2a_layout.argtypes = [_I, _P, _I64, _I, _I, _I64, _P, _P, _P, _P, _P]
    L.dlrm_bottom_mlp_workspace_size.argtypes = [_I, _I, _P]
    L.dlrm_bottom_mlp_workspace_size.restype = ctypes.c_size_t
    L.dlrm_bottom_mlp_fwd.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
    L.dlrm_bottom_mlp_fwd.restype = _I
    for f in ("dlrm_plan_tables", "dlrm_batch_shard", "dlrm_a2a_layout"):
        getattr(L, f).restype = _I
    for f in ("dlrm_emb_fwd", "dlrm_interact_fwd", "dlrm_interact_fwd_cuda_core", "dlrm_emb_interact_fwd",
              "dlrm_emb_interact_fwd_train", "dlrm_emb_interact_bwd", "dlrm_interact_bwd", "dlrm_emb_bwd_sgd", "dlrm_emb_bwd_sgd_noalloc", "dlrm_synth_fill_uniform"):
        getattr(L, f).restype = _I
    if path is None:
        _lib = L
    return L


def dlrm_set_wait_limit(cycles: int) -> int:
    """Bound of the tensor-core kernels' on-chip waits in SM cycles (negative: the default,
    about two seconds); returns the previous bound."""
    return int(load().dlrm_set_wait_limit(int(cycles)))


def dlrm_last_error() -> str:
    return load().dlrm_last_error().decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DLRM_F32
    if t.dtype == torch.float16:
        return DLRM_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != DLRM_OK:
        raise DlrmError(fn, rc, dlrm_last_error())


def dlrm_emb_fwd(tables, row_base, F, D, B, indices, offsets, pooled, flags=0, status=None, stream=None):
    """pooled[b][t] = sum of the rows of bag (t, b); see ``include/dlrm.h``."""
    rc = load().dlrm_emb_fwd(_ptr(tables), _dtype_code(tables), _ptr(row_base), F, D, B, _ptr(indices),
                             _ptr(offsets), indices.numel(), _ptr(pooled), flags, _ptr(status),
                             _stream(stream))
    _check("dlrm_emb_fwd", rc)


def dlrm_interact_fwd(dense, pooled, F, D, B, out, out_cols, status=None, stream=None):
    """out[b] = [dense | strict lower triangle of Z Z^T | 0-pad]; see ``include/dlrm.h``."""
    rc = load().dlrm_interact_fwd(_ptr(dense), _ptr(pooled), _dtype_code(pooled), F, D, B, _ptr(out),
                                  out_cols, _ptr(status), _stream(stream))
    _check("dlrm_interact_fwd", rc)


def dlrm_interact_fwd_cuda_core(dense, pooled, F, D, B, out, out_cols, stream=None):
    """The CUDA-core kernel of the interaction for any shape (cross-check of the tensor-core one)."""
    rc = load().dlrm_interact_fwd_cuda_core(_ptr(dense), _ptr(pooled), _dtype_code(pooled), F, D, B,
                                            _ptr(out), out_cols, _stream(stream))
    _check("dlrm_interact_fwd_cuda_core", rc)


def dlrm_emb_interact_fwd(tables, row_base, F, D, B, indices, offsets, dense, out, out_cols, flags=0,
                          status=None, stream=None):
    """Lookup + interaction in one pass (inference); see ``include/dlrm.h``."""
    rc = load().dlrm_emb_interact_fwd(_ptr(tables), _dtype_code(tables), _ptr(row_base), F, D, B, _ptr(indices),
                                      _ptr(offsets), indices.numel(), _ptr(dense), _ptr(out), out_cols, flags,
                                      _ptr(status), _stream(stream))
    _check("dlrm_emb_interact_fwd", rc)


def dlrm_emb_interact_fwd_train(tables, row_base, F, D, B, indices, offsets, dense, pooled, out, out_cols, flags=0,
                                status=None, stream=None):
    """Training forward in one pass: lookup (pooled written) + interaction; see ``include/dlrm.h``."""
    rc = load().dlrm_emb_interact_fwd_train(_ptr(tables), _dtype_code(tables), _ptr(row_base), F, D, B,
                                            _ptr(indices), _ptr(offsets), indices.numel(), _ptr(dense),
                                            _ptr(pooled), _ptr(out), out_cols, flags, _ptr(status), _stream(stream))
    _check("dlrm_emb_interact_fwd_train", rc)


def dlrm_emb_interact_bwd(tables, row_base, F, D, B, indices, offsets, grad_out, dense, out_cols, grad_dense,
                          grad_pooled, flags=0, status=None, stream=None):
    """Interaction backward with the pooled rows gathered from the tables; see ``include/dlrm.h``."""
    rc = load().dlrm_emb_interact_bwd(_ptr(tables), _dtype_code(tables), _ptr(row_base), F, D, B, _ptr(indices),
                                      _ptr(offsets), indices.numel(), _ptr(grad_out), _ptr(dense), out_cols,
                                      _ptr(grad_dense), _ptr(grad_pooled), flags, _ptr(status), _stream(stream))
    _check("dlrm_emb_interact_bwd", rc)


def dlrm_interact_bwd(grad_out, dense, pooled, F, D, B, out_cols, grad_dense, grad_pooled, stream=None):
    rc = load().dlrm_interact_bwd(_ptr(grad_out), _ptr(dense), _ptr(pooled), _dtype_code(pooled), F, D, B,
                                  out_cols, _ptr(grad_dense), _ptr(grad_pooled), _stream(stream))
    _check("dlrm_interact_bwd", rc)


def dlrm_interact_bwd_f16(grad_out, dense, pooled, F, D, B, out_cols, grad_dense, grad_pooled, status=None,
                          stream=None):
    """Mixed-precision interaction backward (fp16 tensors, tcgen05); see include/dlrm.h."""
    rc = load().dlrm_interact_bwd_f16(_ptr(grad_out), _ptr(dense), _ptr(pooled), F, D, B, out_cols,
                                      _ptr(grad_dense), _ptr(grad_pooled), _ptr(status), _stream(stream))
    _check("dlrm_interact_bwd_f16", rc)


def dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows) -> int:
    return int(load().dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows))


def dlrm_ws_align(nbytes) -> int:
    return int(load().dlrm_ws_align(nbytes))


def dlrm_emb_bwd_sgd(tables, row_base, total_rows, F, D, B, indices, offsets, grad_pooled, lr, workspace,
                     flags=0, status=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dlrm_emb_bwd_sgd(_ptr(tables), _ptr(row_base), total_rows, F, D, B, _ptr(indices),
                                 _ptr(offsets), indices.numel(), _ptr(grad_pooled), float(lr),
                                 _ptr(workspace), ws_bytes, flags, _ptr(status), _stream(stream))
    _check("dlrm_emb_bwd_sgd", rc)


def dlrm_emb_bwd_sgd_noalloc(tables, row_base, total_rows, F, D, B, indices, offsets, grad_pooled, lr,
                             flags=0, status=None, stream=None):
    """dlrm_emb_bwd_sgd without a workspace argument, for callers that cannot
    allocate device memory: the scratch is an array built into the library
    (calls that overlap on the GPU share it and must be serialised)."""
    rc = load().dlrm_emb_bwd_sgd_noalloc(_ptr(tables), _ptr(row_base), total_rows, F, D, B, _ptr(indices),
                                         _ptr(offsets), indices.numel(), _ptr(grad_pooled), float(lr), flags,
                                         _ptr(status), _stream(stream))
    _check("dlrm_emb_bwd_sgd_noalloc", rc)


def dlrm_synth_fill_uniform(dst, seed, first_elem, amplitude=0.05, stream=None):
    rc = load().dlrm_synth_fill_uniform(_ptr(dst), _dtype_code(dst), seed & (2**64 - 1), first_elem,
                                        dst.numel(), amplitude, _stream(stream))
    _check("dlrm_synth_fill_uniform", rc)


# ---------------------------------------------------------------- host planning
# Host-only calls (include/dlrm_plan.h): lists in, lists out, no GPU.

def _host_i64(values):
    return (ctypes.c_int64 * max(len(values), 1))(*values)


def dlrm_plan_tables(table_bytes, gpu_free_bytes) -> list[int]:
    """GPU of each table under the pages' placement heuristic (bottom MLP on GPU 0)."""
    n = len(table_bytes)
    dev = (ctypes.c_int * max(n, 1))()
    rc = load().dlrm_plan_tables(n, _host_i64(table_bytes), len(gpu_free_bytes), _host_i64(gpu_free_bytes), dev)
    _check("dlrm_plan_tables", rc)
    return list(dev[:n])


def dlrm_batch_shard(batch, n_ranks, rank) -> tuple[int, int]:
    first, count = ctypes.c_int64(), ctypes.c_int64()
    rc = load().dlrm_batch_shard(batch, n_ranks, rank, ctypes.byref(first), ctypes.byref(count))
    _check("dlrm_batch_shard", rc)
    return first.value, count.value


def dlrm_a2a_layout(table_device, batch, n_ranks, rank, row_elems):
    """(send_counts, send_displs, recv_counts, recv_displs, slot_table) of the forward exchange."""
    n = len(table_device)
    arrs = [(ctypes.c_int64 * n_ranks)() for _ in range(4)]
    slots = (ctypes.c_int * max(n, 1))()
    rc = load().dlrm_a2a_layout(n, (ctypes.c_int * max(n, 1))(*table_device), batch, n_ranks, rank, row_elems,
                                *arrs, slots)
    _check("dlrm_a2a_layout", rc)
    return tuple(list(a) for a in arrs) + (list(slots[:n]),)


# ---------------------------------------------------------------- bottom MLP
def _dims_arr(dims):
    return (ctypes.c_int * len(dims))(*[int(d) for d in dims])


def dlrm_bottom_mlp_workspace_size(B, dims) -> int:
    return int(load().dlrm_bottom_mlp_workspace_size(B, len(dims) - 1, _dims_arr(dims)))


def dlrm_bottom_mlp_fwd(x, dims, weights, biases, out, workspace, status=None, stream=None):
    """out (fp16 [B][dims[-1]]) = the bottom MLP of x (fp32 [B][dims[0]]); see include/dlrm_mlp.h.

    weights / biases are the packed device buffers (inputs.mlp_pack lays them out)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dlrm_bottom_mlp_fwd(_ptr(x), x.shape[0], len(dims) - 1, _dims_arr(dims), _ptr(weights),
                                    _ptr(biases), _ptr(out), _ptr(workspace), ws_bytes, _ptr(status),
                                    _stream(stream))
    _check("dlrm_bottom_mlp_fwd", rc)
