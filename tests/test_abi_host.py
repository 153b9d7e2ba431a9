"""Host-side checks of the C ABI: the library loads, exports every entry point
declared in include/*.h, and rejects bad arguments before touching the GPU.

No call here reaches a kernel launch: every call either fails validation or
has nothing to do (empty batch), both of which return before any CUDA call.
"""

import ctypes
import glob
import os
import re

import pytest

import dlrm_embeddings_dot_gb300 as dl
from dlrm_embeddings_dot_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = 0x10000          # a 16-byte aligned non-null "device pointer" (never dereferenced)
FAKE_MIS = 0x10004      # misaligned


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return dl.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(dlrm_[a-z0-9_]+)\s*\(", src))
    return names


def test_binding_constants_match_the_header():
    """Every integer macro and enum value of include/dlrm.h that the binding also defines has
    the same value."""
    src = open(os.path.join(ROOT, "include", "dlrm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    macros = {m.group(1): int(m.group(2), 0)
              for m in re.finditer(r"#define\s+(DLRM_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)(?:u|LL|ll|U)?\b", src)}
    macros.update({m.group(1): int(m.group(2))
                   for m in re.finditer(r"\b(DLRM_[A-Z0-9_]+)\s*=\s*(\d+)\s*[,}]", src)})
    assert {"DLRM_MAX_NNZ", "DLRM_FLAG_HASH_INDICES", "DLRM_STATUS_BAD_OFFSETS", "DLRM_OK",
            "DLRM_ERR_INVALID_ARG", "DLRM_F16"} <= set(macros)
    shared = [n for n in macros if hasattr(dl, n)]
    assert len(shared) >= 8
    for n in shared:
        assert getattr(dl, n) == macros[n], n
    assert dl.DLRM_MAX_NNZ == 2**31 - 65


def test_nnz_past_the_bound_is_rejected(L):
    """nnz above DLRM_MAX_NNZ (index positions plus the kernels' position steps must stay
    below 2^31) is an argument error at every entry point that takes it."""
    big = dl.DLRM_MAX_NNZ + 1
    assert L.dlrm_emb_fwd(FAKE, 0, FAKE, 1, 4, 2, FAKE, FAKE, big, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert "DLRM_MAX_NNZ" in _err(L)
    assert L.dlrm_emb_interact_fwd_train(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, big, FAKE, FAKE, FAKE, 480, 0, None,
                                         None) == dl.DLRM_ERR_INVALID_ARG
    assert L.dlrm_emb_interact_fwd(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, big, FAKE, FAKE, 480, 0, None,
                                   None) == dl.DLRM_ERR_INVALID_ARG
    assert L.dlrm_emb_interact_bwd(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, big, FAKE, FAKE, 480, FAKE, FAKE, 0, None,
                                   None) == dl.DLRM_ERR_INVALID_ARG
    assert L.dlrm_emb_bwd_sgd_workspace_size(big, 128, 5000) == 0
    assert L.dlrm_emb_bwd_sgd_workspace_size(dl.DLRM_MAX_NNZ, 128, 5000) > 0
    assert L.dlrm_emb_bwd_sgd(FAKE, FAKE, 50, 2, 16, 50, FAKE, FAKE, big, FAKE, ctypes.c_float(0.1), FAKE, 1 << 40, 0,
                              None, None) == dl.DLRM_ERR_INVALID_ARG


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"dlrm_emb_fwd", "dlrm_interact_fwd", "dlrm_interact_bwd", "dlrm_emb_bwd_sgd",
            "dlrm_emb_bwd_sgd_workspace_size", "dlrm_last_error"} <= names
    for n in names:
        assert hasattr(L, n), f"{n} declared but not exported"


def _exported():
    """dlrm_* functions the built library exports (its dynamic symbol table)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", libbuild.LIB], capture_output=True, text=True,
                         check=True).stdout
    return {parts[-1] for parts in (line.split() for line in out.splitlines())
            if len(parts) >= 3 and parts[-2] in ("T", "t") and parts[-1].startswith("dlrm_")}


def test_every_exported_symbol_is_declared(L):
    """The other direction: a C caller can reach every dlrm_* function the library exports,
    because each one has a prototype in include/*.h."""
    exported = _exported()
    assert {"dlrm_emb_fwd", "dlrm_emb_interact_bwd", "dlrm_emb_bwd_sgd"} <= exported
    missing = sorted(exported - _declared())
    assert not missing, f"exported but declared in no header: {missing}"


def _err(L):
    return L.dlrm_last_error().decode()


def test_emb_fwd_validation(L):
    f = L.dlrm_emb_fwd
    assert f(None, 0, FAKE, 1, 4, 2, FAKE, FAKE, 2, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert "null" in _err(L)
    assert f(FAKE, 0, FAKE, 0, 4, 2, FAKE, FAKE, 2, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, FAKE, 1, 4, -1, FAKE, FAKE, 2, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, FAKE, 1, 4, 2, FAKE, FAKE, -5, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, FAKE, 1, 4, 2, FAKE, FAKE, 2**31, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 7, FAKE, 1, 4, 2, FAKE, FAKE, 2, FAKE, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, FAKE, 1, 4, 2, FAKE, FAKE, 2, FAKE, 8, None, None) == dl.DLRM_ERR_INVALID_ARG
    # 3 fp32 = 12 bytes per row: not a multiple of 16
    assert f(FAKE, 0, FAKE, 1, 3, 2, FAKE, FAKE, 2, FAKE, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE_MIS, 0, FAKE, 1, 4, 2, FAKE, FAKE, 2, FAKE, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 1, 4, 2, FAKE, FAKE, 2, FAKE_MIS, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    # empty batch: nothing to do, returns before any CUDA call
    assert f(FAKE, 0, FAKE, 3, 4, 0, None, FAKE, 0, FAKE, 0, None, None) == dl.DLRM_OK


def test_interact_validation(L):
    f = L.dlrm_interact_fwd
    # F=2, D=4: W = 4 + 3 = 7
    assert f(FAKE, FAKE, 0, 2, 4, 8, FAKE, 6, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert "out_cols" in _err(L)
    assert f(None, FAKE, 0, 2, 4, 8, FAKE, 7, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 0, 0, 4, 8, FAKE, 7, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 1, 2, 4, 8, FAKE, 7, None, None) == dl.DLRM_ERR_UNSUPPORTED   # 4 halves = 8 B
    assert f(FAKE_MIS, FAKE, 0, 2, 4, 8, FAKE, 7, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, 0, 2, 4, 0, FAKE, 7, None, None) == dl.DLRM_OK
    g = L.dlrm_interact_bwd
    assert g(FAKE, FAKE, FAKE, 0, 2, 4, 8, 6, FAKE, FAKE, None) == dl.DLRM_ERR_INVALID_ARG
    assert g(FAKE, FAKE, FAKE, 0, 2, 4, 8, 7, None, FAKE, None) == dl.DLRM_ERR_INVALID_ARG
    assert g(FAKE, FAKE, FAKE, 0, 2, 4, 8, 7, FAKE, FAKE_MIS, None) == dl.DLRM_ERR_UNSUPPORTED
    assert g(FAKE, FAKE, FAKE, 0, 2, 4, 0, 7, FAKE, FAKE, None) == dl.DLRM_OK
    h = L.dlrm_interact_fwd_cuda_core
    assert h(FAKE, FAKE, 0, 2, 4, 8, FAKE, 6, None) == dl.DLRM_ERR_INVALID_ARG


def test_fused_training_forward_validation(L):
    f = L.dlrm_emb_interact_fwd_train
    # tables, dtype, row_base, F, D, B, indices, offsets, nnz, dense, pooled, out, out_cols, flags, status, stream
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 478, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert "out_cols" in _err(L)
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, None, FAKE, 480, 0, None, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 480, 8, None, None) == dl.DLRM_ERR_INVALID_ARG
    # fp16 tables, other F, D, padding past the last group of pairs, misalignment: the two calls instead
    assert f(FAKE, 1, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 480, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 25, 128, 8, FAKE, FAKE, 200, FAKE, FAKE, FAKE, 480, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 64, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 480, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 484, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 482, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE_MIS, FAKE, 480, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE_MIS, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, FAKE, 480, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    # empty batch: nothing to do, returns before any CUDA call
    assert f(FAKE, 0, FAKE, 26, 128, 0, None, FAKE, 0, FAKE, FAKE, FAKE, 480, 0, None, None) == dl.DLRM_OK
    assert f(FAKE, 0, FAKE, 8, 128, 0, None, FAKE, 0, FAKE, FAKE, FAKE, 164, 1, None, None) == dl.DLRM_OK
    # the inference entry takes the same fp32 shapes (no pooled output)
    g = L.dlrm_emb_interact_fwd
    assert g(FAKE, 0, FAKE, 3, 16, 8, FAKE, FAKE, 24, FAKE, FAKE, 22, 0, None, None) == dl.DLRM_ERR_UNSUPPORTED
    assert g(FAKE, 0, FAKE, 26, 128, 0, None, FAKE, 0, FAKE, FAKE, 480, 0, None, None) == dl.DLRM_OK


def test_gathering_backward_validation(L):
    f = L.dlrm_emb_interact_bwd
    # tables, dtype, row_base, F, D, B, indices, offsets, nnz, grad_out, dense, out_cols, gd, gp, flags, status, stream
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, 478, FAKE, FAKE, 0, None, None) == \
        dl.DLRM_ERR_INVALID_ARG
    assert "out_cols" in _err(L)
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, 480, None, FAKE, 0, None, None) == \
        dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, 480, FAKE, FAKE, 2, None, None) == \
        dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 1, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, 480, FAKE, FAKE, 0, None, None) == \
        dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 25, 128, 8, FAKE, FAKE, 200, FAKE, FAKE, 480, FAKE, FAKE, 0, None, None) == \
        dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, 481, FAKE, FAKE, 0, None, None) == \
        dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 128, 8, FAKE, FAKE, 208, FAKE, FAKE, 480, FAKE, FAKE_MIS, 0, None, None) == \
        dl.DLRM_ERR_UNSUPPORTED
    assert f(FAKE, 0, FAKE, 26, 128, 0, None, FAKE, 0, FAKE, FAKE, 480, FAKE, FAKE, 0, None, None) == dl.DLRM_OK


def test_sgd_workspace_grows_with_nnz(L):
    """Callers size one workspace for their largest batch: the size never drops as
    nnz grows, across the edge where short segment items stop (8,192 indices)."""
    ns = list(range(8000, 8400)) + [8192 * 8 - 1, 8192 * 8, 8192 * 8 + 1, 10**6]
    for D in (4, 128, 1024):
        sizes = [L.dlrm_emb_bwd_sgd_workspace_size(n, D, 5000) for n in [1, 31, 32, 33, 256, 257] + ns]
        assert all(x > 0 for x in sizes)
        assert all(a <= b for a, b in zip(sizes, sizes[1:]))


def test_sgd_workspace_and_validation(L):
    ws = L.dlrm_emb_bwd_sgd_workspace_size
    assert ws(-1, 128, 10) == 0 and ws(10, 3, 10) == 0 and ws(10, 128, 0) == 0
    assert ws(10, 128, 2**32) == 0
    a, b = ws(1000, 128, 5000), ws(100000, 128, 5000)
    assert 0 < a < b and a % 256 == 0
    assert L.dlrm_ws_align(1) == 256 and L.dlrm_ws_align(256) == 256 and L.dlrm_ws_align(0) == 0
    f = L.dlrm_emb_bwd_sgd
    need = ws(100, 16, 50)
    args = [FAKE, FAKE, 50, 2, 16, 50, FAKE, FAKE, 100, FAKE, ctypes.c_float(0.1), FAKE, need, 0, None, None]
    bad = list(args); bad[12] = need - 1
    assert f(*bad) == dl.DLRM_ERR_WORKSPACE
    assert "workspace" in _err(L)
    bad = list(args); bad[2] = 0
    assert f(*bad) == dl.DLRM_ERR_INVALID_ARG
    bad = list(args); bad[11] = FAKE + 16                 # workspace not 256-byte aligned
    assert f(*bad) == dl.DLRM_ERR_UNSUPPORTED
    bad = list(args); bad[4] = 6                          # D % 4 != 0
    assert f(*bad) == dl.DLRM_ERR_UNSUPPORTED
    bad = list(args); bad[13] = 8                         # unknown flag
    assert f(*bad) == dl.DLRM_ERR_INVALID_ARG
    ok = list(args); ok[8] = 0; ok[6] = None              # nnz = 0: nothing to do
    assert f(*ok) == dl.DLRM_OK


def test_synth_validation(L):
    f = L.dlrm_synth_fill_uniform
    assert f(None, 0, 1, 0, 10, 0.05, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, 1, 0, -1, 0.05, None) == dl.DLRM_ERR_INVALID_ARG
    assert f(FAKE, 0, 1, 0, 0, 0.05, None) == dl.DLRM_OK


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        dl.load(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("D,limit", [(128, 809_216), (16, 973_632)])
def test_noalloc_capacity_quoted_in_the_header(L, D, limit):
    """The most indices dlrm_emb_bwd_sgd_noalloc takes, as include/dlrm.h quotes them: the
    workspace of `limit` indices fits the built-in scratch and one more does not, whatever
    the table size."""
    src = open(os.path.join(ROOT, "include", "dlrm.h")).read()
    assert f"{limit:,}" in src
    for rows in (10, 9_056_641, 2**32 - 2):
        assert L.dlrm_emb_bwd_sgd_workspace_size(limit, D, rows) <= dl.DLRM_NOALLOC_SCRATCH_BYTES
        assert L.dlrm_emb_bwd_sgd_workspace_size(limit + 1, D, rows) > dl.DLRM_NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_over_capacity_before_any_launch(L):
    """One index past the capacity is refused on the host (nothing reaches the GPU)."""
    rc = L.dlrm_emb_bwd_sgd_noalloc(FAKE, FAKE, 10, 1, 128, 809_217, FAKE, FAKE, 809_217, FAKE,
                                    ctypes.c_float(0.1), 0, None, None)
    assert rc == dl.DLRM_ERR_UNSUPPORTED and "scratch" in _err(L)
