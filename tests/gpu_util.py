"""Helpers for the GPU parity tests: device buffers for a workload, and the
compaction of a sample of a large workload (``inputs.Compact``) so that the
CPU oracle can check it."""

from __future__ import annotations

import numpy as np
import torch

from dlrm_embeddings_dot_gb300 import inputs
from dlrm_embeddings_dot_gb300.inputs import Compact  # noqa: F401  (re-exported for the tests)


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def torch_dtype(dt: int):
    return torch.float16 if dt == inputs.F16 else torch.float32


def np_dtype(dt: int):
    return np.float16 if dt == inputs.F16 else np.float32


def device_tables(dl, w: inputs.Workload, dtype: int | None = None) -> torch.Tensor:
    """Joint table [total_rows][D] generated on the device from the workload's seed."""
    dt = w.dtype if dtype is None else dtype
    t = torch.empty(w.total_rows, w.D, dtype=torch_dtype(dt), device=dev())
    dl.dlrm_synth_fill_uniform(t, w.table_seed, 0)
    return t


def dense_for(w: inputs.Workload, dtype: int | None = None) -> np.ndarray:
    dt = w.dtype if dtype is None else dtype
    return w.dense.astype(np_dtype(dt))
