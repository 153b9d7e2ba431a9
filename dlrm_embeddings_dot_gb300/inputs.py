"""Seeded synthetic inputs for the DLRM embedding + dot-interaction path.

This module only *makes inputs*: table sizes, embedding-table values, Zipf
distributed categorical indices with CSR offsets, the dense bottom-MLP output
and the upstream gradient.  It holds none of the lookup / interaction / SGD
arithmetic; both the CUDA path and the CPU oracle are fed from here.

Workload shapes follow "DLRM For PyTorch" (§Command-line options: 26
categorical tables, ``embedding_dim`` 128, 13 numerical features, bottom MLP
512,256,128; §Model architecture: the bottom-MLP output width equals the
embedding width so that it can enter the dot interaction).  The Criteo
Terabyte dataset the pages train on is not available, so every tensor here is
synthetic and seeded.

Generators (each written from its published definition):

* ``splitmix64`` (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): element ``e`` of a table gets
  ``mix(seed + (e + 1) * 0x9E3779B97F4A7C15)``; its top 24 bits give a
  uniform value on a 2^24-point grid.  The CUDA library carries its own implementation of the same
  generator (``dlrm_synth_fill_uniform``) so that multi-GB tables can be made
  on the device; tests check the two bit for bit.
* bounded Zipf by rejection-inversion (Hörmann & Derflinger, "Rejection-
  inversion to generate variates from monotone discrete distributions", ACM
  TOMACS 1996), P(k) ∝ k^-alpha on ranks 1..N, then a seeded affine bijection
  rank -> row so that hot rows are scattered through the table.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

F32 = 0
F16 = 1


# --------------------------------------------------------------------------
# counter-based uniform generator (splitmix64)
# --------------------------------------------------------------------------
def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """Output ``counters[i]`` (0-based) of the splitmix64 stream started at ``seed``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform_values(seed: int, elems: np.ndarray, amplitude: float) -> np.ndarray:
    """fp32 values in [-amplitude, amplitude) for global element numbers ``elems``.

    ``x = top24(z) - 2**23`` is a signed 24-bit integer (exact in fp32) and the
    value is the single fp32 product ``x * c`` with ``c = fp32(amplitude / 2**23)``.
    The device generator performs exactly these operations.
    """
    z = splitmix64(seed, elems)
    x = ((z >> np.uint64(40)).astype(np.int64) - (1 << 23)).astype(np.float32)
    c = np.float32(float(amplitude) / 8388608.0)
    return x * c


def table_rows(seed: int, global_rows: np.ndarray, D: int, dtype: int,
               amplitude: float = 0.05) -> np.ndarray:
    """Rows ``global_rows`` of the joint table, shape ``[len(rows), D]``, values
    uniform in [-0.05, 0.05).  fp16 tables are the fp32 values rounded once to
    fp16 (round to nearest even).
    """
    rows = np.asarray(global_rows, dtype=np.int64)
    elems = (rows[:, None] * D + np.arange(D, dtype=np.int64)[None, :]).astype(np.uint64)
    v = uniform_values(seed, elems, amplitude)
    if dtype == F16:
        return v.astype(np.float16)
    return v


# --------------------------------------------------------------------------
# bounded Zipf by rejection-inversion
# --------------------------------------------------------------------------
def _helper1(x: np.ndarray) -> np.ndarray:
    """log1p(x)/x, continuous at 0."""
    out = np.ones_like(x)
    nz = np.abs(x) > 1e-8
    out[nz] = np.log1p(x[nz]) / x[nz]
    small = ~nz
    out[small] = 1.0 - x[small] * (0.5 - x[small] / 3.0)
    return out


def _helper2(x: np.ndarray) -> np.ndarray:
    """expm1(x)/x, continuous at 0."""
    out = np.ones_like(x)
    nz = np.abs(x) > 1e-8
    out[nz] = np.expm1(x[nz]) / x[nz]
    small = ~nz
    out[small] = 1.0 + x[small] * 0.5 * (1.0 + x[small] / 3.0)
    return out


class BoundedZipf:
    """P(k) ∝ k^-alpha on k = 1..n, drawn by rejection-inversion.

    H(x) = ∫ t^-alpha dt (offset so that H(1) = 0) is the hat integral; a draw
    inverts H at a uniform point between H(1.5) - 1 and H(n + 0.5), rounds to
    the nearest integer k and accepts when k lies close enough to the inverse
    or when the point falls under the integral of the hat over [k - 1/2, k + 1/2]
    minus h(k).
    """

    def __init__(self, n: int, alpha: float):
        if n < 1 or alpha <= 0:
            raise ValueError("need n >= 1 and alpha > 0")
        self.n = int(n)
        self.a = float(alpha)
        self.h_x1 = float(self._H(np.array([1.5]))[0]) - 1.0
        self.h_n = float(self._H(np.array([self.n + 0.5]))[0])
        self.s = 2.0 - float(self._Hinv(self._H(np.array([2.5])) - self._h(np.array([2.0])))[0])

    def _h(self, x):
        return np.exp(-self.a * np.log(x))

    def _H(self, x):
        lx = np.log(x)
        return _helper2((1.0 - self.a) * lx) * lx

    def _Hinv(self, y):
        t = y * (1.0 - self.a)
        t = np.maximum(t, -1.0)
        return np.exp(_helper1(t) * y)

    def sample(self, rng: np.random.Generator, size: int) -> np.ndarray:
        out = np.empty(size, dtype=np.int64)
        todo = np.arange(size)
        while todo.size:
            u = rng.random(todo.size)
            y = self.h_n + u * (self.h_x1 - self.h_n)
            x = self._Hinv(y)
            k = np.clip(np.floor(x + 0.5), 1, self.n)
            ok = (k - x <= self.s) | (y >= self._H(k + 0.5) - self._h(k))
            out[todo[ok]] = k[ok].astype(np.int64)
            todo = todo[~ok]
        return out


def zipf_map(rng: np.random.Generator, n_rows: int, alpha: float, size: int) -> tuple[int, int]:
    """The (a, c) of the rank -> row map zipf_rows(rng, n_rows, alpha, size) uses."""
    BoundedZipf(n_rows, alpha).sample(rng, size)
    if n_rows == 1:
        return 1, 0
    while True:
        a = int(rng.integers(1, n_rows))
        if math.gcd(a, n_rows) == 1:
            break
    return a, int(rng.integers(0, n_rows))


def zipf_rows(rng: np.random.Generator, n_rows: int, alpha: float, size: int) -> np.ndarray:
    """Zipf ranks mapped to rows by ``row = (a*(k-1) + c) mod n``, gcd(a, n) = 1."""
    k = BoundedZipf(n_rows, alpha).sample(rng, size)
    if n_rows == 1:
        return np.zeros(size, dtype=np.int64)
    while True:
        a = int(rng.integers(1, n_rows))
        if math.gcd(a, n_rows) == 1:
            break
    c = int(rng.integers(0, n_rows))
    return (a * (k - 1) + c) % n_rows


# --------------------------------------------------------------------------
# dense input: the bottom MLP's output
# --------------------------------------------------------------------------
def bottom_mlp(x: np.ndarray, sizes: list[int], seed: int = 0) -> np.ndarray:
    """Bottom MLP of the pages (linear layers, ReLU after each), fp32.

    Xavier-uniform weights, zero biases, ``default_rng(seed)``.  The dense
    features it produces are an *input* of the embedding/interaction path.
    """
    rng = np.random.default_rng(seed)
    h = x.astype(np.float32)
    fan_in = h.shape[1]
    for width in sizes:
        lim = math.sqrt(6.0 / (fan_in + width))
        w = rng.uniform(-lim, lim, size=(fan_in, width)).astype(np.float32)
        h = np.maximum(h @ w, np.float32(0.0))
        fan_in = width
    return h


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------
@dataclass
class Workload:
    """One batch of synthetic inputs.

    ``indices``/``offsets`` are feature-major CSR: bag (t, b) is
    ``indices[offsets[t*B + b] : offsets[t*B + b + 1]]``.
    ``row_base[t]`` is the first row of table t inside the joint table.
    Table values are *not* stored: ``table_rows(table_seed, rows, D, dtype)``
    recomputes any row.
    """
    name: str
    B: int
    F: int
    D: int
    dtype: int
    rows: np.ndarray            # int64 [F]
    row_base: np.ndarray        # int64 [F+1]
    indices: np.ndarray         # int32 [nnz]
    offsets: np.ndarray         # int32 [F*B+1]
    dense: np.ndarray           # fp32 [B][D] (fp16-valued when dtype == F16)
    table_seed: int
    out_cols: int
    grad_out: np.ndarray | None = None   # fp32 [B][out_cols]
    lr: float = 0.1
    meta: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.indices.size)

    @property
    def total_rows(self) -> int:
        return int(self.row_base[-1])

    def full_tables(self) -> np.ndarray:
        """Whole joint table on the host (small workloads only)."""
        return table_rows(self.table_seed, np.arange(self.total_rows), self.D, self.dtype)


def _streams(entropy, n: int) -> list[np.random.Generator]:
    return [np.random.default_rng(s) for s in np.random.SeedSequence(entropy).spawn(n)]


def log_uniform_rows(rng: np.random.Generator, F: int, lo: float, hi: float) -> np.ndarray:
    return np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=F))).astype(np.int64)


def _csr(rng_pool, F: int, B: int, pool_lo: int, pool_hi: int):
    if pool_lo == pool_hi:
        counts = np.full(F * B, pool_lo, dtype=np.int64)
    else:
        counts = rng_pool.integers(pool_lo, pool_hi + 1, size=F * B)
    offsets = np.zeros(F * B + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    return counts, offsets


def make_workload(name: str, B: int, F: int, D: int, dtype: int, rows: np.ndarray,
                  alpha: float, dense: np.ndarray, out_cols: int, seed: int,
                  pool: tuple[int, int] = (1, 1), uniform_indices: bool = False,
                  with_grad: bool = False, grad_sigma: float = 1e-2, lr: float = 0.1,
                  table_seed: int | None = None, batch: int = 0) -> Workload:
    """``batch`` > 0 draws another batch over the same tables: new pooling
    factors, ranks (or uniform rows) and upstream gradient, with each table's
    Zipf rank -> row map unchanged, so the popular rows stay the same."""
    r_idx, r_pool, r_grad = _streams(seed + 1000 if batch == 0 else [seed + 1000, batch], 3)
    rows = np.asarray(rows, dtype=np.int64)
    row_base = np.zeros(F + 1, dtype=np.int64)
    np.cumsum(rows, out=row_base[1:])
    counts, offsets = _csr(r_pool, F, B, pool[0], pool[1])
    nnz = int(offsets[-1])
    if nnz >= 2**31:
        raise ValueError("nnz does not fit int32")
    indices = np.empty(nnz, dtype=np.int32)
    table_rngs = [np.random.default_rng(s) for s in np.random.SeedSequence([seed, 7]).spawn(F)]
    if batch != 0:   # batch 0's positions per table, to replay its draws of each table's rank -> row map
        _, offsets0 = _csr(_streams(seed + 1000, 3)[1], F, B, pool[0], pool[1])
    for t in range(F):
        lo, hi = int(offsets[t * B]), int(offsets[(t + 1) * B])
        n = hi - lo
        if batch == 0:
            if uniform_indices:
                indices[lo:hi] = table_rngs[t].integers(0, rows[t], size=n)
            else:
                indices[lo:hi] = zipf_rows(table_rngs[t], int(rows[t]), alpha, n)
        else:
            rb = np.random.default_rng(np.random.SeedSequence([seed, 7, t, batch]))
            if uniform_indices:
                indices[lo:hi] = rb.integers(0, rows[t], size=n)
            else:
                # the table's rank -> row map as batch 0 draws it (after batch 0's ranks)
                n0 = int(offsets0[(t + 1) * B] - offsets0[t * B])
                a, c = zipf_map(table_rngs[t], int(rows[t]), alpha, n0)
                k = BoundedZipf(int(rows[t]), alpha).sample(rb, n)
                indices[lo:hi] = 0 if int(rows[t]) == 1 else (a * (k - 1) + c) % int(rows[t])
    grad = None
    if with_grad:
        grad = r_grad.normal(0.0, grad_sigma, size=(B, out_cols)).astype(np.float32)
    return Workload(name=name, B=B, F=F, D=D, dtype=dtype, rows=rows, row_base=row_base,
                    indices=indices, offsets=offsets.astype(np.int32), dense=dense,
                    table_seed=(seed * 7919 + 17) if table_seed is None else table_seed,
                    out_cols=out_cols, grad_out=grad, lr=lr,
                    meta=dict(alpha=alpha, pool=pool, uniform=uniform_indices))


def _dense_input(seed: int, B: int, n_features: int, dist: str, mlp: list[int], dtype: int, batch: int = 0):
    rng = np.random.default_rng(np.random.SeedSequence([seed, 3] if batch == 0 else [seed, 3, batch]))
    if dist == "normal":
        x = rng.standard_normal((B, n_features)).astype(np.float32)
    else:
        x = rng.lognormal(0.0, 1.0, size=(B, n_features)).astype(np.float32)
    h = bottom_mlp(x, mlp, seed=0)
    if dtype == F16:
        if np.abs(h).max() >= 65504.0:
            raise ValueError("dense features overflow fp16")
        h = h.astype(np.float16).astype(np.float32)
    return h


def interaction_width(F: int, D: int) -> int:
    """Number of meaningful output columns: D + F(F+1)/2."""
    return D + F * (F + 1) // 2


def tiny_slice(seed: int = 0, B: int = 256, train: bool = False) -> Workload:
    """Batch 256, 4 dense N(0,1) features through a 4->32->16 bottom MLP, three
    tables of 1000 rows x 16 fp32, one index per feature (uniform; Zipf 1.2 when
    ``train`` so that the sparse gradient sees duplicates), 22 outputs."""
    F, D = 3, 16
    dense = _dense_input(seed, B, 4, "normal", [32, 16], F32)
    rows = np.full(F, 1000, dtype=np.int64)
    return make_workload("tiny-slice", B, F, D, F32, rows, alpha=1.2, dense=dense,
                         out_cols=interaction_width(F, D), seed=seed,
                         uniform_indices=not train, with_grad=train)


def dlrm_default(B: int = 65536, dtype: int = F16, alpha: float = 1.05, seed: int = 0,
                 train: bool = False, uniform_indices: bool = False,
                 rows: np.ndarray | None = None, batch: int = 0) -> Workload:
    """26 single-hot tables, D=128, row counts log-uniform in [10, 4e6]; 13
    lognormal dense features through the 13->512->256->128 bottom MLP; the
    27-vector interaction is 351 + 128 = 479 columns, padded to 480."""
    F, D = 26, 128
    if rows is None:
        rows = log_uniform_rows(np.random.default_rng(np.random.SeedSequence([seed, 11])), F, 10, 4e6)
    dense = _dense_input(seed, B, 13, "lognormal", [512, 256, 128], dtype, batch)
    return make_workload("dlrm-default", B, F, D, dtype, rows, alpha=alpha, dense=dense,
                         out_cols=480, seed=seed, with_grad=train,
                         uniform_indices=uniform_indices, batch=batch)


def multi_hot(B: int = 16384, rows_per_table: int = 1_000_000, alpha: float = 1.05,
              seed: int = 0, uniform_indices: bool = False, F: int = 26, batch: int = 0) -> Workload:
    """26 fp32 tables x 1e6 rows x 128, pooling factor uniform in [1, 100]."""
    D = 128
    dense = np.zeros((B, D), dtype=np.float32)
    rows = np.full(F, rows_per_table, dtype=np.int64)
    return make_workload("multi-hot", B, F, D, F32, rows, alpha=alpha, dense=dense,
                         out_cols=interaction_width(F, D), seed=seed, pool=(1, 100),
                         with_grad=True, uniform_indices=uniform_indices, batch=batch)


def large_tables_rows(seed: int = 0) -> np.ndarray:
    """Three tables of 40M rows, the other 23 log-uniform in [10, 4e6]."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 13]))
    rows = np.concatenate([np.full(3, 40_000_000, dtype=np.int64),
                           log_uniform_rows(rng, 23, 10, 4e6)])
    return rows


class Compact:
    """The bags of samples ``samples`` of workload ``w`` over a compacted table.

    Compaction only renames rows: the rows the sample touches are regenerated
    from the seeded generator on the host (never copied from a device) and the
    sample's indices are renumbered into that smaller table, order preserved
    within each table, so sums, sort order and updates are unchanged.
    """

    def __init__(self, w: Workload, samples: np.ndarray, dtype: int | None = None):
        dt = w.dtype if dtype is None else dtype
        samples = np.asarray(samples, dtype=np.int64)
        F, B = w.F, w.B
        self.samples = samples
        self.F, self.D, self.B = F, w.D, samples.size
        rows_per_t, idx_per_bag, counts = [], [], []
        for t in range(F):
            bags = t * B + samples
            s, e = w.offsets[bags], w.offsets[bags + 1]
            per = [w.indices[a:b].astype(np.int64) for a, b in zip(s, e)]
            idx_per_bag.append(per)
            counts.append(e - s)
            allidx = np.concatenate(per) if per else np.zeros(0, np.int64)
            rows_per_t.append(np.unique(allidx))
        self.uniq = rows_per_t                                    # table-local rows, sorted
        self.rows = np.array([max(len(u), 1) for u in rows_per_t], dtype=np.int64)
        self.row_base = np.concatenate([[0], np.cumsum(self.rows)]).astype(np.int64)
        glob_rows = []
        for t in range(F):
            u = rows_per_t[t]
            glob_rows.append(w.row_base[t] + (u if u.size else np.zeros(1, np.int64)))
        self.global_rows = np.concatenate(glob_rows)
        self.tables = table_rows(w.table_seed, self.global_rows, w.D, dt)
        cnt = np.concatenate(counts)                              # feature-major bag sizes
        self.offsets = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        parts = []
        for t in range(F):
            for per in idx_per_bag[t]:
                parts.append(np.searchsorted(rows_per_t[t], per))
        self.indices = (np.concatenate(parts) if parts else np.zeros(0, np.int64)).astype(np.int32)
        self.dense = (w.dense.astype(np.float16) if dt == F16 else w.dense.astype(np.float32))[samples]
        self.grad_out = None if w.grad_out is None else w.grad_out[samples]


def mlp_layers(dims, seed: int = 0):
    """Xavier-uniform fp16 weights [N][K] and small fp32 biases for a bottom MLP of widths dims."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 17]))
    W, b = [], []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        lim = np.sqrt(6.0 / (K + N))
        W.append(rng.uniform(-lim, lim, size=(N, K)).astype(np.float16))
        b.append(rng.uniform(-0.1, 0.1, size=N).astype(np.float32))
    return W, b


def mlp_pack(weights, biases):
    """The packed operands of dlrm_bottom_mlp_fwd: fp16 weights, each layer
    [N][round_up(K, 8)] with zero pad columns, one after another; fp32 biases
    one after another."""
    parts = []
    for w in weights:
        N, K = w.shape
        Kp = (K + 7) // 8 * 8
        pw = np.zeros((N, Kp), dtype=np.float16)
        pw[:, :K] = w
        parts.append(pw.reshape(-1))
    return np.concatenate(parts), np.concatenate([np.asarray(b, np.float32) for b in biases])
