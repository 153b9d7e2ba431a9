"""Benchmark of the DLRM embedding + dot-interaction hot path on GB300.

One step = one pass of the whole path over one batch of 65,536 samples:
    dlrm_emb_fwd -> dlrm_interact_fwd -> dlrm_interact_bwd -> dlrm_emb_bwd_sgd
on the DLRM-default shapes (26 single-hot tables with log-uniform row counts in
[10, 4e6], D = 128, 13 lognormal dense features through the 13-512-256-128
bottom MLP, 480 interaction columns), FP32 master tables, Zipf(1.2) indices,
upstream gradient N(0, 1e-2), SGD lr 0.1.  The forward alone at the same batch
with fp16 tables and Zipf(1.05) indices is reported under "fwd".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  With N > 1 (torchrun) every rank runs its own
replica on its own GPU (weak scaling; the path needs no exchange between GPUs).
"""

from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DLRM emb+interaction samples/s at batch 64K (fwd, fwd+bwd); % of HBM peak"
BATCH = 65536
ALPHA_TRAIN = 1.2
ALPHA_FWD = 1.05
LR = 0.1
L2_BYTES = 129 * 2**20
E2E_MIN_STEPS = 30   # pipelined end-to-end steps at least, whatever --steps is
WORKLOAD = ("dlrm-default 64K training step: 26 single-hot fp32 tables (rows log-uniform 10..4e6), "
            "D=128, Zipf 1.2, 480 interaction columns, SGD lr 0.1")


# ---------------------------------------------------------------- utilities
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when there is one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"dlrm_clocks_{os.getpid()}.csv")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "dlrm_embeddings_dot_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, batch: int = None):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source.  A
    capture on a smaller batch (the recipe's size rule) is scaled to `batch` by the samples
    processed, the kernel's traffic growing in proportion to them; returns (bytes, note)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        e = json.load(f).get(kernel)
    if not e or e.get("source_digest") != source_digest(e.get("source_files", [])):
        return None, None
    dram, cb = e.get("dram_bytes_per_launch"), e.get("captured_batch")
    if batch and cb and cb != batch:
        return int(round(dram * batch / cb)), f"ncu capture at batch {cb} ({dram} B) scaled by {batch}/{cb} samples"
    return dram, f"ncu capture at batch {cb}" if cb else None


# ------------------------------------------------------------ oracle (CPU)
def cpu_oracle_step(w, samples: np.ndarray) -> float:
    """Time the CPU oracle on the step for a sample of the batch; returns seconds."""
    import oracle
    from dlrm_embeddings_dot_gb300.inputs import Compact
    c = Compact(w, samples)
    t0 = time.perf_counter()
    pooled, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    oracle.interact_fwd(c.dense, pooled, w.out_cols)
    _, gp = oracle.interact_bwd(c.grad_out, c.dense, pooled)
    oracle.emb_bwd_sgd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets, gp, w.lr)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for key in ("Model name:", "Vendor ID:"):
            for line in out.splitlines():
                if line.strip().startswith(key):
                    return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


class ThreadedOracleStep:
    """The training step on the CPU oracle, split over host threads.

    The oracle's C functions run unchanged, each on a disjoint part of the
    step: the lookup and the sparse SGD once per table (the tables' rows are
    disjoint, and a table's positions keep their order, so each row's sum is
    taken in the same order as in one call), the interaction and its backward
    once per block of samples.  ctypes releases the interpreter lock during
    each call, so the parts run in parallel.  ``run(threads)`` returns seconds;
    ``outputs()`` the results (checked against one oracle call by the tests)."""

    def __init__(self, w, samples: np.ndarray):
        import ctypes

        import oracle
        from dlrm_embeddings_dot_gb300.inputs import Compact
        c = Compact(w, samples)
        self.L = oracle.lib()
        self.F, self.D, self.B, self.P, self.lr = c.F, c.D, c.B, w.out_cols, float(w.lr)
        F, D, B = self.F, self.D, self.B
        self.tables = np.array(c.tables, dtype=np.float32, order="C")
        self.parts = []
        for t in range(F):
            lo, hi = int(c.offsets[t * B]), int(c.offsets[(t + 1) * B])
            self.parts.append(dict(off=np.ascontiguousarray(np.asarray(c.offsets[t * B:(t + 1) * B + 1]) - lo,
                                                            dtype=np.int32),
                                   idx=np.ascontiguousarray(c.indices[lo:hi], dtype=np.int32),
                                   rb=np.array([0, int(c.row_base[t + 1] - c.row_base[t])], dtype=np.int64),
                                   r0=int(c.row_base[t]), r1=int(c.row_base[t + 1]),
                                   pooled=np.zeros((B, 1, D), np.float32), gp=np.zeros((B, 1, D), np.float32),
                                   status=np.zeros(1, np.uint32)))
        self.dense = np.ascontiguousarray(c.dense, dtype=np.float32)
        self.go = np.ascontiguousarray(c.grad_out, dtype=np.float32)
        self.pooled = np.zeros((B, F, D), np.float32)
        self.out = np.zeros((B, self.P), np.float32)
        self.gd = np.zeros((B, D), np.float32)
        self.gp = np.zeros((B, F, D), np.float32)
        self.ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)

    def run(self, threads: int) -> float:
        from concurrent.futures import ThreadPoolExecutor
        L, ptr, F, D, B, P = self.L, self.ptr, self.F, self.D, self.B, self.P
        blocks = [(int(a[0]), int(a[-1]) + 1) for a in np.array_split(np.arange(B), max(1, threads)) if a.size]

        def lookup(t):
            q = self.parts[t]
            if q["r1"] > q["r0"]:
                L.oracle_emb_fwd(ptr(self.tables[q["r0"]:q["r1"]]), 0, ptr(q["rb"]), 1, D, B, ptr(q["idx"]),
                                 ptr(q["off"]), q["idx"].size, ptr(q["pooled"]), 0, ptr(q["status"]))
            self.pooled[:, t, :] = q["pooled"][:, 0, :]

        def interact(blk):
            b0, b1 = blk
            L.oracle_interact_fwd(ptr(self.dense[b0:b1]), ptr(self.pooled[b0:b1]), 0, F, D, b1 - b0,
                                  ptr(self.out[b0:b1]), P)

        def backward(blk):
            b0, b1 = blk
            L.oracle_interact_bwd(ptr(self.go[b0:b1]), ptr(self.dense[b0:b1]), ptr(self.pooled[b0:b1]), 0, F, D,
                                  b1 - b0, P, ptr(self.gd[b0:b1]), ptr(self.gp[b0:b1]))

        def sgd(t):
            q = self.parts[t]
            q["gp"][:, 0, :] = self.gp[:, t, :]
            if q["r1"] > q["r0"]:
                L.oracle_emb_bwd_sgd(ptr(self.tables[q["r0"]:q["r1"]]), ptr(q["rb"]), 1, D, B, ptr(q["idx"]),
                                     ptr(q["off"]), q["idx"].size, ptr(q["gp"]), self.lr, 0, ptr(q["status"]),
                                     None, None)

        with ThreadPoolExecutor(max(1, threads)) as ex:
            t0 = time.perf_counter()
            list(ex.map(lookup, range(F)))
            list(ex.map(interact, blocks))
            list(ex.map(backward, blocks))
            list(ex.map(sgd, range(F)))
            return time.perf_counter() - t0

    def outputs(self):
        return dict(pooled=self.pooled, out=self.out, gd=self.gd, gp=self.gp, tables=self.tables)


def cpu_baseline(w, n_samples: int) -> dict:
    """The oracle on all host cores (threads over tables and sample blocks) and on one core."""
    samples = np.arange(n_samples)
    cores = host_cores()
    dt1 = cpu_oracle_step(w, samples)
    dtn = ThreadedOracleStep(w, samples).run(cores)
    return {"value": round(n_samples / dtn, 1), "unit": "samples/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "one_core": {"value": round(n_samples / dt1, 1), "unit": "samples/s", "cores": 1, "seconds": round(dt1, 3)},
            "sample": f"first {n_samples} of the {w.B} samples of the same batch (tables compacted to the rows "
                      f"they touch); the C oracle, double accumulation, on {cores} threads (lookup and sparse SGD "
                      f"per table, interaction and its backward per block of samples; {dtn:.2f} s) and in one "
                      f"call on one core ({dt1:.2f} s)"}


# ------------------------------------------------------------- GPU benchmark
def sgd_kernels(total_rows: int) -> int:
    """Kernels of one dlrm_emb_bwd_sgd call: keys (which also counts the first radix digit), scan and
    scatter of the first pass, count + scan + scatter of each later pass, segment, fixup."""
    nbits = int(total_rows).bit_length()
    npasses = (nbits + 7) // 8
    return 1 + 2 + 3 * (npasses - 1) + 2


def kernels_per_step(total_rows: int) -> int:
    # the one-pass training forward, interact_bwd, then the sparse SGD's kernels
    return 2 + sgd_kernels(total_rows)


N_BATCHES = 4   # pre-generated index batches the timed loops rotate through


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import dlrm_embeddings_dot_gb300 as dl
    from dlrm_embeddings_dot_gb300 import inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dl.load()
    stream = torch.cuda.Stream(device=dev)
    B = args.batch

    # ---- inputs (rank-specific seed: each replica trains on its own batches).  Four batches over
    # the same tables (the popular rows stay the same) rotate through the timed loops.
    w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, seed=rank, train=True)
    wb = [w] + [inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, seed=rank, train=True, rows=w.rows,
                                    batch=k) for k in range(1, N_BATCHES)]
    F, D, P = w.F, w.D, w.out_cols
    with torch.cuda.stream(stream):
        tables = torch.empty(w.total_rows, D, dtype=torch.float32, device=dev)
        dl.dlrm_synth_fill_uniform(tables, w.table_seed, 0, stream=stream)
        row_base = torch.from_numpy(w.row_base).to(dev)
        # The upstream gradient of a batch alternates its sign from one round of the four batches to
        # the next: a replayed batch with one fixed gradient would grow its hottest rows geometrically
        # over hundreds of steps (the arithmetic is the same either way).
        dbat = [dict(idx=torch.from_numpy(x.indices).to(dev), off=torch.from_numpy(x.offsets).to(dev),
                     dense=torch.from_numpy(x.dense).to(dev), go=torch.from_numpy(x.grad_out).to(dev))
                for x in wb]
        for d in dbat:
            d["go_neg"] = -d["go"]
        pooled = torch.empty(B, F, D, device=dev)
        out = torch.empty(B, P, device=dev)
        gd = torch.empty(B, D, device=dev)
        gp = torch.empty(B, F, D, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        nnz_max = max(x.nnz for x in wb)
        ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(nnz_max, D, w.total_rows), dtype=torch.uint8,
                         device=dev)
    torch.cuda.synchronize()
    nnz = w.nnz

    ev = {k: [] for k in ("emb_interact_fwd", "interact_bwd", "emb_bwd_sgd")}
    nstep = [0]

    def step(record=False):
        k = nstep[0]
        nstep[0] += 1
        d = dbat[k % N_BATCHES]
        go_k = d["go"] if (k // N_BATCHES) % 2 == 0 else d["go_neg"]
        marks = []
        if record:
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            marks[0].record(stream)
        # lookup + interaction in one pass; the pooled rows are written for the backward
        dl.dlrm_emb_interact_fwd_train(tables, row_base, F, D, B, d["idx"], d["off"], d["dense"], pooled, out, P,
                                       status=status, stream=stream)
        if record:
            marks[1].record(stream)
        dl.dlrm_interact_bwd(go_k, d["dense"], pooled, F, D, B, P, gd, gp, stream=stream)
        if record:
            marks[2].record(stream)
        dl.dlrm_emb_bwd_sgd(tables, row_base, w.total_rows, F, D, B, d["idx"], d["off"], gp, LR, ws, status=status,
                            stream=stream)
        if record:
            marks[3].record(stream)
            for name, (a, b) in zip(ev, zip(marks[:-1], marks[1:])):
                ev[name].append((a, b))

    # ---- warm-up
    for _ in range(max(args.warmup, N_BATCHES)):
        step()
    torch.cuda.synchronize()

    # ---- per-op durations (events on the launching stream), separate from the timed loop
    for _ in range(max(8, min(args.steps, 48))):
        step(record=True)
    torch.cuda.synchronize()
    op_ms = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}

    # ---- the same forward as the two separate calls (context for the one-pass forward)
    two = []
    for i in range(max(8, min(args.steps, 48))):
        d = dbat[i % N_BATCHES]
        m = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        m[0].record(stream)
        dl.dlrm_emb_fwd(tables, row_base, F, D, B, d["idx"], d["off"], pooled, status=status, stream=stream)
        m[1].record(stream)
        dl.dlrm_interact_fwd(d["dense"], pooled, F, D, B, out, P, status=status, stream=stream)
        m[2].record(stream)
        two.append(m)
    torch.cuda.synchronize()
    two_ms = {"emb_fwd": statistics.mean(m[0].elapsed_time(m[1]) for m in two),
              "interact_fwd": statistics.mean(m[1].elapsed_time(m[2]) for m in two)}

    # ---- timed region (inputs > L2: the 4.1 GB tables and 0.9 GB pooled/grad tensors)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = reduce_max(t0.elapsed_time(t1), world, dev)
    st = int(status.item())
    value = B * world * args.steps / (ms / 1e3)
    finite = float(torch.isfinite(out).float().mean().item())

    # ---- forward only, configs' fp16 DLRM-default: Zipf 1.05, tensor-core interaction
    wf = inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD, seed=rank)
    wfb = [wf] + [inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD, seed=rank, rows=wf.rows, batch=k)
                  for k in range(1, N_BATCHES)]
    with torch.cuda.stream(stream):
        tab16 = torch.empty(wf.total_rows, D, dtype=torch.float16, device=dev)
        dl.dlrm_synth_fill_uniform(tab16, wf.table_seed, 0, stream=stream)
        rb16 = torch.from_numpy(wf.row_base).to(dev)
        fbat = [dict(idx=torch.from_numpy(x.indices).to(dev), off=torch.from_numpy(x.offsets).to(dev),
                     dense=torch.from_numpy(x.dense.astype(np.float16)).to(dev)) for x in wfb]
        pooled16 = torch.empty(B, F, D, dtype=torch.float16, device=dev)
        out16 = torch.empty(B, P, dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    fk = [0]

    def fstep():
        d = fbat[fk[0] % N_BATCHES]
        fk[0] += 1
        dl.dlrm_emb_fwd(tab16, rb16, F, D, B, d["idx"], d["off"], pooled16, status=status, stream=stream)
        dl.dlrm_interact_fwd(d["dense"], pooled16, F, D, B, out16, P, status=status, stream=stream)

    for _ in range(max(args.warmup, N_BATCHES)):
        fstep()
    fev = []
    for i in range(max(8, min(args.steps, 48))):
        d = fbat[i % N_BATCHES]
        m = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        m[0].record(stream)
        dl.dlrm_emb_fwd(tab16, rb16, F, D, B, d["idx"], d["off"], pooled16, status=status, stream=stream)
        m[1].record(stream)
        dl.dlrm_interact_fwd(d["dense"], pooled16, F, D, B, out16, P, status=status, stream=stream)
        m[2].record(stream)
        fev.append(m)
    torch.cuda.synchronize()
    f_emb = statistics.mean(m[0].elapsed_time(m[1]) for m in fev)
    f_int = statistics.mean(m[1].elapsed_time(m[2]) for m in fev)
    barrier(world)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        fstep()
    f1.record(stream)
    torch.cuda.synchronize()
    fms = reduce_max(f0.elapsed_time(f1), world, dev)
    uk = [0]

    def fused_step():
        d = fbat[uk[0] % N_BATCHES]
        uk[0] += 1
        dl.dlrm_emb_interact_fwd(tab16, rb16, F, D, B, d["idx"], d["off"], d["dense"], out16, P, status=status,
                                 stream=stream)

    for _ in range(max(args.warmup, N_BATCHES)):
        fused_step()
    torch.cuda.synchronize()
    barrier(world)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(args.steps):
        fused_step()
    u1.record(stream)
    torch.cuda.synchronize()
    ums = reduce_max(u0.elapsed_time(u1), world, dev)
    del tab16, pooled16, out16, fbat

    # ---- the same training step in mixed precision (the pages' --amp): fp16
    # interaction tensors on tcgen05, fp32 master tables, static loss scale
    amp_ops = amp_step_ops(dl, wb, torch, dev, stream, status, tables)
    for _ in range(max(args.warmup, N_BATCHES)):
        for _, fn in amp_ops:
            fn()
    barrier(world)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(args.steps):
        for _, fn in amp_ops:
            fn()
    a1.record(stream)
    torch.cuda.synchronize()
    ams = reduce_max(a0.elapsed_time(a1), world, dev)
    del amp_ops

    # ---- end to end through the public API from pinned host buffers.  Every
    # step uploads its own inputs (dense, indices, offsets, upstream gradient)
    # and reads back its own results (interaction output, dense gradient),
    # pipelined as a training loop with a prefetching loader runs: the next
    # batch is uploaded on a copy stream while this step computes, and this
    # step's results are read back on another stream while the next step
    # computes (inputs and outputs double-buffered; the tables are updated in
    # place by every step, so the steps themselves stay in order).
    # Each batch's inputs sit in one pinned buffer (dense | indices | offsets | upstream gradient,
    # 256-byte aligned), uploaded by one copy into a device buffer the calls take views of; the
    # results come back the same way (one copy per step each way: 1.047 against 1.072 ms per step
    # as six separate copies).
    def layout(nbytes):
        offs, o = [], 0
        for n in nbytes:
            offs.append(o)
            o += (n + 255) // 256 * 256
        return offs, o

    def as_bytes(a):
        return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8))

    hb = []
    for x in wb:
        parts = [x.dense, x.indices, x.offsets, x.grad_out]
        offs, tot = layout([a.nbytes for a in parts])
        packed = []
        for go in (x.grad_out, -x.grad_out):
            h = torch.empty(tot, dtype=torch.uint8).pin_memory()
            for a, o in zip(parts[:3] + [go], offs):
                h[o:o + a.nbytes].copy_(as_bytes(a))
            packed.append(h)
        hb.append(dict(buf=packed, offs=offs, nnz=x.nnz))
    in_max = max(h["buf"][0].numel() for h in hb)
    o_offs, o_tot = layout([B * P * 4, B * D * 4])
    h_res = [torch.empty(o_tot, dtype=torch.uint8).pin_memory() for _ in range(2)]
    h2d = hb[0]["buf"][0].numel()
    d2h = o_tot
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        d_in = [torch.empty(in_max, dtype=torch.uint8, device=dev) for _ in range(2)]
        d_res = [torch.empty(o_tot, dtype=torch.uint8, device=dev) for _ in range(2)]
    torch.cuda.synchronize()

    def in_views(buf, h):
        o = h["offs"]
        return (buf[o[0]:o[0] + B * D * 4].view(torch.float32).view(B, D),
                buf[o[1]:o[1] + h["nnz"] * 4].view(torch.int32),
                buf[o[2]:o[2] + (F * B + 1) * 4].view(torch.int32),
                buf[o[3]:o[3] + B * P * 4].view(torch.float32).view(B, P))

    def res_views(buf):
        return (buf[o_offs[0]:o_offs[0] + B * P * 4].view(torch.float32).view(B, P),
                buf[o_offs[1]:o_offs[1] + B * D * 4].view(torch.float32).view(B, D))

    def e2e_steps(n, start=None):
        if start is not None:
            up.wait_event(start)                     # the first upload is inside the timed region
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]

        def upload(k):
            hx = hb[k % N_BATCHES]
            src = hx["buf"][(k // N_BATCHES) % 2]
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(computed[k % 2])     # step k-2 has consumed this input buffer
                d_in[k % 2][:src.numel()].copy_(src, non_blocking=True)
                uploaded[k % 2].record(up)

        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            stream.wait_event(uploaded[k % 2])
            if k >= 2:
                stream.wait_event(read_back[k % 2])    # step k-2's results have left this output buffer
            dense_k, idx_k, off_k, go_k = in_views(d_in[k % 2], hb[k % N_BATCHES])
            out_k, gd_k = res_views(d_res[k % 2])
            dl.dlrm_emb_interact_fwd_train(tables, row_base, F, D, B, idx_k, off_k, dense_k, pooled, out_k, P,
                                           status=status, stream=stream)
            dl.dlrm_interact_bwd(go_k, dense_k, pooled, F, D, B, P, gd_k, gp, stream=stream)
            dl.dlrm_emb_bwd_sgd(tables, row_base, w.total_rows, F, D, B, idx_k, off_k, gp, LR, ws,
                                status=status, stream=stream)
            computed[k % 2].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[k % 2])
                h_res[k % 2].copy_(d_res[k % 2], non_blocking=True)
                read_back[k % 2].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    e2e_steps(N_BATCHES)
    torch.cuda.synchronize()
    e_steps = max(E2E_MIN_STEPS, args.steps)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(e_steps, start=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = reduce_max(e0.elapsed_time(e1), world, dev)
    # the host copies hold what the last two steps left on the device (bit for bit)
    for k in range(2):
        if not torch.equal(h_res[k], d_res[k].cpu()):
            raise RuntimeError("e2e: results read back differ from the device buffers")
    del d_in, d_res, hb

    # ---- roofline of the dominant kernel (algorithmic bytes per launch / event time)
    peaks = measured_peaks()
    # touched rows per batch (each step processes one of the rotated batches)
    unique_rows = statistics.mean(touched_rows(x) for x in wb)
    s = 4  # fp32
    alg = {
        # offsets + index + row read per lookup, pooled row written once; dense read, output written
        "emb_interact_fwd": B * F * (4 + 4 + D * s) + B * F * D * s + B * (D * s + P * s),
        "interact_bwd": B * (P * 4 + D * s + F * D * s + D * 4 + F * D * 4),
        "emb_bwd_sgd": sgd_alg_bytes(nnz, D, unique_rows),
    }
    dom = max(op_ms, key=op_ms.get)
    kernel_names = {"emb_interact_fwd": "emb_interact_regs_kernel", "interact_bwd": "interact_bwd_regs_kernel",
                    "emb_bwd_sgd": f"emb_bwd_sgd ({sgd_kernels(w.total_rows)} kernels)"}
    achieved = alg[dom] / (op_ms[dom] / 1e3) / 1e9
    traffic, traffic_note = ncu_traffic(dom if dom == "emb_bwd_sgd" else kernel_names[dom], batch=B)
    roof = {"bound": "hbm", "kernel": kernel_names[dom], "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "peak_source": peaks["source"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic, "traffic_note": traffic_note,
            "algorithmic_bytes_per_launch": int(alg[dom]), "launch_ms": round(op_ms[dom], 4)}
    op_frac = {k: round(alg[k] / (v / 1e3) / 1e9 / peaks["hbm_gbs"], 4) for k, v in op_ms.items()}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "samples/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Criteo Terabyte not available)",
        "config": {"workload": WORKLOAD, "global_batch": B * world, "per_gpu_batch": B, "tables": F,
                   "embedding_dim": D, "total_rows": w.total_rows, "nnz": nnz, "out_cols": P,
                   "index_batches": N_BATCHES,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (4.1 GB tables, 0.87 GB pooled/grad tensors per step)"},
        "ops_ms": {k: round(v, 4) for k, v in op_ms.items()},
        "ops_hbm_frac": op_frac,
        "fwd_two_calls_ms": {k: round(v, 4) for k, v in two_ms.items()},
        "fwd": {"value": round(B * world * args.steps / (fms / 1e3), 1), "unit": "samples/s",
                "ms_per_step": round(fms / args.steps, 4), "dtype": "f16 storage, f32 accumulate",
                "workload": "dlrm-default 64K forward: 26 single-hot fp16 tables, Zipf 1.05, 480 columns",
                "ops_ms": {"emb_fwd": round(f_emb, 4), "interact_fwd_tcgen05": round(f_int, 4)},
                "alg_GBps": {"emb_fwd": round(B * F * (8 + 2 * D * 2) / (f_emb / 1e3) / 1e9, 1),
                             "interact_fwd": round(B * (D * 2 + F * D * 2 + P * 2) / (f_int / 1e3) / 1e9, 1)},
                "fused": {"value": round(B * world * args.steps / (ums / 1e3), 1), "unit": "samples/s",
                          "ms_per_step": round(ums / args.steps, 4),
                          "entry_point": "dlrm_emb_interact_fwd (lookup + tcgen05 interaction in one kernel)",
                          "alg_GBps": round(B * (F * (8 + D * 2) + D * 2 + P * 2) / (ums / args.steps / 1e3) / 1e9,
                                            1)}},
        "amp_train": {"value": round(B * world * args.steps / (ams / 1e3), 1), "unit": "samples/s",
                      "ms_per_step": round(ams / args.steps, 4),
                      "dtype": "f16 interaction tensors (tcgen05 forward and backward), fp32 master tables",
                      "workload": "the same 64K training step with the pages' mixed precision: pooled rows rounded "
                                  "to fp16, upstream gradient scaled by the static loss scale 1024, SGD on fp16 "
                                  "gradients with lr/1024"},
        "e2e": {"value": round(B * world * e_steps / (ems / 1e3), 1), "unit": "samples/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
                "pipelining": "next batch uploaded and previous results read back on two copy streams while a "
                              "step computes (double-buffered inputs/outputs; each direction one copy of a "
                              "packed pinned buffer per step)"},
        "gpu_launches": kernels_per_step(w.total_rows) * args.steps,
        "clocks": clk,
        "roofline": roof,
        "device_status": st,
        "finite_output_fraction": round(finite, 6),
    }
    del tables, dbat, pooled, out, gd, gp, ws
    torch.cuda.empty_cache()
    if not args.headline_only:
        # every other workload of the pages' configurations, each with its own device-timed and
        # end-to-end figures (rank 0's GPU only: they are context, not the scaled headline)
        line["configs"] = {}
        for name in DEFAULT_CONFIGS:
            line["configs"][name] = measure_config(args, name)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_samples)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def touched_rows(w) -> int:
    """Distinct global rows a batch's indices touch (the rows the sparse update reads and writes)."""
    bag = np.repeat(np.arange(w.F * w.B), np.diff(w.offsets.astype(np.int64)))
    t = bag // w.B
    n = w.row_base[t + 1] - w.row_base[t]
    idx = w.indices.astype(np.int64)
    ok = (idx >= 0) & (idx < n)
    return int(np.unique(w.row_base[t][ok] + idx[ok]).size)


def sgd_alg_bytes(nnz: int, D: int, touched: float, grad_bytes: int = 4) -> float:
    """Algorithmic bytes of one sparse update: per index its key and value (int32 index and
    offset read) and its gradient row; per touched row one read and one write of the fp32 row."""
    return nnz * (4 + 4 + D * grad_bytes) + touched * 2 * D * 4


def run_op(args) -> None:
    """Run one entry point repeatedly on the DLRM-default shapes (for ncu captures)."""
    import torch

    import dlrm_embeddings_dot_gb300 as dl
    from dlrm_embeddings_dot_gb300 import inputs

    dl.load()
    dev = torch.device("cuda", 0)
    B, F, D, P = args.batch, 26, 128, 480
    g = torch.Generator(device=dev).manual_seed(0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.op in ("interact_fwd", "interact_fwd16", "interact_bwd", "interact_bwd16"):
        dt = torch.float16 if args.op in ("interact_fwd16", "interact_bwd16") else torch.float32
        dense = torch.rand(B, D, generator=g, device=dev).to(dt)
        pooled = ((torch.rand(B, F, D, generator=g, device=dev) - 0.5) * 0.1).to(dt)
        out = torch.empty(B, P, dtype=dt, device=dev)
        go = torch.randn(B, P, generator=g, device=dev) * 1e-2
        gd = torch.empty(B, D, device=dev)
        gp = torch.empty(B, F, D, device=dev)

        go16 = (go * 1024.0).to(torch.float16)
        gd16 = torch.empty(B, D, dtype=torch.float16, device=dev)
        gp16 = torch.empty(B, F, D, dtype=torch.float16, device=dev)

        def once():
            if args.op == "interact_bwd":
                dl.dlrm_interact_bwd(go, dense, pooled, F, D, B, P, gd, gp)
            elif args.op == "interact_bwd16":
                dl.dlrm_interact_bwd_f16(go16, dense, pooled, F, D, B, P, gd16, gp16, status=status)
            else:
                dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=status)
    else:
        dt = inputs.F16 if args.op in ("emb_fwd16", "emb_interact16") else inputs.F32
        rows = None
        if args.small_tables:   # ~10x fewer rows: keeps an ncu capture's device memory to a few hundred MB
            rows = inputs.log_uniform_rows(np.random.default_rng(np.random.SeedSequence([0, 11])), 26, 10, 4e5)
        w = inputs.dlrm_default(B=B, dtype=dt, alpha=ALPHA_FWD if dt == inputs.F16 else ALPHA_TRAIN,
                                train=True, rows=rows)
        tt = torch.float16 if dt == inputs.F16 else torch.float32
        tables = torch.empty(w.total_rows, D, dtype=tt, device=dev)
        dl.dlrm_synth_fill_uniform(tables, w.table_seed, 0)
        rb = torch.from_numpy(w.row_base).to(dev)
        idx = torch.from_numpy(w.indices).to(dev)
        off = torch.from_numpy(w.offsets).to(dev)
        pooled = torch.empty(B, F, D, dtype=tt, device=dev)
        gp = torch.randn(B, F, D, generator=g, device=dev) * 1e-2
        ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, D, w.total_rows), dtype=torch.uint8,
                         device=dev)

        dense16 = torch.from_numpy(w.dense.astype(np.float16)).to(dev) if dt == inputs.F16 else None
        out16 = torch.empty(B, P, dtype=torch.float16, device=dev) if dt == inputs.F16 else None
        dense32 = torch.from_numpy(w.dense).to(dev) if dt == inputs.F32 else None
        out32 = torch.empty(B, P, device=dev) if dt == inputs.F32 else None

        def once():
            if args.op == "emb_bwd_sgd":
                dl.dlrm_emb_bwd_sgd(tables, rb, w.total_rows, F, D, B, idx, off, gp, LR, ws, status=status)
            elif args.op == "emb_interact16":
                dl.dlrm_emb_interact_fwd(tables, rb, F, D, B, idx, off, dense16, out16, P, status=status)
            elif args.op == "emb_interact_train":
                dl.dlrm_emb_interact_fwd_train(tables, rb, F, D, B, idx, off, dense32, pooled, out32, P,
                                               status=status)
            else:
                dl.dlrm_emb_fwd(tables, rb, F, D, B, idx, off, pooled, status=status)
    for _ in range(args.warmup):
        once()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        once()
    t1.record()
    torch.cuda.synchronize()
    print(json.dumps({"op": args.op, "batch": B, "ms_per_launch": t0.elapsed_time(t1) / args.steps,
                      "status": int(status.item())}), flush=True)


def _time_ops(torch, stream, ops, steps, warmup):
    """Per-op mean ms (events around each op) and total ms per step (one event pair)."""
    for _ in range(warmup):
        for _, fn in ops:
            fn()
    torch.cuda.synchronize()
    per = {name: 0.0 for name, _ in ops}
    for _ in range(steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)]
        ev[0].record(stream)
        for k, (_, fn) in enumerate(ops):
            fn()
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        for k, (name, _) in enumerate(ops):
            per[name] += ev[k].elapsed_time(ev[k + 1])
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        for _, fn in ops:
            fn()
    t1.record(stream)
    torch.cuda.synchronize()
    return {k: v / steps for k, v in per.items()}, t0.elapsed_time(t1) / steps


CONFIGS = {
    "tiny": "batch 256, 3 fp32 tables x 1000 rows x 16, one uniform index per feature, 22 outputs; forward",
    "tiny-train": "the tiny slice with Zipf 1.2 indices: forward + interaction backward + sparse SGD (lr 0.1)",
    "default-fwd": "batch 65536, 26 single-hot fp16 tables (rows log-uniform 10..4e6), D=128, Zipf 1.05, 480 "
                   "columns; forward (lookup + tcgen05 interaction)",
    "train-64k": WORKLOAD,
    "multi-hot": "batch 16384, 26 fp32 tables x 1e6 rows x 128, pooling U{1..100}, Zipf 1.05; forward lookup, "
                 "then backward + SGD from an N(0,1e-2) grad_pooled",
    "large-tables": "26 fp16 tables D=128 (three of 40M rows, 23 log-uniform 10..4e6), single-hot Zipf 1.05; "
                    "forward at batch 1K..1M",
    "bottom-mlp": "bottom MLP 13 -> 512 -> 256 -> 128 (linear + ReLU, fp16 tensors, fp32 accumulate) on the "
                  "tensor cores, batch 65536, lognormal(0,1) dense features; and MLP + fused lookup/interaction "
                  "(the whole embedding-side forward from raw features)",
    "train-64k-amp": "the 64K training step in mixed precision (the pages' --amp): fp32 master tables pooled to "
                     "fp16, fp16 dense, tcgen05 interaction forward and backward, upstream gradient N(0,1e-2) "
                     "scaled by the static loss scale 1024 in fp16, sparse SGD on the fp16 gradients with lr/1024",
    "default-fwd-uniform": "control: the default-fwd shapes with uniform indices (no Zipf reuse, so algorithmic "
                           "bytes ~ DRAM bytes)",
    "multi-hot-uniform": "control: the multi-hot shapes with uniform indices (no Zipf reuse); forward lookup, then "
                         "backward + SGD",
}


# the workloads the default run measures besides the headline (which is train-64k)
DEFAULT_CONFIGS = ["tiny", "tiny-train", "default-fwd", "default-fwd-uniform", "train-64k-amp", "multi-hot",
                   "multi-hot-uniform", "large-tables", "bottom-mlp"]


def _roofline(alg: dict, per: dict, peaks: dict) -> dict:
    """The op with the largest mean time, its algorithmic bytes over that time against HBM."""
    dom = max(per, key=per.get)
    achieved = alg[dom] / (per[dom] / 1e3) / 1e9
    return {"bound": "hbm", "op": dom, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "peak_source": peaks["source"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "bytes": "algorithmic (every lookup counted as a row read: Zipf-hot rows served by L2 count too)"}


def _pack_host(torch, parts):
    """One pinned buffer holding the device tensors' bytes, 256-byte aligned, in order."""
    offs, tot = _pack_layout([t.numel() * t.element_size() for _, t in parts])
    h = torch.empty(tot, dtype=torch.uint8).pin_memory()
    for (_, t), o in zip(parts, offs):
        n = t.numel() * t.element_size()
        h[o:o + n].copy_(t.detach().contiguous().view(-1).view(torch.uint8).cpu())
    return h


def _pack_layout(nbytes):
    offs, o = [], 0
    for n in nbytes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    return offs, o


def _packed_views(torch, dev, parts):
    """A device buffer laid out as _pack_host lays the parts out, and views of it shaped like them."""
    offs, tot = _pack_layout([t.numel() * t.element_size() for _, t in parts])
    buf = torch.empty(tot, dtype=torch.uint8, device=dev)
    views = {}
    for (name, t), o in zip(parts, offs):
        n = t.numel() * t.element_size()
        views[name] = buf[o:o + n].view(t.dtype).view(t.shape)
    return buf, views


def _e2e_pipelined(torch, stream, ops, bind, d_in, h_in, d_out, steps: int, batch: int) -> dict:
    """The step through the public API with its inputs copied up from pinned host memory and its
    results read back, every step, inside the timed region, in two schedules: pipelined (the next
    step's inputs go up on one copy stream and the previous step's results come down on another
    while a step computes) and in stream order; the faster is reported, the other beside it.
    d_in / d_out: the two slots' packed device buffers; bind(s) points the calls at slot s."""
    up, down = torch.cuda.Stream(device=stream.device), torch.cuda.Stream(device=stream.device)
    h_out = [torch.empty(d_out[0].numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]

    def run(n, start=None):
        if start is not None:
            up.wait_event(start)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]

        def upload(k):
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(computed[k % 2])     # step k-2 has consumed this input buffer
                d_in[k % 2].copy_(h_in, non_blocking=True)
                uploaded[k % 2].record(up)

        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            stream.wait_event(uploaded[k % 2])
            if k >= 2:
                stream.wait_event(read_back[k % 2])    # step k-2's results have left this output buffer
            bind(k % 2)
            for _, fn in ops:
                fn()
            computed[k % 2].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[k % 2])
                h_out[k % 2].copy_(d_out[k % 2], non_blocking=True)
                read_back[k % 2].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    def in_order(n):
        # small steps: the cross-stream waits cost more than the overlap saves, so the copies and
        # the calls also run in stream order on one slot
        bind(0)
        with torch.cuda.stream(stream):
            for _ in range(n):
                d_in[0].copy_(h_in, non_blocking=True)
                for _, fn in ops:
                    fn()
                h_out[0].copy_(d_out[0], non_blocking=True)

    def timed(fn):
        fn(4)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if fn is run:
            run(steps, start=e0)
        else:
            fn(steps)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_pipe = timed(run)
    for k in range(2):
        if not torch.equal(h_out[k], d_out[k].cpu()):
            raise RuntimeError("e2e: results read back differ from the device buffers")
    ms_seq = timed(in_order)
    if not torch.equal(h_out[0], d_out[0].cpu()):
        raise RuntimeError("e2e: results read back differ from the device buffers")
    pipe = ms_pipe <= ms_seq
    ms, other = (ms_pipe, ms_seq) if pipe else (ms_seq, ms_pipe)
    how = ("next step's inputs up and previous step's results back on two copy streams while a step computes "
           "(double-buffered, each direction one copy of a packed buffer)") if pipe else \
          "in stream order on one buffer set (each direction one copy of a packed buffer)"
    return {"value": round(batch / (ms / 1e3), 1), "unit": "samples/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h_in.numel()), "d2h_bytes_per_step": int(d_out[0].numel()),
            "pipelining": how,
            "other_schedule": {"value": round(batch / (other / 1e3), 1), "ms_per_step": round(other, 4),
                               "pipelined": not pipe}}


def _e2e(torch, stream, ops, h2d: list, d2h: list, steps: int, batch: int) -> dict:
    """The same step through the public API with every per-step input copied up from pinned host
    memory and every per-step output read back, in stream order (no overlap), inside the timed
    region.  h2d / d2h: lists of (device tensor, pinned host tensor)."""
    def once():
        for dv, hv in h2d:
            dv.copy_(hv, non_blocking=True)
        for _, fn in ops:
            fn()
        for dv, hv in d2h:
            hv.copy_(dv, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            once()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            once()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(batch / (ms / 1e3), 1), "unit": "samples/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(sum(h.numel() * h.element_size() for _, h in h2d)),
            "d2h_bytes_per_step": int(sum(h.numel() * h.element_size() for _, h in d2h)),
            "pipelining": "none (copies and kernels in one stream)"}


def _pinned(torch, t):
    return torch.empty(t.shape, dtype=t.dtype).pin_memory()


def run_bottom_mlp(args, dl, inputs, torch, dev, stream, status) -> list:
    """The tensor-core bottom MLP alone, then MLP + fused lookup/interaction."""
    B = args.batch
    dims = [13, 512, 256, 128]
    x = np.random.default_rng(np.random.SeedSequence([0, 3])).lognormal(0.0, 1.0, size=(B, 13)).astype(np.float32)
    W, bias = inputs.mlp_layers(dims, seed=0)
    wp, bp = inputs.mlp_pack(W, bias)
    xd, wd, bd = (torch.from_numpy(a).to(dev) for a in (x, wp, bp))
    ws = torch.empty(dl.dlrm_bottom_mlp_workspace_size(B, dims), dtype=torch.uint8, device=dev)
    dense = torch.empty(B, 128, dtype=torch.float16, device=dev)
    mlp = ("bottom_mlp", lambda: dl.dlrm_bottom_mlp_fwd(xd, dims, wd, bd, dense, ws, status=status, stream=stream))
    per, ms = _time_ops(torch, stream, [mlp], args.steps, args.warmup)
    flop = 2.0 * B * sum(dims[l] * dims[l + 1] for l in range(3))
    peak = measured_peaks()
    tflops = flop / (ms / 1e3) / 1e12
    w = inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD)
    with torch.cuda.stream(stream):
        tab = torch.empty(w.total_rows, w.D, dtype=torch.float16, device=dev)
        dl.dlrm_synth_fill_uniform(tab, w.table_seed, 0, stream=stream)
        rb, idx, off = (torch.from_numpy(a).to(dev) for a in (w.row_base, w.indices, w.offsets))
    torch.cuda.synchronize()
    out = torch.empty(B, w.out_cols, dtype=torch.float16, device=dev)
    fused = ("emb_interact_fwd", lambda: dl.dlrm_emb_interact_fwd(tab, rb, w.F, w.D, B, idx, off, dense, out,
                                                                 w.out_cols, status=status, stream=stream))
    per2, ms2 = _time_ops(torch, stream, [mlp, fused], args.steps, args.warmup)
    e2e = _e2e(torch, stream, [mlp, fused],
               [(xd, torch.from_numpy(x).pin_memory()), (idx, torch.from_numpy(w.indices).pin_memory()),
                (off, torch.from_numpy(w.offsets).pin_memory())], [(out, _pinned(torch, out))],
               max(E2E_MIN_STEPS, args.steps), B)
    return [{
        "config": "bottom-mlp", "workload": CONFIGS["bottom-mlp"], "batch": B, "steps": args.steps,
        "ms_per_step": round(ms, 4), "samples_per_s": round(B / (ms / 1e3), 1),
        "tflops": round(tflops, 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(tflops / peak["bf16_tflops"], 4),
                     "peak_note": f"dense bf16 burst ({peak['source']}); fp16 has the same nominal rate"},
        "with_fused_fwd": {"ms_per_step": round(ms2, 4), "samples_per_s": round(B / (ms2 / 1e3), 1),
                           "ops_ms": {k: round(v, 4) for k, v in per2.items()}, "e2e": e2e},
        "device_status": int(status.item())}]


LOSS_SCALE = 1024.0


def amp_step_ops(dl, wb, torch, dev, stream, status, tab, buffers=None, alternate=True, io=None):
    """The mixed-precision training step's four calls, on device buffers; the calls rotate
    through the batches of ``wb`` (a workload or a list of workloads over the same tables).
    ``buffers``, if a dict, receives the first batch's input and output tensors; ``io``, if a
    dict, is read at each call instead: its "in" (idx, off, dense, g), "out" and "gd" tensors."""
    wb = wb if isinstance(wb, list) else [wb]
    w = wb[0]
    F, D, B, P = w.F, w.D, w.B, w.out_cols
    rb = torch.from_numpy(w.row_base).to(dev)
    bat = [dict(idx=torch.from_numpy(x.indices).to(dev), off=torch.from_numpy(x.offsets).to(dev),
                dense=torch.from_numpy(x.dense.astype(np.float16)).to(dev),
                g=torch.from_numpy((x.grad_out.astype(np.float64) * LOSS_SCALE).astype(np.float16)).to(dev))
           for x in wb]
    for d in bat:
        d["g_neg"] = -d["g"]
    pooled = torch.empty(B, F, D, dtype=torch.float16, device=dev)
    out = torch.empty(B, P, dtype=torch.float16, device=dev)
    gd = torch.empty(B, D, dtype=torch.float16, device=dev)
    gp = torch.empty(B, F, D, dtype=torch.float16, device=dev)
    ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(max(x.nnz for x in wb), D, w.total_rows), dtype=torch.uint8,
                     device=dev)
    lr = float(np.float32(w.lr / LOSS_SCALE))
    if buffers is not None:
        buffers.update(bat[0], out=out, gd=gd)
    # step k uses batch k % n; a batch's upstream gradient alternates its sign from one round of the
    # batches to the next (keeps the replayed tables bounded)
    k = [0]
    cur = {}

    def fwd():
        if io is not None:
            d = io["in"]
            cur["d"], cur["g"] = d, d["g"]
        else:
            d = bat[k[0] % len(bat)]
            cur["d"], cur["g"] = d, d["g"] if not alternate or (k[0] // len(bat)) % 2 == 0 else d["g_neg"]
        k[0] += 1
        dl.dlrm_emb_fwd(tab, rb, F, D, B, d["idx"], d["off"], pooled, flags=dl.DLRM_FLAG_POOLED_F16, status=status,
                        stream=stream)

    return [
        ("emb_fwd", fwd),
        ("interact_fwd", lambda: dl.dlrm_interact_fwd(cur["d"]["dense"], pooled, F, D, B,
                                                      out if io is None else io["out"], P, status=status,
                                                      stream=stream)),
        ("interact_bwd", lambda: dl.dlrm_interact_bwd_f16(cur["g"], cur["d"]["dense"], pooled, F, D, B, P,
                                                          gd if io is None else io["gd"], gp, status=status,
                                                          stream=stream)),
        ("emb_bwd_sgd", lambda: dl.dlrm_emb_bwd_sgd(tab, rb, w.total_rows, F, D, B, cur["d"]["idx"],
                                                    cur["d"]["off"], gp, lr, ws, flags=dl.DLRM_FLAG_GRAD_F16,
                                                    status=status, stream=stream)),
    ]


def run_train_amp(args, dl, inputs, torch, dev, stream, status) -> list:
    B = args.batch
    w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, train=True)
    wb = [w] + [inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, train=True, rows=w.rows, batch=k)
                for k in range(1, N_BATCHES)]
    with torch.cuda.stream(stream):
        tab = torch.empty(w.total_rows, w.D, dtype=torch.float32, device=dev)
        dl.dlrm_synth_fill_uniform(tab, w.table_seed, 0, stream=stream)
    torch.cuda.synchronize()
    ops = amp_step_ops(dl, wb, torch, dev, stream, status, tab)
    per, ms = _time_ops(torch, stream, ops, args.steps, args.warmup)
    F, D, P, nnz = w.F, w.D, w.out_cols, w.nnz
    # end to end on one batch: its indices, offsets, dense rows and scaled gradient up, the
    # interaction output and the dense gradient back, every step (both schedules, as the configs)
    bufs = {}
    amp_step_ops(dl, [w], torch, dev, stream, status, tab, buffers=bufs, alternate=False)
    in_parts = [(n_, bufs[n_]) for n_ in ("idx", "off", "dense", "g")]
    out_parts = [("out", bufs["out"]), ("gd", bufs["gd"])]
    h_in = _pack_host(torch, in_parts)
    slots_in = [_packed_views(torch, dev, in_parts) for _ in range(2)]
    slots_out = [_packed_views(torch, dev, out_parts) for _ in range(2)]
    io = {}
    eops = amp_step_ops(dl, [w], torch, dev, stream, status, tab, alternate=False, io=io)

    def bind(slot):
        io["in"] = slots_in[slot][1]
        io["out"] = slots_out[slot][1]["out"]
        io["gd"] = slots_out[slot][1]["gd"]

    e2e = _e2e_pipelined(torch, stream, eops, bind, [x[0] for x in slots_in], h_in, [x[0] for x in slots_out],
                         max(E2E_MIN_STEPS, args.steps), B)
    del slots_in, slots_out, bufs
    touched = statistics.mean(touched_rows(x) for x in wb)
    alg = {"emb_fwd": nnz * (4 + 4 + D * 4) + B * F * D * 2,
           "interact_fwd": B * (D * 2 + F * D * 2 + P * 2),
           "interact_bwd": B * (P * 2 + D * 2 + F * D * 2 + D * 2 + F * D * 2),
           "emb_bwd_sgd": sgd_alg_bytes(nnz, D, touched, grad_bytes=2)}
    return [{
        "config": "train-64k-amp", "workload": CONFIGS["train-64k-amp"], "batch": B, "nnz": nnz,
        "index_batches": N_BATCHES, "steps": args.steps, "ms_per_step": round(ms, 4),
        "step_samples_per_s": round(B / (ms / 1e3), 1),
        "ops_ms": {k: round(v, 4) for k, v in per.items()},
        "alg_GBps": {k: round(alg[k] / (v / 1e3) / 1e9, 1) for k, v in per.items()},
        "roofline": _roofline(alg, per, measured_peaks()), "e2e": e2e,
        "device_status": int(status.item())}]


def measure_config(args, name) -> list:
    """Measure one workload of the pages' configurations; one result per batch size."""
    import torch

    import dlrm_embeddings_dot_gb300 as dl
    from dlrm_embeddings_dot_gb300 import inputs

    dl.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if name == "bottom-mlp":
        return run_bottom_mlp(args, dl, inputs, torch, dev, stream, status)
    if name == "train-64k-amp":
        return run_train_amp(args, dl, inputs, torch, dev, stream, status)
    peaks = measured_peaks()

    def setup(w, tt):
        with torch.cuda.stream(stream):
            tab = torch.empty(w.total_rows, w.D, dtype=tt, device=dev)
            dl.dlrm_synth_fill_uniform(tab, w.table_seed, 0, stream=stream)
        torch.cuda.synchronize()
        return tab, torch.from_numpy(w.row_base).to(dev)

    def make(B, batch=0, rows=None):
        if name in ("tiny", "tiny-train"):
            return inputs.tiny_slice(seed=batch, train=(name == "tiny-train"))
        if name in ("default-fwd", "default-fwd-uniform"):
            return inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD, rows=rows, batch=batch,
                                       uniform_indices=name.endswith("-uniform"))
        if name == "train-64k":
            return inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, train=True, rows=rows, batch=batch)
        if name in ("multi-hot", "multi-hot-uniform"):
            return inputs.multi_hot(B=16384 if B == BATCH else B, uniform_indices=name.endswith("-uniform"),
                                    batch=batch)
        return inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD, rows=inputs.large_tables_rows(),
                                   batch=batch)

    results = []
    batches = [args.batch] if name != "large-tables" else [1024, 4096, 16384, 65536, 262144, 1048576]
    for B in batches:
        w = make(B)
        # rotate four index batches over the same tables where they are cheap to draw (up to 4M
        # indices); the tiny slice draws its other batches with other seeds (its tables are the
        # same 3 x 1000 rows for every seed)
        nb = N_BATCHES if w.nnz <= 4_000_000 else 1
        wb = [w] + [make(B, batch=k, rows=w.rows) for k in range(1, nb)]
        tt = torch.float16 if w.dtype == inputs.F16 else torch.float32
        es = 2 if tt == torch.float16 else 4
        F, D, Bw, P = w.F, w.D, w.B, w.out_cols
        tab, rb = setup(w, tt)
        with torch.cuda.stream(stream):
            bat = [dict(idx=torch.from_numpy(x.indices).to(dev), off=torch.from_numpy(x.offsets).to(dev),
                        dense=torch.from_numpy(x.dense.astype(np.float16 if tt == torch.float16 else np.float32))
                        .to(dev)) for x in wb]
        torch.cuda.synchronize()
        cur = {"k": 0, "d": bat[0]}

        def nxt():
            cur["d"] = bat[cur["k"] % len(bat)]
            cur["k"] += 1

        pooled = torch.empty(Bw, F, D, dtype=tt, device=dev)
        out = torch.empty(Bw, P, dtype=tt, device=dev)
        multi = name.startswith("multi-hot")
        train = name in ("tiny-train", "train-64k") or multi

        def emb_fwd():
            nxt()
            dl.dlrm_emb_fwd(tab, rb, F, D, Bw, cur["d"]["idx"], cur["d"]["off"], pooled, status=status, stream=stream)

        ops = [("emb_fwd", emb_fwd)]
        if not multi:
            ops.append(("interact_fwd", lambda: dl.dlrm_interact_fwd(cur["d"]["dense"], pooled, F, D, Bw, out, P,
                                                                     status=status, stream=stream)))
        ws = gp = go = gd = None
        if train:
            gp = torch.empty(Bw, F, D, device=dev)
            ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(max(x.nnz for x in wb), D, w.total_rows),
                             dtype=torch.uint8, device=dev)
            if multi:
                gp.normal_(0.0, 1e-2)
            else:
                for d, x in zip(bat, wb):
                    d["go"] = torch.from_numpy(x.grad_out).to(dev)
                gd = torch.empty(Bw, D, device=dev)
                ops.append(("interact_bwd", lambda: dl.dlrm_interact_bwd(cur["d"]["go"], cur["d"]["dense"], pooled,
                                                                         F, D, Bw, P, gd, gp, stream=stream)))
            ops.append(("emb_bwd_sgd", lambda: dl.dlrm_emb_bwd_sgd(tab, rb, w.total_rows, F, D, Bw, cur["d"]["idx"],
                                                                   cur["d"]["off"], gp, w.lr, ws, status=status,
                                                                   stream=stream)))
        per, ms = _time_ops(torch, stream, ops, args.steps, max(args.warmup, len(bat)))
        fused_train = None
        if train and not multi and tt == torch.float32 and F in (8, 26) and D == 128:
            def fwd_train():
                nxt()
                dl.dlrm_emb_interact_fwd_train(tab, rb, F, D, Bw, cur["d"]["idx"], cur["d"]["off"],
                                               cur["d"]["dense"], pooled, out, P, status=status, stream=stream)
            fops = [("emb_interact_fwd_train", fwd_train)] + ops[2:]
            fper, fms = _time_ops(torch, stream, fops, args.steps, args.warmup)
            fused_train = {"ms_per_step": round(fms, 4), "step_samples_per_s": round(Bw / (fms / 1e3), 1),
                           "ops_ms": {k: round(v, 4) for k, v in fper.items()}}
        if multi and tt == torch.float32 and F in (8, 26) and D == 128:
            # the forward of a multi-hot batch: lookup + interaction as two calls, and the training
            # forward call (which itself runs two launches for bags this large); 480 columns rather
            # than 479, as the one-pass kernel writes whole float4 columns
            P4 = (P + 3) // 4 * 4
            out4 = torch.empty(Bw, P4, dtype=tt, device=dev)
            two = [ops[0], ("interact_fwd", lambda: dl.dlrm_interact_fwd(cur["d"]["dense"], pooled, F, D, Bw, out4,
                                                                         P4, status=status, stream=stream))]

            def fwd_train4():
                nxt()
                dl.dlrm_emb_interact_fwd_train(tab, rb, F, D, Bw, cur["d"]["idx"], cur["d"]["off"],
                                               cur["d"]["dense"], pooled, out4, P4, status=status, stream=stream)
            _, two_ms = _time_ops(torch, stream, two, args.steps, args.warmup)
            _, one_ms = _time_ops(torch, stream, [("emb_interact_fwd_train", fwd_train4)], args.steps, args.warmup)
            fused_train = {"fwd_two_calls_ms": round(two_ms, 4), "fwd_train_call_ms": round(one_ms, 4)}
        fused_ms = None
        if tt == torch.float16 and not train:
            def fused():
                nxt()
                dl.dlrm_emb_interact_fwd(tab, rb, F, D, Bw, cur["d"]["idx"], cur["d"]["off"], cur["d"]["dense"], out,
                                         P, status=status, stream=stream)
            _, fused_ms = _time_ops(torch, stream, [("emb_interact_fwd", fused)], args.steps, args.warmup)
        nnz = w.nnz
        touched = statistics.mean(touched_rows(x) for x in wb) if train else 0
        alg = {"emb_fwd": nnz * (4 + D * es) + Bw * F * (4 + D * es),
               "interact_fwd": Bw * (D * es + F * D * es + P * es),
               "interact_bwd": Bw * (P * 4 + D * es + F * D * es + D * 4 + F * D * 4),
               "emb_bwd_sgd": sgd_alg_bytes(nnz, D, touched)}
        fwd_ms = per["emb_fwd"] + per.get("interact_fwd", 0.0)
        # end to end: one batch's inputs up from pinned memory and the step's results back, every
        # step, pipelined as in the headline (inputs and outputs double-buffered, each direction one
        # copy of a packed buffer per step); the calls take views of the slot's device buffers
        d0 = bat[0]
        in_parts = [("idx", d0["idx"]), ("off", d0["off"])]
        if not multi:
            in_parts.append(("dense", d0["dense"]))
        if train and not multi:
            in_parts.append(("go", d0["go"]))
        if multi:
            in_parts.append(("gp", gp))
        out_parts = [("out", out)] if not multi else [("pooled", pooled)]
        if train and not multi:
            out_parts.append(("gd", gd))
        h_in = _pack_host(torch, in_parts)
        slots_in = [_packed_views(torch, dev, in_parts) for _ in range(2)]
        slots_out = [_packed_views(torch, dev, out_parts) for _ in range(2)]
        bat_save = bat

        def bind(slot):
            nonlocal bat, out, gd, pooled, gp
            v, o = slots_in[slot][1], slots_out[slot][1]
            bat = [{k_: v[k_] for k_ in ("idx", "off", "dense", "go") if k_ in v}]
            cur["k"] = 0
            gp = v.get("gp", gp)
            out = o.get("out", out)
            gd = o.get("gd", gd)
            pooled = o.get("pooled", pooled)

        e2e = _e2e_pipelined(torch, stream, ops, bind, [x[0] for x in slots_in], h_in,
                             [x[0] for x in slots_out], max(E2E_MIN_STEPS, args.steps), Bw)
        bat = bat_save
        del slots_in, slots_out
        line = {"config": name, "workload": CONFIGS[name], "batch": Bw, "nnz": nnz, "index_batches": len(wb),
                "steps": args.steps, "ms_per_step": round(ms, 4), "ops_ms": {k: round(v, 4) for k, v in per.items()},
                "alg_GBps": {k: round(alg[k] / (v / 1e3) / 1e9, 1) for k, v in per.items()},
                "fwd_samples_per_s": round(Bw / (fwd_ms / 1e3), 1),
                "step_samples_per_s": round(Bw / (ms / 1e3), 1),
                "roofline": _roofline(alg, per, peaks), "e2e": e2e, "device_status": int(status.item())}
        if train:
            line["touched_rows"] = round(touched, 1)
        if fused_train is not None:
            line["one_pass_forward"] = fused_train
        if fused_ms is not None:
            line["fused_fwd"] = {"ms": round(fused_ms, 4), "samples_per_s": round(Bw / (fused_ms / 1e3), 1),
                                 "alg_GBps": round(Bw * (F * (8 + D * 2) + D * 2 + P * 2) / (fused_ms / 1e3) / 1e9,
                                                   1)}
        results.append(line)
        del tab, pooled, out, bat, wb, ws, gp, gd
        torch.cuda.empty_cache()
    return results


def run_config(args, name) -> None:
    for line in measure_config(args, name):
        print(json.dumps(line), flush=True)


def run_reference(args) -> None:
    """The CPU oracle, timed as it stands on all host cores, on bounded samples of the workload:
    step k runs the oracle on samples [k*n, (k+1)*n) (wrapping) of the 65,536-sample batch."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from dlrm_embeddings_dot_gb300 import inputs
    w = inputs.dlrm_default(B=BATCH, dtype=inputs.F32, alpha=ALPHA_TRAIN, seed=0, train=True)
    n = args.ref_samples
    cores = host_cores()
    steps = [ThreadedOracleStep(w, np.arange(n) + (i * n) % (w.B - n)) for i in range(args.warmup + args.steps)]
    for i in range(args.warmup):
        steps[i].run(cores)
    total = 0.0
    for i in range(args.steps):
        total += steps[args.warmup + i].run(cores)
    value = n * args.steps / total
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "samples/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": BATCH, "per_gpu_batch": BATCH,
                   "samples_per_step": n},
        "cpu_baseline": {"value": round(value, 1), "unit": "samples/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{n} samples of the 65,536-sample batch per step (ms_per_step is the time of "
                                   f"that slice, not of the whole batch); the C oracle on {cores} threads"},
        "e2e": {"value": round(value, 1), "unit": "samples/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=BATCH)
    ap.add_argument("--cpu-samples", type=int, default=32768,
                    help="samples of the batch the CPU-oracle baseline runs on (about 10 s of CPU)")
    ap.add_argument("--ref-samples", type=int, default=4096,
                    help="samples per step of the --impl reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="the headline line without the other workloads' measurements")
    ap.add_argument("--config", choices=sorted(CONFIGS), action="append",
                    help="measure one of the pages' workloads instead of the headline step (repeatable)")
    ap.add_argument("--op", choices=["emb_fwd", "emb_fwd16", "interact_fwd", "interact_fwd16", "interact_bwd",
                                     "interact_bwd16",
                                     "emb_bwd_sgd", "emb_interact16", "emb_interact_train"],
                    help="time one entry point alone on the DLRM-default shapes (used for ncu captures)")
    ap.add_argument("--small-tables", action="store_true",
                    help="with --op: tables with 10x fewer rows (log-uniform in [10, 4e5])")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.config:
        for name in args.config:
            run_config(args, name)
    elif args.op:
        run_op(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
