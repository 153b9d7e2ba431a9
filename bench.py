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


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        e = json.load(f).get(kernel)
    if not e or e.get("source_digest") != source_digest(e.get("source_files", [])):
        return None
    return e.get("dram_bytes_per_launch")


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


def cpu_baseline(w, n_samples: int) -> dict:
    samples = np.arange(n_samples)
    dt = cpu_oracle_step(w, samples)
    return {"value": n_samples / dt, "unit": "samples/s", "cores": 1, "kind": "oracle",
            "sample": f"first {n_samples} of the {w.B} samples of the same batch (tables compacted to the "
                      f"rows they touch); single-threaded C oracle, double accumulation; {dt:.2f} s"}


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

    # ---- inputs (rank-specific seed: each replica trains on its own batch)
    w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, seed=rank, train=True)
    F, D, P = w.F, w.D, w.out_cols
    with torch.cuda.stream(stream):
        tables = torch.empty(w.total_rows, D, dtype=torch.float32, device=dev)
        dl.dlrm_synth_fill_uniform(tables, w.table_seed, 0, stream=stream)
        row_base = torch.from_numpy(w.row_base).to(dev)
        idx = torch.from_numpy(w.indices).to(dev)
        off = torch.from_numpy(w.offsets).to(dev)
        dense = torch.from_numpy(w.dense).to(dev)
        grad_out = torch.from_numpy(w.grad_out).to(dev)
        # The same synthetic batch is replayed every step; with one fixed upstream
        # gradient the hottest rows would grow geometrically over hundreds of
        # steps.  Alternating its sign keeps the replayed tables bounded (the
        # arithmetic is the same either way).
        grad_out_neg = -grad_out
        pooled = torch.empty(B, F, D, device=dev)
        out = torch.empty(B, P, device=dev)
        gd = torch.empty(B, D, device=dev)
        gp = torch.empty(B, F, D, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, D, w.total_rows), dtype=torch.uint8,
                         device=dev)
    torch.cuda.synchronize()
    nnz = w.nnz

    ev = {k: [] for k in ("emb_interact_fwd", "interact_bwd", "emb_bwd_sgd")}

    nstep = [0]

    def step(record=False):
        go_k = grad_out if nstep[0] % 2 == 0 else grad_out_neg
        nstep[0] += 1
        marks = []
        if record:
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            marks[0].record(stream)
        # lookup + interaction in one pass; the pooled rows are written for the backward
        dl.dlrm_emb_interact_fwd_train(tables, row_base, F, D, B, idx, off, dense, pooled, out, P, status=status,
                                       stream=stream)
        if record:
            marks[1].record(stream)
        dl.dlrm_interact_bwd(go_k, dense, pooled, F, D, B, P, gd, gp, stream=stream)
        if record:
            marks[2].record(stream)
        dl.dlrm_emb_bwd_sgd(tables, row_base, w.total_rows, F, D, B, idx, off, gp, LR, ws, status=status,
                            stream=stream)
        if record:
            marks[3].record(stream)
            for k, (a, b) in zip(ev, zip(marks[:-1], marks[1:])):
                ev[k].append((a, b))

    # ---- warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- per-op durations (events on the launching stream), separate from the timed loop
    for _ in range(max(5, min(args.steps, 50))):
        step(record=True)
    torch.cuda.synchronize()
    op_ms = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}

    # ---- the same forward as the two separate calls (context for the one-pass forward)
    two = []
    for _ in range(max(5, min(args.steps, 50))):
        m = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        m[0].record(stream)
        dl.dlrm_emb_fwd(tables, row_base, F, D, B, idx, off, pooled, status=status, stream=stream)
        m[1].record(stream)
        dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=status, stream=stream)
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
    with torch.cuda.stream(stream):
        tab16 = torch.empty(wf.total_rows, D, dtype=torch.float16, device=dev)
        dl.dlrm_synth_fill_uniform(tab16, wf.table_seed, 0, stream=stream)
        rb16 = torch.from_numpy(wf.row_base).to(dev)
        idx16 = torch.from_numpy(wf.indices).to(dev)
        off16 = torch.from_numpy(wf.offsets).to(dev)
        dense16 = torch.from_numpy(wf.dense.astype(np.float16)).to(dev)
        pooled16 = torch.empty(B, F, D, dtype=torch.float16, device=dev)
        out16 = torch.empty(B, P, dtype=torch.float16, device=dev)
    torch.cuda.synchronize()

    def fstep():
        dl.dlrm_emb_fwd(tab16, rb16, F, D, B, idx16, off16, pooled16, status=status, stream=stream)
        dl.dlrm_interact_fwd(dense16, pooled16, F, D, B, out16, P, status=status, stream=stream)

    for _ in range(args.warmup):
        fstep()
    fev = []
    for _ in range(max(5, min(args.steps, 50))):
        m = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        m[0].record(stream)
        dl.dlrm_emb_fwd(tab16, rb16, F, D, B, idx16, off16, pooled16, status=status, stream=stream)
        m[1].record(stream)
        dl.dlrm_interact_fwd(dense16, pooled16, F, D, B, out16, P, status=status, stream=stream)
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

    def fused_step():
        dl.dlrm_emb_interact_fwd(tab16, rb16, F, D, B, idx16, off16, dense16, out16, P, status=status,
                                 stream=stream)

    for _ in range(args.warmup):
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
    del tab16, pooled16, out16

    # ---- the same training step in mixed precision (the pages' --amp): fp16
    # interaction tensors on tcgen05, fp32 master tables, static loss scale
    amp_ops = amp_step_ops(dl, w, torch, dev, stream, status, tables)
    for _ in range(args.warmup):
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
    h_dense = torch.from_numpy(w.dense).pin_memory()
    h_idx = torch.from_numpy(w.indices).pin_memory()
    h_off = torch.from_numpy(w.offsets).pin_memory()
    h_go = [torch.from_numpy(w.grad_out).pin_memory(), torch.from_numpy(-w.grad_out).pin_memory()]
    h_out = [torch.empty(B, P).pin_memory() for _ in range(2)]
    h_gd = [torch.empty(B, D).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_dense, h_idx, h_off, h_go[0]))
    d2h = h_out[0].numel() * 4 + h_gd[0].numel() * 4
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        bufs = [dict(dense=torch.empty_like(dense), idx=torch.empty_like(idx), off=torch.empty_like(off),
                     go=torch.empty_like(grad_out), out=torch.empty_like(out), gd=torch.empty_like(gd))
                for _ in range(2)]
    torch.cuda.synchronize()

    def e2e_steps(n, start=None):
        if start is not None:
            up.wait_event(start)                     # the first upload is inside the timed region
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]

        def upload(k):
            bb = bufs[k % 2]
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(computed[k % 2])     # step k-2 has consumed this input buffer
                bb["dense"].copy_(h_dense, non_blocking=True)
                bb["idx"].copy_(h_idx, non_blocking=True)
                bb["off"].copy_(h_off, non_blocking=True)
                bb["go"].copy_(h_go[k % 2], non_blocking=True)
                uploaded[k % 2].record(up)

        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            bb = bufs[k % 2]
            stream.wait_event(uploaded[k % 2])
            if k >= 2:
                stream.wait_event(read_back[k % 2])    # step k-2's results have left this output buffer
            dl.dlrm_emb_interact_fwd_train(tables, row_base, F, D, B, bb["idx"], bb["off"], bb["dense"], pooled,
                                           bb["out"], P, status=status, stream=stream)
            dl.dlrm_interact_bwd(bb["go"], bb["dense"], pooled, F, D, B, P, bb["gd"], gp, stream=stream)
            dl.dlrm_emb_bwd_sgd(tables, row_base, w.total_rows, F, D, B, bb["idx"], bb["off"], gp, LR, ws,
                                status=status, stream=stream)
            computed[k % 2].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[k % 2])
                h_out[k % 2].copy_(bb["out"], non_blocking=True)
                h_gd[k % 2].copy_(bb["gd"], non_blocking=True)
                read_back[k % 2].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    e2e_steps(3)
    torch.cuda.synchronize()
    e_steps = max(3, args.steps // 4)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(e_steps, start=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = reduce_max(e0.elapsed_time(e1), world, dev)
    # the host copies hold what the last two steps left on the device (bit for bit)
    for k in range(2):
        if not (torch.equal(h_out[k].view(torch.int32), bufs[k]["out"].cpu().view(torch.int32)) and
                torch.equal(h_gd[k].view(torch.int32), bufs[k]["gd"].cpu().view(torch.int32))):
            raise RuntimeError("e2e: results read back differ from the device buffers")

    # ---- roofline of the dominant kernel (algorithmic bytes per launch / event time)
    peaks = measured_peaks()
    unique_rows = None
    keys = ws[: 4 * nnz].view(torch.int32)
    k = keys[keys != -1]
    if k.numel():
        unique_rows = int(torch.unique_consecutive(k).numel())
    s = 4  # fp32
    alg = {
        # offsets + index + row read per lookup, pooled row written once; dense read, output written
        "emb_interact_fwd": B * F * (4 + 4 + D * s) + B * F * D * s + B * (D * s + P * s),
        "interact_bwd": B * (P * 4 + D * s + F * D * s + D * 4 + F * D * 4),
        "emb_bwd_sgd": nnz * (4 + 4 + D * 4) + (unique_rows or 0) * 2 * D * 4,
    }
    dom = max(op_ms, key=op_ms.get)
    kernel_names = {"emb_interact_fwd": "emb_interact_regs_kernel", "interact_bwd": "interact_bwd_regs_kernel",
                    "emb_bwd_sgd": f"emb_bwd_sgd ({sgd_kernels(w.total_rows)} kernels)"}
    achieved = alg[dom] / (op_ms[dom] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": kernel_names[dom], "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "peak_source": peaks["source"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": ncu_traffic(dom if dom == "emb_bwd_sgd" else kernel_names[dom]),
            "algorithmic_bytes_per_launch": alg[dom], "launch_ms": round(op_ms[dom], 4)}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "samples/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Criteo Terabyte not available)",
        "config": {"workload": WORKLOAD, "global_batch": B * world, "per_gpu_batch": B, "tables": F,
                   "embedding_dim": D, "total_rows": w.total_rows, "nnz": nnz, "out_cols": P,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (4.1 GB tables, 0.87 GB pooled/grad tensors per step)"},
        "ops_ms": {k: round(v, 4) for k, v in op_ms.items()},
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
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelining": "next batch uploaded and previous results read back on two copy streams while a "
                              "step computes (double-buffered inputs/outputs)"},
        "gpu_launches": kernels_per_step(w.total_rows) * args.steps,
        "clocks": clk,
        "roofline": roof,
        "device_status": st,
        "finite_output_fraction": round(finite, 6),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_samples)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


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


def run_bottom_mlp(args, dl, inputs, torch, dev, stream, status) -> None:
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
    print(json.dumps({
        "config": "bottom-mlp", "workload": CONFIGS["bottom-mlp"], "batch": B, "steps": args.steps,
        "ms_per_step": round(ms, 4), "samples_per_s": round(B / (ms / 1e3), 1),
        "tflops": round(tflops, 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(tflops / peak["bf16_tflops"], 4),
                     "peak_note": f"dense bf16 burst ({peak['source']}); fp16 has the same nominal rate"},
        "with_fused_fwd": {"ms_per_step": round(ms2, 4), "samples_per_s": round(B / (ms2 / 1e3), 1),
                           "ops_ms": {k: round(v, 4) for k, v in per2.items()}},
        "device_status": int(status.item())}), flush=True)


LOSS_SCALE = 1024.0


def amp_step_ops(dl, w, torch, dev, stream, status, tab):
    """The mixed-precision training step's four calls, on device buffers."""
    F, D, B, P = w.F, w.D, w.B, w.out_cols
    rb, idx, off = (torch.from_numpy(a).to(dev) for a in (w.row_base, w.indices, w.offsets))
    dense = torch.from_numpy(w.dense.astype(np.float16)).to(dev)
    g16 = torch.from_numpy((w.grad_out.astype(np.float64) * LOSS_SCALE).astype(np.float16)).to(dev)
    pooled = torch.empty(B, F, D, dtype=torch.float16, device=dev)
    out = torch.empty(B, P, dtype=torch.float16, device=dev)
    gd = torch.empty(B, D, dtype=torch.float16, device=dev)
    gp = torch.empty(B, F, D, dtype=torch.float16, device=dev)
    ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, D, w.total_rows), dtype=torch.uint8, device=dev)
    lr = float(np.float32(w.lr / LOSS_SCALE))
    # the replayed batch's upstream gradient alternates its sign (keeps the tables bounded)
    gs, k = (g16, -g16), [0]

    def bwd():
        g = gs[k[0] % 2]
        k[0] += 1
        dl.dlrm_interact_bwd_f16(g, dense, pooled, F, D, B, P, gd, gp, status=status, stream=stream)

    return [
        ("emb_fwd", lambda: dl.dlrm_emb_fwd(tab, rb, F, D, B, idx, off, pooled, flags=dl.DLRM_FLAG_POOLED_F16,
                                            status=status, stream=stream)),
        ("interact_fwd", lambda: dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=status, stream=stream)),
        ("interact_bwd", bwd),
        ("emb_bwd_sgd", lambda: dl.dlrm_emb_bwd_sgd(tab, rb, w.total_rows, F, D, B, idx, off, gp, lr, ws,
                                                    flags=dl.DLRM_FLAG_GRAD_F16, status=status, stream=stream)),
    ]


def run_train_amp(args, dl, inputs, torch, dev, stream, status) -> None:
    B = args.batch
    w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, train=True)
    with torch.cuda.stream(stream):
        tab = torch.empty(w.total_rows, w.D, dtype=torch.float32, device=dev)
        dl.dlrm_synth_fill_uniform(tab, w.table_seed, 0, stream=stream)
    torch.cuda.synchronize()
    ops = amp_step_ops(dl, w, torch, dev, stream, status, tab)
    per, ms = _time_ops(torch, stream, ops, args.steps, args.warmup)
    F, D, P, nnz = w.F, w.D, w.out_cols, w.nnz
    alg = {"emb_fwd": nnz * (4 + 4 + D * 4) + B * F * D * 2,
           "interact_fwd": B * (D * 2 + F * D * 2 + P * 2),
           "interact_bwd": B * (P * 2 + D * 2 + F * D * 2 + D * 2 + F * D * 2),
           "emb_bwd_sgd": nnz * (4 + 4 + D * 2)}
    print(json.dumps({
        "config": "train-64k-amp", "workload": CONFIGS["train-64k-amp"], "batch": B, "nnz": nnz,
        "steps": args.steps, "ms_per_step": round(ms, 4), "step_samples_per_s": round(B / (ms / 1e3), 1),
        "ops_ms": {k: round(v, 4) for k, v in per.items()},
        "alg_GBps": {k: round(alg[k] / (v / 1e3) / 1e9, 1) for k, v in per.items()},
        "device_status": int(status.item())}), flush=True)


def run_config(args, name) -> None:
    """Measure one workload of the pages' configurations and print a JSON line."""
    import torch

    import dlrm_embeddings_dot_gb300 as dl
    from dlrm_embeddings_dot_gb300 import inputs

    dl.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if name == "bottom-mlp":
        run_bottom_mlp(args, dl, inputs, torch, dev, stream, status)
        return
    if name == "train-64k-amp":
        run_train_amp(args, dl, inputs, torch, dev, stream, status)
        return

    def setup(w, tt):
        with torch.cuda.stream(stream):
            tab = torch.empty(w.total_rows, w.D, dtype=tt, device=dev)
            dl.dlrm_synth_fill_uniform(tab, w.table_seed, 0, stream=stream)
            rb = torch.from_numpy(w.row_base).to(dev)
            idx = torch.from_numpy(w.indices).to(dev)
            off = torch.from_numpy(w.offsets).to(dev)
        torch.cuda.synchronize()
        return tab, rb, idx, off

    batches = [args.batch]
    if name == "large-tables":
        batches = [1024, 4096, 16384, 65536, 262144, 1048576]
    for B in batches:
        if name in ("tiny", "tiny-train"):
            w = inputs.tiny_slice(seed=0, train=(name == "tiny-train"))
        elif name in ("default-fwd", "default-fwd-uniform"):
            w = inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD,
                                    uniform_indices=name.endswith("-uniform"))
        elif name == "train-64k":
            w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=ALPHA_TRAIN, train=True)
        elif name in ("multi-hot", "multi-hot-uniform"):
            w = inputs.multi_hot(B=B if B != BATCH else 16384, uniform_indices=name.endswith("-uniform"))
        else:
            w = inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=ALPHA_FWD, rows=inputs.large_tables_rows())
        tt = torch.float16 if w.dtype == inputs.F16 else torch.float32
        es = 2 if tt == torch.float16 else 4
        F, D, Bw, P = w.F, w.D, w.B, w.out_cols
        tab, rb, idx, off = setup(w, tt)
        pooled = torch.empty(Bw, F, D, dtype=tt, device=dev)
        dense = torch.from_numpy(w.dense.astype(np.float16 if tt == torch.float16 else np.float32)).to(dev)
        out = torch.empty(Bw, P, dtype=tt, device=dev)
        ops = [("emb_fwd", lambda: dl.dlrm_emb_fwd(tab, rb, F, D, Bw, idx, off, pooled, status=status,
                                                   stream=stream))]
        multi = name.startswith("multi-hot")
        if not multi:
            ops.append(("interact_fwd", lambda: dl.dlrm_interact_fwd(dense, pooled, F, D, Bw, out, P,
                                                                     status=status, stream=stream)))
        train = name in ("tiny-train", "train-64k") or multi
        if train:
            gp = torch.empty(Bw, F, D, device=dev)
            ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, D, w.total_rows), dtype=torch.uint8,
                             device=dev)
            if multi:
                gp.normal_(0.0, 1e-2)
            else:
                go = torch.from_numpy(w.grad_out).to(dev)
                gd = torch.empty(Bw, D, device=dev)
                ops.append(("interact_bwd", lambda: dl.dlrm_interact_bwd(go, dense, pooled, F, D, Bw, P, gd, gp,
                                                                         stream=stream)))
            ops.append(("emb_bwd_sgd", lambda: dl.dlrm_emb_bwd_sgd(tab, rb, w.total_rows, F, D, Bw, idx, off, gp,
                                                                   w.lr, ws, status=status, stream=stream)))
        per, ms = _time_ops(torch, stream, ops, args.steps, args.warmup)
        fused_train = None
        if train and not multi and tt == torch.float32 and F in (8, 26) and D == 128:
            fops = [("emb_interact_fwd_train",
                     lambda: dl.dlrm_emb_interact_fwd_train(tab, rb, F, D, Bw, idx, off, dense, pooled, out, P,
                                                            status=status, stream=stream))] + ops[2:]
            fper, fms = _time_ops(torch, stream, fops, args.steps, args.warmup)
            fused_train = {"ms_per_step": round(fms, 4), "step_samples_per_s": round(Bw / (fms / 1e3), 1),
                           "ops_ms": {k: round(v, 4) for k, v in fper.items()}}
        if multi and tt == torch.float32 and F in (8, 26) and D == 128:
            # the forward of a multi-hot batch: lookup + interaction as two calls, and the training
            # forward call (which itself runs two launches for bags this large); 480 columns rather
            # than 479, as the one-pass kernel writes whole float4 columns
            P4 = (P + 3) // 4 * 4
            out4 = torch.empty(Bw, P4, dtype=tt, device=dev)
            two = [ops[0], ("interact_fwd", lambda: dl.dlrm_interact_fwd(dense, pooled, F, D, Bw, out4, P4,
                                                                         status=status, stream=stream))]
            one = [("emb_interact_fwd_train",
                    lambda: dl.dlrm_emb_interact_fwd_train(tab, rb, F, D, Bw, idx, off, dense, pooled, out4, P4,
                                                           status=status, stream=stream))]
            _, two_ms = _time_ops(torch, stream, two, args.steps, args.warmup)
            _, one_ms = _time_ops(torch, stream, one, args.steps, args.warmup)
            fused_train = {"fwd_two_calls_ms": round(two_ms, 4), "fwd_train_call_ms": round(one_ms, 4)}
        fused_ms = None
        if tt == torch.float16 and not train:
            fop = [("emb_interact_fwd", lambda: dl.dlrm_emb_interact_fwd(tab, rb, F, D, Bw, idx, off, dense, out, P,
                                                                         status=status, stream=stream))]
            _, fused_ms = _time_ops(torch, stream, fop, args.steps, args.warmup)
        nnz = w.nnz
        alg = {"emb_fwd": nnz * (4 + D * es) + Bw * F * (4 + D * es),
               "interact_fwd": Bw * (D * es + F * D * es + P * es),
               "interact_bwd": Bw * (P * 4 + D * es + F * D * es + D * 4 + F * D * 4),
               "emb_bwd_sgd": nnz * (4 + 4 + D * 4)}
        fwd_ms = per["emb_fwd"] + per.get("interact_fwd", 0.0)
        line = {"config": name, "workload": CONFIGS[name], "batch": Bw, "nnz": nnz, "steps": args.steps,
                "ms_per_step": round(ms, 4), "ops_ms": {k: round(v, 4) for k, v in per.items()},
                "alg_GBps": {k: round(alg[k] / (v / 1e3) / 1e9, 1) for k, v in per.items()},
                "fwd_samples_per_s": round(Bw / (fwd_ms / 1e3), 1),
                "step_samples_per_s": round(Bw / (ms / 1e3), 1), "device_status": int(status.item())}
        if fused_train is not None:
            line["one_pass_forward"] = fused_train
        if fused_ms is not None:
            line["fused_fwd"] = {"ms": round(fused_ms, 4), "samples_per_s": round(Bw / (fused_ms / 1e3), 1),
                                 "alg_GBps": round(Bw * (F * (8 + D * 2) + D * 2 + P * 2) / (fused_ms / 1e3) / 1e9,
                                                   1)}
        print(json.dumps(line), flush=True)
        del tab, pooled, out, dense
        torch.cuda.empty_cache()


def run_reference(args) -> None:
    """The CPU oracle, timed as it stands, on bounded samples of the same workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from dlrm_embeddings_dot_gb300 import inputs
    w = inputs.dlrm_default(B=BATCH, dtype=inputs.F32, alpha=ALPHA_TRAIN, seed=0, train=True)
    n = args.ref_samples
    for i in range(args.warmup):
        cpu_oracle_step(w, np.arange(n) + (i * n) % (w.B - n))
    total = 0.0
    for i in range(args.steps):
        total += cpu_oracle_step(w, np.arange(n) + ((i + args.warmup) * n) % (w.B - n))
    value = n * args.steps / total
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "samples/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps * (BATCH / n), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": BATCH, "per_gpu_batch": BATCH},
        "cpu_baseline": {"value": round(value, 1), "unit": "samples/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} samples of the 65,536-sample batch per step"},
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
    ap.add_argument("--ref-samples", type=int, default=512,
                    help="samples per step of the --impl reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
