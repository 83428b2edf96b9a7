#!/usr/bin/env python3
"""Benchmark of the fused linear cross-entropy (FLCE) forward+backward on GB300.

One step = one flce_forward_backward call over the whole batch of a synthetic
LM-head workload (default: the DeepSeek-V3-shaped head, N=32768 rows, H=7168,
V=129280, Zipf(1.1) labels with 3% ignored, fp32 grad_W accumulator): forward
GEMM with the fused statistics epilogue, merge, dlogits, grad_h GEMM and grad_W
GEMM for every row chunk. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dsv3] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the
single-GPU path has no exchange step); rank 0 prints the whole-job line.
`--impl reference` times the CPU fp64 oracle on bounded row samples of the
same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "FLCE fwd+bwd tokens/s and TFLOP/s (6·N·H·V) as % of GB300 bf16 tensor peak"
# Nominal dense tf32 / bf16 tensor rate of GB300 (1.1 / 2.25 PFLOP/s): the tf32
# path's peak is the measured bf16 peak scaled by it.
TF32_OVER_BF16 = 1.1 / 2.25
NOMINAL_TF32_TFLOPS = 1100.0  # GB300 dense tf32, nominal
CPU_SAMPLE_SECONDS = 15.0      # oracle work in the cpu_baseline sample
REFERENCE_STEP_ROWS = 256      # rows per step of the reference (oracle) arm
UNIT = "tokens/s"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_burst": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def _config(w: workloads.Workload, chunk_rows: int, chunk_used: int = 0):
    return {"workload": f"{w.name}: N={w.n_rows} H={w.hidden} V={w.vocab} "
                        f"{'zipf(%g)' % w.zipf_s if w.labels == 'zipf' else 'uniform'} labels, "
                        f"{int(round(w.ignore_frac * 100))}% ignored, T={w.softcap}, m={w.out_mult}, "
                        f"mode={w.mode}",
            "n_rows": w.n_rows, "hidden": w.hidden, "vocab": w.vocab, "softcap": w.softcap,
            "out_mult": w.out_mult, "mode": w.mode, "chunk_rows": chunk_rows,
            "outputs": {"fwd_bwd": "loss, token_accuracy, grad_h, grad_W",
                        "fwd_grad_h": "loss, token_accuracy, grad_h",
                        "ce_only": "loss, token_accuracy"}[w.mode]
                       + (", predicted_tokens" if w.return_predicted and w.mode != "ce_only" else ""),
            **({"chunk_rows_used": chunk_used} if chunk_used else {}),
            "l2": "inputs larger than L2 (no flush needed)"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    try:
                        rows.append((float(parts[1]), float(parts[2]), float(parts[3]) if parts[3] not in
                                     ("[N/A]", "N/A") else 0.0, parts[5:9]))
                    except ValueError:
                        pass
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r[2] for r in rows)}


# Throttle reasons that void a timed region's number (sw_power_cap is kept and noted).
REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks: dict):
    """Why a timed region's clock record voids its number, or None: a thermal or
    hardware slowdown, or an SM clock far below its maximum with no reason
    given (a clock lock left by someone else)."""
    reasons = set(clocks.get("reasons") or [])
    bad = sorted(reasons & set(REJECTING_REASONS))
    if bad:
        return "throttled: " + ", ".join(bad)
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm and mx and sm < 0.75 * mx and not reasons:
        return f"SM clock {sm:.0f} of {mx:.0f} MHz under load with no reason given"
    return None


def timed_steps(flce, step, steps: int, local: int, dist):
    """`steps` calls of step() between barriers and synchronisations on both
    sides, with CUDA events between the steps on the current stream, the
    library's per-launch events, and clock samples. Returns (ms per step,
    per-step ms, {kernel: (launches, ms)}, launches, clocks)."""
    stream = torch.cuda.current_stream(torch.device("cuda", local))
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    launches0 = flce.flce_launch_count()
    flce.flce_profile_begin(True)
    with ClockSampler(local) as clk:
        _barrier(dist)
        torch.cuda.synchronize()
        marks[0].record(stream)
        for k in range(steps):
            step()
            marks[k + 1].record(stream)
        torch.cuda.synchronize()
        _barrier(dist)
    kernels = flce.flce_profile_read()
    flce.flce_profile_begin(False)
    launches = flce.flce_launch_count() - launches0
    ms = marks[0].elapsed_time(marks[-1]) / steps
    per_step = [marks[k].elapsed_time(marks[k + 1]) for k in range(steps)]
    return ms, per_step, kernels, launches, clk.summary()


def timed_steps_checked(flce, step, steps: int, local: int, dist):
    """timed_steps, taken once more when the clock record of the first run voids
    it (on any rank); returns its result and a note on the voided run, or None."""
    r = timed_steps(flce, step, steps, local, dist)
    why = clocks_rejected(r[4])
    if _max_over_ranks(dist, 1.0 if why else 0.0) > 0:
        note = {"ms_per_step": r[0], "clocks": r[4], "why": why or "clocks of another rank"}
        return timed_steps(flce, step, steps, local, dist), note
    return r, None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return ws, rank, local, dist
    return 1, 0, 0, None


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def weight_f64(W_cpu: torch.Tensor) -> np.ndarray:
    return W_cpu.float().numpy().astype(np.float64)


def cpu_oracle_rate(w: workloads.Workload, W64: np.ndarray, h_rows: torch.Tensor, lab_rows: torch.Tensor,
                    steps: int = 1, warmup: bool = False):
    """The CPU fp64 oracle, as it stands, on bounded row samples of the workload:
    full forward+backward (logits over all V, grad_h rows, grad_W) for the sampled rows."""
    from oracle import flce_oracle
    times = []
    R = h_rows.shape[0]
    need_w = w.mode == "fwd_bwd"
    need_h = w.mode != "ce_only"
    if warmup:  # one untimed call: BLAS thread start-up, first touch of the big buffers
        flce_oracle(h_rows, W64, lab_rows, softcap=w.softcap, out_mult=w.out_mult,
                    need_grad_h=need_h, need_grad_W=need_w)
    for _ in range(steps):
        t0 = time.perf_counter()
        flce_oracle(h_rows, W64, lab_rows, softcap=w.softcap, out_mult=w.out_mult,
                    need_grad_h=need_h, need_grad_W=need_w)
        times.append(time.perf_counter() - t0)
    return R, times


def cpu_baseline_fwd_bwd(args, w, W_cpu, h_cpu, lab_cpu) -> dict:
    """The oracle, as it stands, on a bounded sample of the workload's rows: an
    untimed call on a few rows (thread start-up, first touch), then samples of
    16 and 64 rows, then one grown to about CPU_SAMPLE_SECONDS. The oracle's
    time has a fixed part (the [V, H] weight gradient) and a part per row; the
    last two samples give both, and the full-step time is extrapolated from
    them."""
    W64 = weight_f64(W_cpu)
    N = w.n_rows
    r0 = min(4, N)
    cpu_oracle_rate(w, W64, h_cpu[:r0], lab_cpu[:r0])
    sizes = [args.sample_rows] if args.sample_rows else [min(16, N), min(64, N)]
    runs = []
    for R in sizes:
        n, t = cpu_oracle_rate(w, W64, h_cpu[:R], lab_cpu[:R])
        runs.append((n, t[0]))
    if not args.sample_rows and len(runs) == 2 and runs[1][0] > runs[0][0]:
        per_row = max((runs[1][1] - runs[0][1]) / (runs[1][0] - runs[0][0]), 1e-9)
        if runs[1][1] < CPU_SAMPLE_SECONDS / 2 and runs[1][0] < N:
            R = int(min(N, runs[1][0] + (CPU_SAMPLE_SECONDS - runs[1][1]) / per_row))
            n, t = cpu_oracle_rate(w, W64, h_cpu[:R], lab_cpu[:R])
            runs.append((n, t[0]))
    n, sec = runs[-1]
    out = {"value": n / sec, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
           "sample": f"first {n} rows of the workload, full fp64 forward+backward over all {w.vocab} logits "
                     f"(numpy), after an untimed call on {r0} rows and timed samples of "
                     f"{', '.join(str(r[0]) for r in runs[:-1]) or 'none'} rows",
           "seconds": sec, "samples": [{"rows": r[0], "seconds": r[1]} for r in runs]}
    if len(runs) >= 2 and runs[-1][0] > runs[-2][0]:
        per_row = max((runs[-1][1] - runs[-2][1]) / (runs[-1][0] - runs[-2][0]), 0.0)
        fixed = max(runs[-1][1] - per_row * runs[-1][0], 0.0)
        out["extrapolated_full_step_s"] = fixed + per_row * N
        out["extrapolation"] = ("fixed seconds + seconds per row x the workload's rows, fitted to the last two "
                                "samples; extrapolated, not measured")
    return out


def run_reference(args, w):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return
    R = args.sample_rows or REFERENCE_STEP_ROWS
    h, W, lab = workloads.make_inputs(w, n_rows=R * (args.steps + args.warmup))
    W64 = weight_f64(W)
    times = []
    for s in range(args.warmup + args.steps):
        hs, ls = h[s * R:(s + 1) * R], lab[s * R:(s + 1) * R]
        _, t = cpu_oracle_rate(w, W64, hs, ls)
        if s >= args.warmup:
            times.append(t[0])
    total = sum(times)
    value = R * len(times) / total
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w, 0),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{R} rows of the {w.name} head per step (all {w.vocab} logits, "
                                       f"grad_h and grad_W), numpy fp64"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


KERNEL_SOURCES = ["gemm_tc.cu", "flce_device.cuh", "flce_epilogue.cuh", "flce_internal.h", "kernels_aux.cu",
                  "kernels_ce.cu"]


def code_only(src: str) -> str:
    """C++ / CUDA source without comments, trailing blanks and empty lines: what
    the compiler sees, so that editing a comment keeps a recorded figure valid."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """sha256 over the code of the kernel sources: a recorded DRAM traffic
    figure is only reported while the kernels are the ones it was measured on."""
    import hashlib
    hsh = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "linear_cross_entropy_02_gb300", "csrc", f)) as fh:
            hsh.update(code_only(fh.read()).encode())
    return hsh.hexdigest()


def _traffic_key(args, w):
    """The key of a bench line's recorded traffic: the workload and the variant
    of the path it runs. Lines with overridden sizes have none."""
    if args.rows or args.vocab or args.chunk_rows or args.vocab_slab or getattr(args, "vocab_shards", 0):
        return None
    if args.ce_logits:
        return w.name + "-ce_logits"
    return (w.name + ("-lowmem" if args.low_memory else "") + ("-fp32" if args.fp32 else "")
            + ("-tile128" if args.tile128 else "") + ("-pair" if getattr(args, "pair", False) else "")
            + ("-3pass" if getattr(args, "fp32_3pass", False) else ""))


def recorded_traffic(workload, kernel: str, chunk_rows: int = 8192):
    """Per-launch dram__bytes_read.sum + dram__bytes_write.sum from the committed
    ncu capture summary, or None when absent, taken on other kernel sources, or
    taken with another number of rows per chunk (launches of another size)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if workload is None or not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_sha256") != kernel_source_hash() or e.get("chunk_rows", 8192) != chunk_rows:
        return None
    return e["bytes_per_launch"]


GOLDEN_DIR = os.path.join(ROOT, "tests", "golden", "configs")
GOLDEN_FOR = {"llama": "llama", "muse": "muse", "dsv3": "dsv3", "frozen_ce": "frozen", "frozen_grad_h": "frozen"}
NEAR_TIE = 1e-3


def parity_against_goldens(flce, w, h, W, lab, inputs_cpu, kw, forward=None):
    """One flce_forward of the timed workload (outside the timed region)
    compared row by row with the stored full-size oracle forward of the same
    inputs (tests/golden/configs, written by the oracle alone): the loss, every
    row's lse, every predicted token, and the correct count. Rows whose oracle
    top-2 gap is below 1e-3 relative may predict the other token; they are
    counted here. `forward` (optional) runs the line's own path and returns
    loss, lse and predicted; by default flce_forward with the line's flags.
    None when the workload has no stored oracle forward."""
    g = GOLDEN_FOR.get(w.name)
    if g is None or not os.path.exists(os.path.join(GOLDEN_DIR, g + ".json")):
        return None
    with open(os.path.join(GOLDEN_DIR, g + ".json")) as f:
        meta = json.load(f)
    arr = np.load(os.path.join(GOLDEN_DIR, g + ".npz"))
    hashes = {k: workloads.tensor_sha256(t) for k, t in zip(("h", "W", "labels"), inputs_cpu)}
    if hashes != meta["sha256"]:
        return {"oracle": f"tests/golden/configs/{g}", "skipped": "inputs differ from the stored oracle's"}
    f = forward() if forward is not None else flce.flce_forward(h, W, lab, return_lse=True, **kw)
    torch.cuda.synchronize()
    pred = f["predicted"].reshape(-1).cpu().numpy()
    lse = f["lse"].reshape(-1).cpu().double().numpy()
    y = inputs_cpu[2].numpy()
    valid = y != -100
    pred_o = arr["predicted"].astype(np.int64)
    near = arr["near_tie"].astype(bool)
    mism = pred != pred_o
    correct = int(np.sum((pred == y) & valid))
    loss = float(f["loss"])
    return {"oracle": f"tests/golden/configs/{g} (fp64, all {len(y)} rows)",
            "loss": loss, "loss_oracle": meta["loss"], "loss_rel_err": abs(loss - meta["loss"]) / abs(meta["loss"]),
            "lse_max_abs_err": float(np.abs(lse - arr["lse"].astype(np.float64)).max()),
            "near_tie_rows": int(near.sum()), "near_tie_threshold": NEAR_TIE,
            "predicted_mismatches": int(mism.sum()), "predicted_mismatches_on_near_ties": int((mism & near).sum()),
            "predicted_mismatches_off_near_ties": int((mism & ~near).sum()),
            "correct": correct, "correct_oracle": meta["correct"], "n_valid": int(valid.sum())}


def run_ours(args, w):
    world, rank, local, dist = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import linear_cross_entropy_02_gb300 as flce

    if args.ce_logits:
        return run_ce_logits(args, w, world, rank, local, dist, flce)
    h_cpu, W_cpu, lab_cpu = workloads.make_inputs(w)
    inputs_bf16 = (h_cpu, W_cpu, lab_cpu)
    if args.fp32:  # the same bf16-valued inputs carried in fp32: the tf32 tensor-core path
        h_cpu, W_cpu = h_cpu.float(), W_cpu.float()
    h = h_cpu.to(dev)
    W = W_cpu.to(dev)
    lab = lab_cpu.to(dev)
    gW = torch.zeros(W.shape, dtype=torch.float32, device=dev) if w.mode == "fwd_bwd" else None
    kw = dict(softcap=w.softcap, out_mult=w.out_mult, chunk_rows=args.chunk_rows,
              flags=(flce.FLCE_FLAG_TILE128 if args.tile128 else 0) | (flce.FLCE_FLAG_CTA_PAIR if args.pair else 0)
              | (flce.FLCE_FLAG_F32_3PASS if args.fp32_3pass else 0))
    bkw = dict(low_memory=args.low_memory, vocab_slab=args.vocab_slab)

    def step():
        if w.mode == "ce_only":
            return flce.flce_ce_only(h, W, lab, **kw)
        return flce.flce_forward_backward(h, W, lab, grad_W=gW, need_grad_h=True,
                                          return_predicted=w.return_predicted, **kw, **bkw)

    vp_forward = None
    status_workspaces = []  # explicit workspaces whose status words are checked too
    if args.vocab_shards:
        # The vocabulary-parallel form, its S shards run one after another on
        # this GPU: every shard's forward, the gather (a stack in shard order),
        # every shard's backward into one fp32 grad_h and its rows of grad_W,
        # then grad_h rounded to bf16. The same work S GPUs would share.
        S = args.vocab_shards
        offsets = [round(k * w.vocab / S) for k in range(S + 1)]
        shards = [W[offsets[k]:offsets[k + 1]] for k in range(S)]
        gW_sh = [None if gW is None else gW[offsets[k]:offsets[k + 1]] for k in range(S)]
        gh32 = torch.empty((w.n_rows, w.hidden), dtype=torch.float32, device=dev)
        vkw = dict(softcap=w.softcap, out_mult=w.out_mult, chunk_rows=args.chunk_rows, flags=kw["flags"])
        # --vp-stored: each shard keeps its logits between its two calls, in a
        # workspace of its own (FLCE_FLAG_VP_STORED)
        vp_ws = [None] * S
        if args.vp_stored:
            vkw["flags"] |= flce.FLCE_FLAG_VP_STORED
            vp_ws = [flce.flce_vp_workspace(h, shards[k], keep_logits=True, chunk_rows=args.chunk_rows)
                     for k in range(S)]
            status_workspaces.extend(vp_ws)

        def step():
            parts = [flce.flce_vp_forward(h, shards[k], lab, offsets[k], w.vocab, workspace=vp_ws[k], **vkw)
                     for k in range(S)]
            allp = torch.stack(parts)
            gh32.zero_()
            out = None
            for k in range(S):
                out = flce.flce_vp_backward(h, shards[k], lab, allp, offsets, offsets[k], w.vocab,
                                            grad_h_partial=gh32 if w.mode != "ce_only" else None,
                                            grad_W=gW_sh[k], vocab_slab=args.vocab_slab,
                                            return_predicted=w.return_predicted, workspace=vp_ws[k], **vkw)
            if w.mode != "ce_only":
                flce.flce_scale_gradient(gh32, None, out_dtype=h.dtype)
            return out

        def vp_forward():
            parts = [flce.flce_vp_forward(h, shards[k], lab, offsets[k], w.vocab, workspace=vp_ws[k], **vkw)
                     for k in range(S)]
            return flce.flce_vp_backward(h, shards[0], lab, torch.stack(parts), offsets, 0, w.vocab,
                                         return_predicted=True, return_lse=True, workspace=vp_ws[0], **vkw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if flce.flce_get_status() != 0 or any(flce.flce_get_status(workspace=x) for x in status_workspaces):
        raise RuntimeError(f"device status {flce.flce_get_status()} after warm-up")

    (ms, per_step, kernels, launches, clocks), remeasured = timed_steps_checked(flce, step, args.steps, local, dist)
    if flce.flce_get_status() != 0 or any(flce.flce_get_status(workspace=x) for x in status_workspaces):
        raise RuntimeError(f"device status {flce.flce_get_status()} after timed steps")
    ms_max = _max_over_ranks(dist, ms)
    rows_total = _sum_over_ranks(dist, float(w.n_rows))
    value = rows_total / (ms_max / 1e3)

    # End to end through the C ABI with host buffers: h and the labels in
    # page-locked host memory, copied by the library chunk by chunk under its
    # own kernels; the loss and accuracy come back to host memory.
    h_pin = h_cpu.pin_memory()
    lab_pin = lab_cpu.pin_memory()
    res = [0.0, 0.0]

    def e2e_step():
        if w.mode == "ce_only":
            loss, acc = flce.flce_ce_only_from_host(h_pin, W, lab_pin, **kw)
        else:
            o = flce.flce_forward_backward_from_host(h_pin, W, lab_pin, grad_W=gW, need_grad_h=True,
                                                     return_predicted=w.return_predicted, **kw, **bkw)
            loss, acc = o["loss"], o["token_accuracy"]
        torch.cuda.current_stream(dev).synchronize()
        res[0], res[1] = float(loss), float(acc)

    e2e_value = None
    if not args.vocab_shards:
        e2e_step()
        _barrier(dist)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / args.steps
        e2e_max = _max_over_ranks(dist, e2e_s)
        e2e_value = rows_total / e2e_max

    peaks = _peaks()
    flops = w.flops
    tflops = flops / (ms / 1e3) / 1e12
    step_peak = peaks["bf16_sustained"] * (TF32_OVER_BF16 if args.fp32 else 1.0)
    line = None
    parity = None
    if rank == 0 and not (args.rows or args.vocab):
        parity = parity_against_goldens(flce, w, h, W, lab, inputs_bf16,
                                        dict(softcap=w.softcap, out_mult=w.out_mult, chunk_rows=args.chunk_rows,
                                             flags=kw["flags"]),
                                        forward=vp_forward if args.vocab_shards else None)
    if rank == 0:
        chunk_used = flce.flce_chunk_rows(
            w.n_rows, w.hidden, w.vocab,
            mode=flce.FLCE_MODE_CE_ONLY if w.mode == "ce_only" else flce.FLCE_MODE_FORWARD_BACKWARD,
            need_grad_W=w.mode == "fwd_bwd", chunk_rows=args.chunk_rows,
            flags=(flce.FLCE_FLAG_RECOMPUTE if args.low_memory else 0) | kw["flags"],
            dtype=torch.float32 if args.fp32 else torch.bfloat16)
        # roofline of the dominant kernel, from the per-launch events of the timed region
        gemm_flops = {"fwd_gemm_stats": 2.0 * w.n_rows * w.hidden * w.vocab,
                      "grad_h_gemm": 2.0 * w.n_rows * w.hidden * w.vocab,
                      "grad_W_gemm": 2.0 * w.n_rows * w.hidden * w.vocab,
                      "recompute_dz_gemm": 2.0 * w.n_rows * w.hidden * w.vocab}
        total_ms = sum(v[1] for v in kernels.values()) or 1.0
        dom = max(kernels.items(), key=lambda kv: kv[1][1])[0] if kernels else None
        roof = None
        if dom in gemm_flops:
            n_launch, tms = kernels[dom]
            per_launch_flops = gemm_flops[dom] * args.steps / n_launch
            achieved = per_launch_flops / (tms / n_launch / 1e3) / 1e12
            peak = peaks["bf16_sustained"] * (TF32_OVER_BF16 if args.fp32 else 1.0)
            roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": (f"bf16_tflops_sustained ({peaks['source']}) x 1.1/2.25 nominal tf32/bf16"
                                    if args.fp32 else f"bf16_tflops_sustained ({peaks['source']})"),
                    "traffic": recorded_traffic(_traffic_key(args, w), dom, chunk_used),
                    "traffic_unit": "bytes per launch (dram read + write, ncu)",
                    "algorithmic_flops_per_launch": per_launch_flops,
                    "avg_launch_ms": tms / n_launch}
            if args.fp32:
                # the tf32 figure above is derived (bf16 sustained x the nominal ratio);
                # NVIDIA's nominal dense tf32 rate for GB300 is 1.1 PFLOP/s
                roof["nominal_tf32_peak"] = NOMINAL_TF32_TFLOPS
                roof["frac_of_nominal"] = achieved / NOMINAL_TF32_TFLOPS
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline_fwd_bwd(args, w, W_cpu, h_cpu, lab_cpu)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "ms_per_step_median": statistics.median(per_step), "ms_per_step_min": min(per_step),
            "vs_baseline": None,
            "dtype": ("f32 (three-pass tf32 products, fp32 accuracy)" if args.fp32_3pass else
                      "f32 inputs, tf32 products" if args.fp32 else "bf16"), "data": "synthetic",
            "config": _config(w, args.chunk_rows, chunk_used),
            "tflops": tflops, "pct_of_peak": 100.0 * tflops / step_peak,
            "peak_tflops": step_peak, "peak_source": peaks["source"] + (" x tf32/bf16 nominal" if args.fp32 else ""),
            "flops_per_step": flops,
            "executed_tensor_flops_per_step": flops * (4.0 / 3.0 if (args.low_memory or (args.vocab_shards and
                                                                                       not args.vp_stored))
                                                       and w.mode == "fwd_bwd" else 1.0)
                                                    * (3.0 if args.fp32_3pass else 1.0),
            "backward": ("recompute (low memory)" if (args.low_memory or (args.vocab_shards and not args.vp_stored))
                         else "stored logits"),
            "gemm_cta_tile": ("128x256, two accumulators" if args.tile128
                              else "per GEMM: 256x256 unless too few tiles to fill the SMs evenly"
                              + ("; each on a CTA pair (cta_group::2), two accumulators per SM"
                                 if args.pair else "")),
            "roofline": roof, "cpu_baseline": cpu,
            **({"vocab_shards": {"shards": args.vocab_shards, "run": "in turn on one GPU",
                                 "logits": "kept between the shard calls" if args.vp_stored else "recomputed",
                                 "exchange_bytes_per_step": 16 * w.n_rows * args.vocab_shards}}
               if args.vocab_shards else {}),
            "e2e": None if e2e_value is None else {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": h.numel() * h.element_size() + lab.numel() * 8, "d2h_bytes_per_step": 8,
                    "path": "flce_*_from_host: host h and labels, copied by the library in chunks under its "
                            "kernels; the loss and token accuracy come back to host memory",
                    "resident_outputs": ("none (CE-only)" if w.mode == "ce_only" else
                                         "grad_h" + (", grad_W" if w.mode == "fwd_bwd" else "")
                                         + (", predicted" if w.return_predicted else "")
                                         + " stay in device memory (a training step consumes them there)")},
            "parity": parity,
            "gpu_launches": launches,
            "clocks": clocks,
            **({"remeasured": remeasured} if remeasured else {}),
            "kernels": {k: {"launches": v[0], "ms": v[1], "share": v[1] / total_ms} for k, v in kernels.items()},
            "workspace_bytes": flce.flce_workspace_size(
                w.n_rows, w.hidden, w.vocab, chunk_rows=args.chunk_rows,
                mode=flce.FLCE_MODE_CE_ONLY if w.mode == "ce_only" else flce.FLCE_MODE_FORWARD_BACKWARD,
                need_grad_W=w.mode == "fwd_bwd",
                flags=(flce.FLCE_FLAG_RECOMPUTE if args.low_memory else 0) | kw["flags"],
                dtype=torch.float32 if args.fp32 else torch.bfloat16),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def cpu_ce_logits_rate(args, w, x_cpu, lab_cpu):
    """The oracle of cross-entropy on materialised logits, as it stands, on a
    bounded row sample sized to about CPU_SAMPLE_SECONDS."""
    if args.no_cpu_baseline:
        return None
    from oracle import oracle_ce_logits
    kw = dict(softcap=w.softcap, out_mult=w.out_mult, need_grad=True)
    r0 = min(64, w.n_rows)
    t0 = time.perf_counter()
    oracle_ce_logits(x_cpu[:r0], lab_cpu[:r0], **kw)        # untimed: thread start-up, first touch
    per_row = (time.perf_counter() - t0) / r0
    R = args.sample_rows or int(max(16, min(w.n_rows, CPU_SAMPLE_SECONDS / max(per_row, 1e-9))))
    t1 = time.perf_counter()
    oracle_ce_logits(x_cpu[:R], lab_cpu[:R], **kw)
    sec = time.perf_counter() - t1
    return {"value": R / sec, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"first {R} rows of the {w.n_rows} x {w.vocab} bf16 logits, fp64 loss and gradient (numpy), "
                      f"after an untimed call on {r0} rows", "seconds": sec}


def run_ce_logits(args, w, world, rank, local, dist, flce):
    """Cross-entropy on materialised bf16 logits [N, V] (the workload's N and V)
    with dL/dlogits: two streaming kernels, bounded by HBM bandwidth."""
    dev = torch.device("cuda", local)
    g = torch.Generator(device="cpu").manual_seed(w.seed * 16 + 9)
    x_cpu = torch.empty((w.n_rows, w.vocab), dtype=torch.bfloat16)
    step_rows = max(1, (1 << 26) // w.vocab)
    for r0 in range(0, w.n_rows, step_rows):
        r1 = min(w.n_rows, r0 + step_rows)
        x_cpu[r0:r1] = (torch.randn((r1 - r0, w.vocab), generator=g) * 1.28).to(torch.bfloat16)
    lab_cpu = workloads.make_labels(w.n_rows, w.vocab, w.seed, w.ignore_frac, w.labels, w.zipf_s)
    x = x_cpu.to(dev)
    lab = lab_cpu.to(dev)
    kw = dict(softcap=w.softcap, out_mult=w.out_mult, chunk_rows=args.chunk_rows)

    def step():
        return flce.flce_cross_entropy(x, lab, need_grad=True, return_predicted=False, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if flce.flce_get_status() != 0:
        raise RuntimeError("device status after warm-up")
    (ms, per_step, kernels, launches, clocks), remeasured = timed_steps_checked(flce, step, args.steps, local, dist)
    ms_max = _max_over_ranks(dist, ms)
    rows_total = _sum_over_ranks(dist, float(w.n_rows))

    x_pin = x_cpu.pin_memory()
    lab_pin = lab_cpu.pin_memory()
    res_pin = torch.empty(2, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(x)
    lab_dev = torch.empty_like(lab)

    def e2e_step():
        x_dev.copy_(x_pin, non_blocking=True)
        lab_dev.copy_(lab_pin, non_blocking=True)
        o = flce.flce_cross_entropy(x_dev, lab_dev, need_grad=True, return_predicted=False, **kw)
        res_pin[0:1].copy_(o["loss"].view(1), non_blocking=True)
        res_pin[1:2].copy_(o["token_accuracy"].view(1), non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    e2e_step()
    _barrier(dist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_max = _max_over_ranks(dist, (time.perf_counter() - t0) / args.steps)
    if rank == 0:
        peaks = _peaks()
        nv = float(w.n_rows) * w.vocab
        # algorithmic bytes: the statistics pass reads the logits once; the
        # gradient pass reads them again and writes dL/dlogits
        algo = {"ce_stats": nv * 2, "ce_grad": nv * 4}
        total_ms = sum(v[1] for v in kernels.values()) or 1.0
        dom = max(kernels.items(), key=lambda kv: kv[1][1])[0]
        n_launch, tms = kernels[dom]
        per_launch = algo.get(dom, 0.0) * args.steps / n_launch
        achieved = per_launch / (tms / n_launch / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": rows_total / (ms_max / 1e3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "ms_per_step_median": statistics.median(per_step),
            "ms_per_step_min": min(per_step), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(_config(w, args.chunk_rows), mode="cross_entropy on materialised bf16 logits [N, V]",
                           l2="logits larger than L2 (no flush needed)"),
            "tflops": None,
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "peak_source": f"hbm_gbs ({peaks['source']})",
                         "traffic": recorded_traffic(_traffic_key(args, w), dom),
                         "algorithmic_bytes_per_launch": per_launch, "avg_launch_ms": tms / n_launch},
            "cpu_baseline": cpu_ce_logits_rate(args, w, x_cpu, lab_cpu) if world == 1 else None,
            "e2e": {"value": rows_total / e2e_max, "unit": UNIT, "h2d_bytes_per_step": x.numel() * 2 + lab.numel() * 8,
                    "d2h_bytes_per_step": 8},
            "gpu_launches": launches, "clocks": clocks,
            **({"remeasured": remeasured} if remeasured else {}),
            "kernels": {k: {"launches": v[0], "ms": v[1], "share": v[1] / total_ms} for k, v in kernels.items()},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--chunk-rows", type=int, default=0)
    ap.add_argument("--sample-rows", type=int, default=0,
                    help="rows per oracle sample (0: %d per reference-arm step; the cpu_baseline sizes its own "
                         "sample to about %d s)" % (REFERENCE_STEP_ROWS, CPU_SAMPLE_SECONDS))
    ap.add_argument("--rows", type=int, default=0, help="override N (profiling captures only)")
    ap.add_argument("--vocab", type=int, default=0, help="override V (profiling captures only)")
    ap.add_argument("--low-memory", action="store_true",
                    help="recompute backward: no stored logits, dlogits per vocab slab")
    ap.add_argument("--vocab-slab", type=int, default=0)
    ap.add_argument("--fp32", action="store_true", help="fp32 h and W: the tf32 tensor-core path")
    ap.add_argument("--fp32-3pass", action="store_true",
                    help="with --fp32: three-pass tf32 products for fp32 accuracy (FLCE_FLAG_F32_3PASS)")
    ap.add_argument("--tile128", action="store_true",
                    help="128-row GEMM tiles with two accumulators (FLCE_FLAG_TILE128), for comparison")
    ap.add_argument("--ce-logits", action="store_true",
                    help="time the cross-entropy on materialised bf16 logits [N, V] instead")
    ap.add_argument("--pair", action="store_true",
                    help="256 x 256 GEMM tiles on CTA pairs (FLCE_FLAG_CTA_PAIR)")
    ap.add_argument("--vp-stored", action="store_true",
                    help="with --vocab-shards: each shard keeps its logits between its two calls "
                         "(FLCE_FLAG_VP_STORED; 6NHV instead of 8NHV)")
    ap.add_argument("--vocab-shards", type=int, default=0,
                    help="time the vocabulary-parallel form with this many shards, run in turn on one GPU")
    ap.add_argument("--predicted", action="store_true",
                    help="also return the predicted tokens (the epilogue then computes the argmax)")
    ap.add_argument("--no-predicted", action="store_true",
                    help="return no predicted tokens (the epilogue keeps only what the accuracy needs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = workloads.WORKLOADS[args.workload]
    import dataclasses
    if args.rows or args.vocab:
        # a smaller case of the same head (used for profiler captures, never for the bench line)
        w = dataclasses.replace(w, name=f"{w.name}-small", n_rows=args.rows or w.n_rows,
                                vocab=args.vocab or w.vocab)
    if args.predicted and w.mode != "ce_only":
        w = dataclasses.replace(w, return_predicted=True)
    if args.no_predicted:
        w = dataclasses.replace(w, return_predicted=False)
    if args.fp32_3pass:
        args.fp32 = True
    if args.impl == "reference":
        run_reference(args, w)
    else:
        import __graft_entry__
        __graft_entry__.build()
        run_ours(args, w)


if __name__ == "__main__":
    main()
