"""Benchmark: the Q4_K x M-row decode step on synthetic 27B-shaped weights.

One step = every matrix of the stack (64 layers x {qkv, o, gate_up, down} + lm_head,
12.71 GB of Q4_K super-blocks) multiplied against its own M fp16 activation rows, replayed
as one CUDA graph of libqmm runs.  Headline: M = 12 (4 streams x (1 token + 2 drafts)).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is weight GB/s of the whole job (weights streamed
per step x steps / time, summed over ranks); `tok_s` is rows per second.  `--impl reference`
times the CPU oracle (the reference arm of this build) on a bounded sample of the same
workload on the host cores.  Under torchrun every rank runs its own replica of the step
(the method runs on one GPU; ranks do not exchange data).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q4K x M-row decode GEMM: weight GB/s (% of HBM peak) and step tok/s at M=1/12/64"
HEADLINE_M = 12
EXTRA_M = (1, 64)
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=synth.LAYERS, help="(testing) fewer layers")
    ap.add_argument("--no-extra", action="store_true", help="skip the M=1 and M=64 lines")
    ap.add_argument("--no-parity", action="store_true", help="skip the sampled oracle check")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--single", default=None,
                    help="profiling mode: run one matrix of the stack (proj4096, qkv, o, gate_up, "
                         "down, lm_head) --steps times at --m rows and print its timing")
    ap.add_argument("--m", type=int, default=HEADLINE_M)
    ap.add_argument("--backend", type=int, default=0, help="0 auto, 1 mma.sync, 2 tcgen05")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------- workload
class Stack:
    """All matrices of the step resident on the GPU, with activations and outputs."""

    def __init__(self, layers: int, m_max: int, torch, seed: int = 0):
        from bit_weight_streaming_q4_gb300 import Qmm
        self.torch = torch
        self.mats = synth.stack(layers)
        self.m_max = m_max
        self.qs = []
        for mat in self.mats:
            blocks = synth.q4k_matrix(mat.n, mat.k, seed=seed, tensor_id=mat.tensor_id)
            dev = torch.from_numpy(blocks.reshape(-1)).cuda()
            self.qs.append(Qmm(dev, mat.n, mat.k, m_max=m_max))
            del dev
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self.weight_bytes = sum(m.weight_bytes for m in self.mats)
        # activations for every matrix (own stream per matrix), rows 0..m_max-1
        self.x_off, off = [], 0
        for mat in self.mats:
            self.x_off.append(off)
            off += m_max * mat.k
        xh = np.empty(off, dtype=np.float16)
        for mat, o in zip(self.mats, self.x_off):
            xh[o:o + m_max * mat.k] = synth.x_f16(m_max, mat.k, seed=seed,
                                                    tensor_id=synth.X_ID_OFFSET + mat.tensor_id).ravel()
        self.x_host = xh
        self.x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.float16)
        self.y_off, off = [], 0
        for mat in self.mats:
            self.y_off.append(off)
            off += m_max * mat.n
        self.y = torch.zeros(off, dtype=torch.float32, device="cuda")

    def x_ptrs(self):
        # rows 0..m-1 of matrix i start at x_off[i] (row stride K); m_max rows reserved
        return [self.x[o:].data_ptr() for o in self.x_off]

    def y_ptrs(self):
        return [self.y[o:].data_ptr() for o in self.y_off]

    def bytes_for(self, m):
        xb = sum(m * mat.k * 2 for mat in self.mats)
        yb = sum(m * mat.n * 4 for mat in self.mats)
        return self.weight_bytes, xb, yb


def time_graph(torch, step, steps, warmup, stream):
    for _ in range(warmup):
        step.launch(stream.cuda_stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step.launch(stream.cuda_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def sampled_parity(stack, m, rng_seed=0, rows_per_matrix=2, matrices=None):
    """Recompute a few output rows per matrix with the oracle, from regenerated blocks."""
    import oracle
    torch = stack.torch
    y = stack.y.cpu().numpy()
    rng = np.random.default_rng(rng_seed)
    worst, checked = 0.0, 0
    idx = range(len(stack.mats)) if matrices is None else matrices
    for i in idx:
        mat = stack.mats[i]
        rows = np.sort(rng.choice(mat.n, size=min(rows_per_matrix, mat.n), replace=False))
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=rows)
        x = stack.x_host[stack.x_off[i]:stack.x_off[i] + m * mat.k].reshape(m, mat.k)
        y_ref, s_ref = oracle.qmm(blocks, x)
        got = y[stack.y_off[i]:stack.y_off[i] + m * mat.n].reshape(m, mat.n)[:, rows]
        ratio = np.abs(got - y_ref) / (2e-3 * s_ref + 1e-6)
        worst = max(worst, float(ratio.max()))
        checked += ratio.size
    del torch
    return {"checked_outputs": checked, "max_err_over_bound": worst, "pass": worst <= 1.0}


# ------------------------------------------------------------------------------- oracle arm
def cpu_oracle_sample(target_s: float, layers: int = synth.LAYERS, m: int = HEADLINE_M):
    """Time the oracle on a bounded sample of the step: a contiguous block of rows of each of
    the five matrix shapes (layer 0 and lm_head), sized so the run takes ~target_s seconds.
    Returns weight GB/s of the oracle and a description."""
    import oracle
    oracle.build()
    shapes = synth.layer_matrices(0) + [synth.LM_HEAD]
    # calibrate on a small block
    mat = shapes[0]
    rows = 64
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=np.arange(rows))
    x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    t0 = time.perf_counter()
    oracle.qmm(blocks, x)
    per_weight = (time.perf_counter() - t0) / (rows * mat.k)
    weights_target = target_s / max(per_weight, 1e-12)
    per_shape = weights_target / len(shapes)
    total_w, total_t = 0, 0.0
    parts = []
    for mat in shapes:
        r = int(max(16, min(mat.n, per_shape // mat.k)))
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=np.arange(r))
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
        t0 = time.perf_counter()
        oracle.qmm(blocks, x)
        total_t += time.perf_counter() - t0
        total_w += r * mat.k
        parts.append(f"{mat.name}[:{r}]")
    gbs = total_w * 144 / 256 / total_t / 1e9
    return {"gbs": gbs, "seconds": total_t, "cores": oracle.max_threads(),
            "sample": f"M={m}, rows {', '.join(parts)} ({total_w * 144 // 256 / 1e6:.1f} MB of "
                      f"weights, {total_t:.1f} s); scaled to the full step by weight bytes"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    full_bytes = sum(m.weight_bytes for m in synth.stack(args.layers))
    per_step_s = max(1.0, args.cpu_seconds / max(args.steps, 1))
    for _ in range(min(args.warmup, 1)):
        cpu_oracle_sample(0.5)
    samples = [cpu_oracle_sample(per_step_s) for _ in range(max(1, min(args.steps, 5)))]
    gbs = statistics.median(s["gbs"] for s in samples)
    step_s = full_bytes / (gbs * 1e9)
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": len(samples), "warmup": min(args.warmup, 1), "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"decode step M={HEADLINE_M}: {args.layers} x {{qkv, o, gate_up, down}} "
                               f"+ lm_head, Q4_K", "m": HEADLINE_M, "weight_bytes": full_bytes},
        "tok_s": HEADLINE_M / step_s,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": samples[0]["cores"],
                         "kind": "oracle", "sample": samples[0]["sample"]},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from bit_weight_streaming_q4_gb300 import Step

    torch.cuda.set_device(local_rank)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    m_max = max((HEADLINE_M,) + (() if args.no_extra else EXTRA_M))
    stack = Stack(args.layers, m_max, torch)
    stream = torch.cuda.Stream()
    n_mats = len(stack.mats)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def measure(m, steps, warmup):
        with torch.cuda.stream(stream):
            step = Step(stack.qs, stack.x_ptrs(), stack.y_ptrs(), m, stream=stream.cuda_stream)
        barrier()
        t = time_graph(torch, step, steps, warmup, stream)
        step.close()
        if world > 1:
            tt = torch.tensor([t], device="cuda")
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            t = float(tt.item())
        return t

    # headline: M = 12, timed with the clocks sampled
    barrier()
    with torch.cuda.stream(stream):
        step = Step(stack.qs, stack.x_ptrs(), stack.y_ptrs(), HEADLINE_M,
                    stream=stream.cuda_stream)
    for _ in range(args.warmup):
        step.launch(stream.cuda_stream)
    barrier()
    with ClockSampler(local_rank) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step.launch(stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    if world > 1:
        tt = torch.tensor([t], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    step.close()
    clocks = clk.summary()
    wb, xb, yb = stack.bytes_for(HEADLINE_M)
    step_s = t / args.steps
    value = wb * args.steps * world / t / 1e9
    alg_bytes = wb + xb + yb
    achieved = alg_bytes / step_s / 1e9
    parity = None
    if not args.no_parity:
        parity = sampled_parity(stack, HEADLINE_M)

    # end to end through the public API with host buffers: each step copies every matrix's
    # M activation rows from pinned host memory (one dense slab), replays the recorded step,
    # and copies every output back (one dense slab)
    xo, yo, offx, offy = [], [], 0, 0
    for mat in stack.mats:
        xo.append(offx)
        yo.append(offy)
        offx += HEADLINE_M * mat.k
        offy += HEADLINE_M * mat.n
    x_dense = np.concatenate([stack.x_host[o:o + HEADLINE_M * mat.k]
                              for mat, o in zip(stack.mats, stack.x_off)])
    x_pin = torch.from_numpy(x_dense.view(np.int16)).view(torch.float16).pin_memory()
    y_pin = torch.empty(offy, dtype=torch.float32).pin_memory()
    xd = torch.empty(offx, dtype=torch.float16, device="cuda")
    yd = torch.empty(offy, dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        e2e_step = Step(stack.qs, [xd[o:].data_ptr() for o in xo], [yd[o:].data_ptr() for o in yo],
                        HEADLINE_M, stream=stream.cuda_stream)

    def e2e_once():
        with torch.cuda.stream(stream):
            xd.copy_(x_pin, non_blocking=True)
            e2e_step.launch(stream.cuda_stream)
            y_pin.copy_(yd, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_once()
    barrier()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(e2e_steps):
        e2e_once()
    a1.record(stream)
    torch.cuda.synchronize()
    te = a0.elapsed_time(a1) / 1e3
    if world > 1:
        tt = torch.tensor([te], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        te = float(tt.item())
    e2e_step.close()
    ydev = stack.y.cpu().numpy()
    yh = y_pin.numpy()
    e2e_ok = all(np.array_equal(yh[a:a + HEADLINE_M * mat.n].view(np.uint32),
                                ydev[b:b + HEADLINE_M * mat.n].view(np.uint32))
                 for mat, a, b in zip(stack.mats, yo, stack.y_off))

    by_m = {str(HEADLINE_M): {"weight_gbs": value / world, "tok_s": HEADLINE_M / step_s,
                              "ms_per_step": step_s * 1e3}}
    if not args.no_extra:
        for m in EXTRA_M:
            steps_m = max(20, args.steps // (4 if m > 16 else 1))
            tm = measure(m, steps_m, 3)
            sm = tm / steps_m
            wbm, xbm, ybm = stack.bytes_for(m)
            by_m[str(m)] = {"weight_gbs": wbm / sm / 1e9, "tok_s": m / sm, "ms_per_step": sm * 1e3,
                            "frac_of_hbm_measured": wbm / sm / 1e9 / hbm}

    cpu = None
    if rank == 0:
        c = cpu_oracle_sample(args.cpu_seconds)
        cpu = {"value": c["gbs"], "unit": "GB/s", "cores": c["cores"], "kind": "oracle",
               "sample": c["sample"]}

    info = stack.qs[0].info()
    launches_per_step = sum(-(-HEADLINE_M // q.info().m_per_launch) for q in stack.qs)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"decode step M={HEADLINE_M} (4 streams x (1 token + 2 drafts)): "
                               f"{args.layers} x {{qkv 5120->8192, o 6144->5120, gate_up 5120->34816, "
                               f"down 17408->5120}} + lm_head 5120->151936, Q4_K 144 B/256 weights",
                   "m": HEADLINE_M, "matrices": n_mats, "weight_bytes": wb,
                   "l2": "inputs larger than L2 (12.7 GB of weights streamed per step; no flush)",
                   "backend": int(info.backend), "ctas": int(info.grid),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tok_s": HEADLINE_M * world / step_s,
        "frac_of_hbm": {"measured": value / world / hbm, "nominal_8TBs": value / world / NOMINAL_HBM_GBS},
        "by_m": by_m,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": None,
                     "note": f"algorithmic bytes per step (weights + x + y) / step time; peak is "
                             f"{peak_kind} copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": {"value": wb * e2e_steps / te / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": xb, "d2h_bytes_per_step": yb,
                "ms_per_step": te / e2e_steps * 1e3, "outputs_match_device_run": e2e_ok,
                "steps": e2e_steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "parity": parity,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_single(args):
    """One matrix, --steps launches after --warmup, on rotating copies (inputs > L2)."""
    import torch
    from bit_weight_streaming_q4_gb300 import Qmm
    torch.cuda.set_device(0)
    shapes = {"proj4096": synth.SINGLE_PROJECTION, "lm_head": synth.LM_HEAD}
    shapes.update({m.name.split(".")[1]: m for m in synth.layer_matrices(0)})
    mat = shapes[args.single]
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    dev = torch.from_numpy(blocks.reshape(-1)).cuda()
    copies = max(1, -(-400_000_000 // mat.weight_bytes))
    qs = [Qmm(dev, mat.n, mat.k, m_max=max(args.m, 1), backend=args.backend) for _ in range(copies)]
    del dev
    x = torch.from_numpy(synth.x_f16(args.m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
                         .view(np.int16)).cuda().view(torch.float16)
    y = torch.empty((args.m, mat.n), dtype=torch.float32, device="cuda")
    for i in range(args.warmup):
        qs[i % copies].run(x, y, args.m)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        qs[i % copies].run(x, y, args.m)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / max(args.steps, 1)
    print(json.dumps({"single": mat.name, "m": args.m, "backend": int(qs[0].info().backend),
                      "us_per_launch": us, "weight_gbs": mat.weight_bytes / us / 1e3,
                      "copies": copies}), flush=True)


def main():
    args = parse()
    if args.single:
        run_single(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
