"""Benchmark: the Q4_K x M-row decode step on synthetic 27B-shaped weights.

One step = every matrix of the stack (64 layers x {qkv, o, gate_up, down} + lm_head,
12.71 GB of Q4_K super-blocks) multiplied against its own M fp16 activation rows: one libqmm
step (a persistent kernel streaming all 257 matrices, the runs independent since each matrix
has its own synthetic activations).  Headline: M = 12 (4 streams x (1 token + 2 drafts)); the
same step as a chain of dependent runs is reported beside it.

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
# DRAM bytes per work unit of each backend's launch, measured by ncu
# (profiles/stream_kernel_step_m12.md: the persistent mma.sync step at M = 12;
# profiles/tc_kernel_lm_head_m64.md: a tcgen05 launch at M = 64); each is valid only for the
# kernel source it was taken from
TRAFFIC_PER_UNIT = {
    1: {"source": "bit_weight_streaming_q4_gb300/csrc/qmm_b1.cu",
        "sha256": "a44227027e9ff57bf6103abe0de8b75fe722a45bb0c243cfd7e945ad0f9933f5",
        "bytes": 37262.0},
    2: {"source": "bit_weight_streaming_q4_gb300/csrc/qmm_b2.cu",
        "sha256": "8293ef0cab229e6bb6adca8f48745f550dd78e9897daa68e8b1cb56de9e94397",
        "bytes": 18799.1},
}
KERNEL_NAME = {1: "qmm::b1::stream_kernel<2>", 2: "qmm::b2::tc_kernel<16>"}
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
                         "down, lm_head) --steps times at --m rows, or the decode attention "
                         "(attention) --steps times, and print its timing")
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

    def __init__(self, layers: int, m_max: int, torch, seed: int = 0, wide_m: int = 0,
                 narrow_m: int = 0):
        """Handles for runs of up to m_max rows (qs); with wide_m, a second set of handles for
        runs of up to wide_m rows (qs_wide), and with narrow_m a third for runs of up to
        narrow_m rows (qs_narrow), all created from the same blocks (the automatic backend
        follows each set's m_max)."""
        from bit_weight_streaming_q4_gb300 import Qmm
        self.torch = torch
        self.mats = synth.stack(layers)
        self.m_max = m_max
        rows = max(m_max, wide_m)
        self.narrow_m = narrow_m
        self.qs, self.qs_wide, self.qs_narrow = [], [], []
        for mat in self.mats:
            blocks = synth.q4k_matrix(mat.n, mat.k, seed=seed, tensor_id=mat.tensor_id)
            dev = torch.from_numpy(blocks.reshape(-1)).cuda()
            self.qs.append(Qmm(dev, mat.n, mat.k, m_max=m_max))
            if wide_m:
                self.qs_wide.append(Qmm(dev, mat.n, mat.k, m_max=wide_m))
            if narrow_m:
                self.qs_narrow.append(Qmm(dev, mat.n, mat.k, m_max=narrow_m))
            del dev
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self.weight_bytes = sum(m.weight_bytes for m in self.mats)
        # activations for every matrix (own stream per matrix), `rows` rows reserved each
        self.x_off, off = [], 0
        for mat in self.mats:
            self.x_off.append(off)
            off += rows * mat.k
        xh = np.empty(off, dtype=np.float16)
        for mat, o in zip(self.mats, self.x_off):
            xh[o:o + rows * mat.k] = synth.x_f16(rows, mat.k, seed=seed,
                                                  tensor_id=synth.X_ID_OFFSET + mat.tensor_id).ravel()
        self.x_host = xh
        self.x = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.float16)
        self.y_off, off = [], 0
        for mat in self.mats:
            self.y_off.append(off)
            off += rows * mat.n
        self.y = torch.zeros(off, dtype=torch.float32, device="cuda")

    def handles(self, m):
        if self.narrow_m and m <= self.narrow_m:
            return self.qs_narrow
        return self.qs if m <= self.m_max else self.qs_wide

    def x_ptrs(self):
        # rows 0..m-1 of matrix i start at x_off[i] (row stride K); m_max rows reserved
        return [self.x[o:].data_ptr() for o in self.x_off]

    def y_ptrs(self):
        return [self.y[o:].data_ptr() for o in self.y_off]

    def bytes_for(self, m):
        xb = sum(m * mat.k * 2 for mat in self.mats)
        yb = sum(m * mat.n * 4 for mat in self.mats)
        return self.weight_bytes, xb, yb


def measured_traffic(handles):
    """DRAM bytes of one step launch over `handles` from the ncu capture of their backend,
    scaled by the launch's units; None when there is no capture or the kernel source differs
    from the one the counters were taken from."""
    import hashlib
    ref = TRAFFIC_PER_UNIT.get(int(handles[0].info().backend))
    if ref is None:
        return None
    path = os.path.join(ROOT, ref["source"])
    try:
        with open(path, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != ref["sha256"]:
                return None
    except OSError:
        return None
    units = sum(q.info().units for q in handles)
    return ref["bytes"] * units


def lm_head_verify(stack, m, stream, reps=50):
    """Per-launch time of the lm_head run that writes y[m, 151936], of the fused argmax
    (qmm_run_argmax) on the same handle and activations, and of the split alternative (the
    run that writes y followed by a separate reduction of y); the fused argmax is checked
    against the plain run's y (exact: same arithmetic)."""
    torch = stack.torch
    i = len(stack.mats) - 1
    q = stack.handles(m)[i]
    mat = stack.mats[i]
    x = stack.x[stack.x_off[i]:].data_ptr()
    y = stack.y[stack.y_off[i]:]
    idx = torch.empty(m, dtype=torch.int32, device="cuda")
    val = torch.empty(m, dtype=torch.float32, device="cuda")
    s = stream.cuda_stream

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    us_y = timed(lambda: q.run(x, y.data_ptr(), m, s))
    yh = y[:m * mat.n].view(m, mat.n).cpu().numpy()
    us_a = timed(lambda: q.run_argmax(x, idx, val, m, s))
    ih, vh = idx.cpu().numpy(), val.cpu().numpy()
    ref = np.argmax(yh, axis=1)
    ok = bool(np.array_equal(ih, ref) and
              np.array_equal(vh.view(np.uint32), yh[np.arange(m), ref].view(np.uint32)))
    # the alternative to the fused call: write y, then reduce it in a separate pass (a library
    # reduction over the [m, 151936] fp32 logits, on the same stream), for comparison only
    ym = y[:m * mat.n].view(m, mat.n)

    def split():
        q.run(x, y.data_ptr(), m, s)
        with torch.cuda.stream(stream):
            torch.max(ym, dim=1)

    us_split = timed(split)
    wb = mat.weight_bytes
    return {"backend": int(q.info().backend), "us_write_y": us_y, "us_argmax": us_a,
            "us_write_y_then_separate_argmax": us_split,
            "fused_faster_than_split": us_a < us_split,
            "weight_gbs_write_y": wb / us_y / 1e3, "weight_gbs_argmax": wb / us_a / 1e3,
            "y_bytes_not_written": 4 * m * mat.n, "argmax_matches_y": ok}


def format_line(torch, fmt, code, m, stream, parity, reps=50):
    """Per-launch time of one lm_head-shaped matrix (151936 x 5120) in another block format
    at M rows, its weight GB/s, and a sampled oracle check of three rows."""
    from bit_weight_streaming_q4_gb300 import Qmm
    mat = synth.LM_HEAD
    blocks = synth.fmt_matrix(fmt, mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    dev = torch.from_numpy(blocks.reshape(-1)).cuda()
    q = Qmm(dev, mat.n, mat.k, m_max=16, format=code)
    del dev
    x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    yd = torch.empty((m, mat.n), dtype=torch.float32, device="cuda")
    s = stream.cuda_stream
    for _ in range(3):
        q.run(xd, yd, m, s)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        q.run(xd, yd, m, s)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    info = q.info()
    line = {"matrix": f"lm_head {mat.n} x {mat.k}", "m": m, "backend": int(info.backend),
            "weight_bytes": int(info.weight_bytes), "us_per_launch": us,
            "weight_gbs": info.weight_bytes / us / 1e3}
    if parity:
        import oracle
        rows = np.array([0, mat.n // 2, mat.n - 1])
        y_ref, s_ref = oracle.qmm(blocks[rows], x)
        got = yd.cpu().numpy()[:, rows]
        ratio = np.abs(got - y_ref) / (2e-3 * s_ref + 1e-6)
        line["parity"] = {"checked_outputs": int(ratio.size), "max_err_over_bound": float(ratio.max()),
                          "pass": bool(ratio.max() <= 1.0)}
    q.close()
    return line


def attention_line(torch, stream, hbm, parity, reps=50, w=synth.ATTN_DECODE, name=None):
    """Stacked-row decode attention of one layer (48 query heads over 8 KV heads, q8_0 KV in a
    shared paged pool): time per call, KV GB/s (every page read once per query tile of an
    agent) and a sampled oracle check of two rows.  The default workload is the pages' decode
    step (4 agents with 23,000 cached tokens, 1 token + 2 drafts each)."""
    from bit_weight_streaming_q4_gb300.qmm import ATTN_QUERY_TILE, AttnDims, attn_decode, attn_workspace_bytes
    table, total, ra, rl = w.build(seed=0)
    pool = synth.kv_pool(total, w.kv_heads, seed=0, tensor_id=60)
    q = synth.attn_q(len(ra), w.heads, seed=0, tensor_id=61)
    agent_rows = np.concatenate([[0], np.cumsum(np.bincount(ra, minlength=table.shape[0]))]).astype(np.int32)
    pool_d = torch.from_numpy(pool).cuda()
    table_d = torch.from_numpy(table).cuda()
    ar_d = torch.from_numpy(agent_rows).cuda()
    rl_d = torch.from_numpy(rl).cuda()
    q_d = torch.from_numpy(q.view(np.int16)).cuda().view(torch.float16)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    s = stream.cuda_stream
    dims = AttnDims(w.heads, w.kv_heads, table.shape[0], table.shape[1], total, w.rows_per_agent)
    ws = torch.empty(attn_workspace_bytes(dims, len(ra)), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        attn_decode(pool_d, table_d, ar_d, rl_d, q_d, out, w.kv_heads, s, ws, err, max_agent_rows=w.rows_per_agent)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        attn_decode(pool_d, table_d, ar_d, rl_d, q_d, out, w.kv_heads, s, ws, err, max_agent_rows=w.rows_per_agent)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    group = w.heads // w.kv_heads
    tiles = -(-w.rows_per_agent * group // ATTN_QUERY_TILE)  # query tiles per agent: each reads its pages
    kv_bytes = sum(w.pages_of()) * w.kv_heads * synth.KV_RECORD_BYTES * tiles
    agents = len(w.cache)
    line = {"workload": name or (f"{agents} agents x {w.cache[0]:,} cached tokens, {w.rows_per_agent} rows each "
                                 f"(1 token + {w.rows_per_agent - 1} drafts), {w.heads} query heads over "
                                 f"{w.kv_heads} KV heads of 128, q8_0 KV pool in 64-token pages; one layer"),
            "query_tiles_per_agent": tiles,
            "kv_bytes": kv_bytes, "us_per_call": us, "kv_gbs": kv_bytes / us / 1e3,
            "frac_of_hbm_measured": kv_bytes / us / 1e3 / hbm, "error_word": int(err.item()),
            "kernels_per_call": 2}
    if parity:
        import oracle
        rows = np.array([0, len(ra) - 1])
        ref, sabs = oracle.attn(pool, table, q[rows], ra[rows], rl[rows], w.kv_heads)
        got = out.cpu().numpy()[rows]
        ratio = np.abs(got - ref) / (2e-3 * sabs + 1e-6)
        line["parity"] = {"checked_outputs": int(ratio.size), "max_err_over_bound": float(ratio.max()),
                          "pass": bool(ratio.max() <= 1.0)}
    return line


def timed_calls(torch, stream, fn, calls, warmup=3):
    """Seconds for `calls` calls of fn(i) on `stream` after `warmup` untimed ones."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(calls):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def graph_of(torch, stream, fn):
    """fn() captured once into a CUDA graph on `stream` (calls short enough that the host's
    launch cost would otherwise set the pace); returns a function that replays it on
    `stream`."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()

    def replay():
        with torch.cuda.stream(stream):
            g.replay()

    replay.graph = g
    return replay


def copies_for(weight_bytes, floor=4):
    """Handles of one matrix to rotate through so that every call reads weights from HBM:
    at least `floor`, and at least 4 x L2 (129 MB) of weights in total."""
    return max(floor, -(-4 * 129_000_000 // weight_bytes))


def single_projection_line(torch, stream, hbm, parity, calls=400):
    """The single projection 4096 x 4096 at M = 1 (9.4 MB, L2-sized): cold weight GB/s over
    rotating copies (55 handles, 4 x L2) replayed from a CUDA graph, and the latency of one
    isolated call (the median of 20 calls, each timed alone on an idle GPU)."""
    from bit_weight_streaming_q4_gb300 import Qmm
    mat = synth.SINGLE_PROJECTION
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    dev = torch.from_numpy(blocks.reshape(-1)).cuda()
    n = copies_for(mat.weight_bytes)
    qs = [Qmm(dev, mat.n, mat.k, m_max=1) for _ in range(n)]
    del dev
    x = synth.x_f16(1, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    yd = torch.empty((1, mat.n), dtype=torch.float32, device="cuda")
    s = stream.cuda_stream

    def sweep():
        for q in qs:
            q.run(xd, yd, 1, s)

    replay = graph_of(torch, stream, sweep)
    reps = max(1, calls // n)
    t = timed_calls(torch, stream, lambda i: replay(), reps)
    calls = reps * n
    lat = []
    for i in range(20):
        lat.append(timed_calls(torch, stream, lambda j: qs[(i + j) % n].run(xd, yd, 1, s), 1, warmup=0) * 1e6)
    us = t * 1e6 / calls
    line = {"matrix": f"{mat.n} x {mat.k}", "m": 1, "backend": int(qs[0].info().backend), "copies": n,
            "us_per_call": us, "weight_gbs": mat.weight_bytes / us / 1e3,
            "frac_of_hbm_measured": mat.weight_bytes / us / 1e3 / hbm,
            "single_call_us_median": statistics.median(lat)}
    if parity:
        import oracle
        y_ref, s_ref = oracle.qmm(blocks, x)
        ratio = np.abs(yd.cpu().numpy() - y_ref) / (2e-3 * s_ref + 1e-6)
        line["parity"] = {"checked_outputs": int(ratio.size), "max_err_over_bound": float(ratio.max()),
                          "pass": bool(ratio.max() <= 1.0)}
    for q in qs:
        q.close()
    return line


SWEEP_M = (1, 2, 4, 8, 12, 16, 32, 64)


def m_sweep_line(torch, stream, hbm, calls=40):
    """gate_up (5120 -> 34816) and down (17408 -> 5120) of layer 0 at every M of the sweep:
    weight GB/s of the pair, run back to back on rotating copies (4 per handle set; the pair
    is 150.4 MB), replayed from a CUDA graph.  Handles per set: m_max 8 (mma.sync) for M <= 8,
    and 16, 32, 64 (tcgen05)."""
    from bit_weight_streaming_q4_gb300 import Qmm
    mats = [m for m in synth.layer_matrices(0) if m.name.endswith(("gate_up", "down"))]
    pair_bytes = sum(m.weight_bytes for m in mats)
    sets = {}
    devs = [torch.from_numpy(synth.q4k_matrix(m.n, m.k, seed=0, tensor_id=m.tensor_id).reshape(-1)).cuda()
            for m in mats]
    for mm in (8, 16, 32, 64):
        sets[mm] = [[Qmm(d, m.n, m.k, m_max=mm) for d, m in zip(devs, mats)] for _ in range(4)]
    del devs
    xs = [torch.from_numpy(synth.x_f16(64, m.k, seed=0, tensor_id=synth.X_ID_OFFSET + m.tensor_id)
                           .view(np.int16)).cuda().view(torch.float16) for m in mats]
    ys = [torch.empty((64, m.n), dtype=torch.float32, device="cuda") for m in mats]
    s = stream.cuda_stream
    out = {}
    for m in SWEEP_M:
        mm = 8 if m <= 8 else (16 if m <= 16 else (32 if m <= 32 else 64))
        hs = sets[mm]

        def four_pairs():
            for pair in hs:
                for q, x, y in zip(pair, xs, ys):
                    q.run(x, y, m, s)

        replay = graph_of(torch, stream, four_pairs)
        reps = max(1, calls // 4)
        t = timed_calls(torch, stream, lambda i: replay(), reps)
        per = t / (4 * reps)
        out[str(m)] = {"backend": int(hs[0][0].info().backend), "m_max": mm, "us_per_pair": per * 1e6,
                       "weight_gbs": pair_bytes / per / 1e9, "frac_of_hbm_measured": pair_bytes / per / 1e9 / hbm,
                       "tok_s": m / per}
    for hs in sets.values():
        for pair in hs:
            for q in pair:
                q.close()
    return {"matrices": "layer 0 gate_up 5120->34816 + down 17408->5120 (150.4 MB), independent runs",
            "by_m": out}


PREFILL_M = 524


def prefill_line(torch, stream, peaks, parity, steps=3, layers=synth.LAYERS):
    """Chunked prefill: M = 524 rows (512 prompt + 12 decode) through the 64-layer set without
    lm_head, activations N(0,1) with 1 % outliers x 20, handles with m_max = 524 (tcgen05, 128
    rows per launch: every matrix streams its weights 5 times).  Tensor-bound: reported
    against the measured bf16 tensor peak (fp16 runs at the same rate)."""
    from bit_weight_streaming_q4_gb300 import Qmm
    mats = synth.stack(layers, lm_head=False)
    m = PREFILL_M
    qs, xs, ys, flops, wb = [], [], [], 0, 0
    for mat in mats:
        dev = torch.from_numpy(synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id).reshape(-1)).cuda()
        qs.append(Qmm(dev, mat.n, mat.k, m_max=m))
        del dev
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id, outlier_p=0.01)
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.empty((m, mat.n), dtype=torch.float32, device="cuda"))
        flops += 2 * m * mat.n * mat.k
        wb += mat.weight_bytes
    s = stream.cuda_stream

    def step(_):
        for q, x, y in zip(qs, xs, ys):
            q.run(x, y, m, s)

    t = timed_calls(torch, stream, step, steps, warmup=1) / steps
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
    tflops = flops / t / 1e12
    line = {"workload": f"chunked prefill M={m} (512 prompt + 12 decode rows): {layers} x {{qkv, o, gate_up, down}}, "
                        f"no lm_head, x with 1% outliers x20",
            "m": m, "backend": int(qs[0].info().backend), "launches_per_run": -(-m // 128),
            "ms_per_step": t * 1e3, "tok_s": m / t, "weight_gbs": wb / t / 1e9, "tflops": tflops,
            "tensor_peak_tflops": peak, "frac_of_tensor_peak": tflops / peak,
            "note": "peak = measured bf16 sustained (fp16 has the same dense rate)"}
    if parity:
        import oracle
        worst, checked = 0.0, 0
        for i in (0, 1, 2, 3, len(mats) - 1):
            mat = mats[i]
            rows = np.array([0, mat.n // 2, mat.n - 1])
            blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=rows)
            x = xs[i].view(torch.int16).cpu().numpy().view(np.float16)
            y_ref, s_ref = oracle.qmm(blocks, x)
            got = ys[i].cpu().numpy()[:, rows]
            ratio = np.abs(got - y_ref) / (2e-3 * s_ref + 1e-6)
            worst = max(worst, float(ratio.max()))
            checked += ratio.size
        line["parity"] = {"checked_outputs": checked, "max_err_over_bound": worst, "pass": worst <= 1.0}
    for q in qs:
        q.close()
    del xs, ys
    torch.cuda.empty_cache()
    return line


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
class OracleWalk:
    """The oracle over a walk of the step's weights: five cursors, one per matrix shape (qkv,
    o, gate_up, down of layer 0, 1, 2, ... and lm_head), take turns running the next chunk of
    rows of their matrix against that matrix's M activation rows.  A sample runs chunks until
    it has taken ~target_s seconds of oracle time and continues where the last one stopped, so
    consecutive samples cover the step's shapes in proportion."""

    CHUNK_WEIGHTS = 8 << 20

    def __init__(self, layers: int = synth.LAYERS, m: int = HEADLINE_M):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.m = m
        self.lists = [[synth.layer_matrices(layer)[t] for layer in range(layers)] for t in range(4)]
        self.lists.append([synth.LM_HEAD])
        self.cur = [[0, 0] for _ in self.lists]   # (matrix index in its list, next row)
        self.turn = 0
        self.seen: dict[str, int] = {}
        self._x = {}
        oracle.qmm(synth.q4k_matrix(64, 5120, seed=0, tensor_id=9999),
                   synth.x_f16(m, 5120, seed=0, tensor_id=9999))  # start the thread pool

    def _x_for(self, mat):
        if mat.name not in self._x:
            self._x = {mat.name: synth.x_f16(self.m, mat.k, seed=0,
                                             tensor_id=synth.X_ID_OFFSET + mat.tensor_id)}
        return self._x[mat.name]

    def _chunk(self):
        for _ in range(len(self.lists)):
            t = self.turn
            self.turn = (self.turn + 1) % len(self.lists)
            i, r0 = self.cur[t]
            if i >= len(self.lists[t]):
                continue
            mat = self.lists[t][i]
            r1 = min(mat.n, r0 + max(16, self.CHUNK_WEIGHTS // mat.k))
            self.cur[t] = [i + 1, 0] if r1 == mat.n else [i, r1]
            return mat, r0, r1
        self.cur = [[0, 0] for _ in self.lists]   # walked the whole step: start again
        return self._chunk()

    def sample(self, target_s: float):
        """Returns (weights processed, oracle seconds)."""
        w, t = 0, 0.0
        while t < target_s:
            mat, r0, r1 = self._chunk()
            blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id,
                                      rows=np.arange(r0, r1))
            x = self._x_for(mat)
            t0 = time.perf_counter()
            self.oracle.qmm(blocks, x)
            t += time.perf_counter() - t0
            w += (r1 - r0) * mat.k
            self.seen[mat.name] = self.seen.get(mat.name, 0) + (r1 - r0)
        return w, t

    def describe(self, w, t):
        names = list(self.seen)
        shown = ", ".join(f"{n}[{self.seen[n]} rows]" for n in names[:6])
        more = f" and {len(names) - 6} more matrices" if len(names) > 6 else ""
        return (f"M={self.m}: {shown}{more} ({w * 144 // 256 / 1e6:.1f} MB of weights, {t:.1f} s "
                f"of oracle time); weight GB/s, the full step scaled by weight bytes")

    def cores(self):
        return self.oracle.max_threads()


def cpu_oracle_sample(target_s: float, layers: int = synth.LAYERS, m: int = HEADLINE_M):
    walk = OracleWalk(layers, m)
    w, t = walk.sample(target_s)
    return {"gbs": w * 144 / 256 / t / 1e9, "seconds": t, "cores": walk.cores(),
            "sample": walk.describe(w, t)}


def workload_config(layers: int, m: int, weight_bytes: int) -> dict:
    return {"workload": f"decode step M={m} (4 streams x (1 token + 2 drafts)): {layers} x "
                        f"{{qkv 5120->8192, o 6144->5120, gate_up 5120->34816, down 17408->5120}} "
                        f"+ lm_head 5120->151936, Q4_K 144 B/256 weights",
            "m": m, "matrices": 4 * layers + 1, "weight_bytes": weight_bytes,
            "l2": "inputs larger than L2 (12.7 GB of weights streamed per step; no flush)"}


def run_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores.  Each step is a bounded
    sample of the step's weights (a walk over its matrices), so that K steps take about
    --cpu-seconds of oracle time in total."""
    if rank != 0:
        return
    full_bytes = sum(m.weight_bytes for m in synth.stack(args.layers))
    per_step_s = max(0.02, args.cpu_seconds / max(args.steps, 1))
    walk = OracleWalk(args.layers, HEADLINE_M)
    for _ in range(args.warmup):
        walk.sample(per_step_s)
    walk.seen.clear()
    w, t = 0, 0.0
    for _ in range(args.steps):
        dw, dt = walk.sample(per_step_s)
        w += dw
        t += dt
    gbs = w * 144 / 256 / t / 1e9
    step_s = full_bytes / (gbs * 1e9)
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args.layers, HEADLINE_M, full_bytes),
        "tok_s": HEADLINE_M / step_s,
        "ms_per_step_extrapolated": "ms_per_step is the full step's weight bytes at the oracle's "
                                    "rate on the sampled matrices (no full step was run)",
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": walk.cores(), "kind": "oracle",
                         "sample": walk.describe(w, t)},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------- replicas
# With N GPUs the step runs as N independent replicas (one process per GPU, nothing of the
# data path crosses ranks): the timed region is bracketed by a barrier on every rank, the
# time is the maximum over ranks, and the job's figure counts the work of all ranks.
def ranks_barrier(world: int, cuda: bool) -> None:
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        torch.cuda.synchronize()


def ranks_max(t: float, world: int, device: str) -> float:
    """The largest of the ranks' values of t (every rank gets it)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        tt = torch.tensor([t], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    return t


def job_gbs(weight_bytes_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Weight GB/s of the whole job: every rank streams the step's weights once per step."""
    return weight_bytes_per_step * steps * world / seconds / 1e9


# ------------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    from bit_weight_streaming_q4_gb300 import Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_INDEPENDENT, STEP_PERSISTENT

    torch.cuda.set_device(local_rank)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    # decode handles: up to 16 rows (the automatic backend: mma.sync) for M = 12 and M = 1, up to
    # 64 rows (tcgen05) for M = 64
    wide = 0 if args.no_extra else max(m for m in EXTRA_M)
    stack = Stack(args.layers, 16, torch, wide_m=wide if wide > 16 else 0)
    stream = torch.cuda.Stream()
    n_mats = len(stack.mats)

    def barrier():
        ranks_barrier(world, cuda=True)

    def max_over_ranks(t):
        return ranks_max(t, world, "cuda")

    def make_step(m, flags, xs=None, ys=None, qs=None):
        with torch.cuda.stream(stream):
            return Step(stack.handles(m) if qs is None else qs, stack.x_ptrs() if xs is None else xs,
                        stack.y_ptrs() if ys is None else ys, m, stream=stream.cuda_stream, flags=flags)

    def measure(m, flags, steps, warmup, qs=None):
        step = make_step(m, flags, qs=qs)
        barrier()
        t = time_graph(torch, step, steps, warmup, stream)
        step.close()
        return max_over_ranks(t)

    # Headline: M = 12.  Every matrix has its own synthetic activations and no run reads
    # another's output, so the step is created with STEP_INDEPENDENT (one persistent kernel
    # streams all 257 matrices).  Timed with the clocks sampled.
    step = make_step(HEADLINE_M, STEP_INDEPENDENT)
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
    t = max_over_ranks(e0.elapsed_time(e1) / 1e3)
    step.close()
    clocks = clk.summary()
    wb, xb, yb = stack.bytes_for(HEADLINE_M)
    step_s = t / args.steps
    value = job_gbs(wb, args.steps, world, t)
    alg_bytes = wb + xb + yb
    achieved = alg_bytes / step_s / 1e9
    parity = None
    if not args.no_parity:
        parity = sampled_parity(stack, HEADLINE_M)

    # End to end through the public API with host buffers: each step copies every matrix's M
    # activation rows from pinned host memory (one dense slab), launches the step, and copies
    # every output back (one dense slab).
    xo, yo, offx, offy = [], [], 0, 0
    for mat in stack.mats:
        xo.append(offx)
        yo.append(offy)
        offx += HEADLINE_M * mat.k
        offy += HEADLINE_M * mat.n
    x_dense = np.concatenate([stack.x_host[o:o + HEADLINE_M * mat.k]
                              for mat, o in zip(stack.mats, stack.x_off)])
    x_pin = torch.from_numpy(x_dense.view(np.int16)).view(torch.float16).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    # (1) serialised: each step's copies and launch one after the other on one stream
    y_pin = torch.empty(offy, dtype=torch.float32).pin_memory()
    xd = torch.empty(offx, dtype=torch.float16, device="cuda")
    yd = torch.empty(offy, dtype=torch.float32, device="cuda")
    e2e_step = make_step(HEADLINE_M, STEP_INDEPENDENT, [xd[o:].data_ptr() for o in xo],
                         [yd[o:].data_ptr() for o in yo])

    def e2e_once():
        # the C-ABI host-buffer call: copy in, run, copy out, all on one stream
        e2e_step.launch_host(x_pin, y_pin, stream.cuda_stream)

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
    te_serial = max_over_ranks(a0.elapsed_time(a1) / 1e3)
    e2e_step.close()
    ydev = stack.y.cpu().numpy()

    def matches(yh):
        return all(np.array_equal(yh[a:a + HEADLINE_M * mat.n].view(np.uint32),
                                  ydev[b:b + HEADLINE_M * mat.n].view(np.uint32))
                   for mat, a, b in zip(stack.mats, yo, stack.y_off))

    e2e_ok = matches(y_pin.numpy())
    # (2) pipelined, as a server streams steps: two sets of device buffers (two steps), called
    # alternately through the same C-ABI call on one stream, with the copies in and out on
    # two more streams: step i's inputs are copied in while step i - 1 runs, and its outputs
    # copied out while step i + 1 runs.  Timed from the first input copy to the last output copy.
    xds = [xd, torch.empty(offx, dtype=torch.float16, device="cuda")]
    yds = [yd, torch.empty(offy, dtype=torch.float32, device="cuda")]
    ypins = [y_pin, torch.empty(offy, dtype=torch.float32).pin_memory()]
    steps2 = [make_step(HEADLINE_M, STEP_INDEPENDENT, [xds[b][o:].data_ptr() for o in xo],
                        [yds[b][o:].data_ptr() for o in yo]) for b in (0, 1)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(n):
        for i in range(n):
            b = i % 2
            steps2[b].launch_host(x_pin, ypins[b], stream.cuda_stream, h2d.cuda_stream, d2h.cuda_stream)

    pipelined(3)
    torch.cuda.synchronize()
    barrier()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(h2d)
    pipelined(e2e_steps)
    d2h.wait_stream(stream)
    p1.record(d2h)
    torch.cuda.synchronize()
    te = max_over_ranks(p0.elapsed_time(p1) / 1e3)
    e2e_ok = e2e_ok and matches(ypins[(e2e_steps - 1) % 2].numpy())
    for st2 in steps2:
        st2.close()

    head_backend = int(stack.handles(HEADLINE_M)[0].info().backend)
    by_m = {str(HEADLINE_M): {"weight_gbs": value / world, "tok_s": HEADLINE_M / step_s,
                              "ms_per_step": step_s * 1e3, "runs": "independent", "backend": head_backend}}
    # the same step as a chain of dependent runs (each matrix may read the previous one's
    # output): a CUDA graph of runs linked by programmatic dependent launch
    steps_dep = max(20, args.steps // 2)
    td = measure(HEADLINE_M, 0, steps_dep, 3) / steps_dep
    dependent = {"weight_gbs": wb / td / 1e9, "tok_s": HEADLINE_M / td, "ms_per_step": td * 1e3,
                 "runs": "dependent (CUDA graph)", "backend": head_backend}
    if stack.qs_wide and int(stack.qs_wide[0].info().backend) == 2:
        # the dependent step on tcgen05 handles (the wide set) at M = 12: as a graph, and as one
        # persistent launch (QMM_STEP_PERSISTENT, which only the tcgen05 kernel supports)
        tdg = measure(HEADLINE_M, 0, steps_dep, 3, qs=stack.qs_wide) / steps_dep
        tdp = measure(HEADLINE_M, STEP_PERSISTENT, steps_dep, 3, qs=stack.qs_wide) / steps_dep
        dependent["tcgen05"] = {
            "graph": {"weight_gbs": wb / tdg / 1e9, "ms_per_step": tdg * 1e3},
            "persistent": {"weight_gbs": wb / tdp / 1e9, "ms_per_step": tdp * 1e3,
                           "runs": "dependent, one persistent launch (QMM_STEP_PERSISTENT)"},
            "handles": f"m_max {max(EXTRA_M)} (tcgen05)"}
    if not args.no_extra:
        for m in EXTRA_M:
            steps_m = max(20, args.steps // (4 if m > 16 else 1))
            tm = measure(m, STEP_INDEPENDENT, steps_m, 3)
            sm = tm / steps_m
            wbm, xbm, ybm = stack.bytes_for(m)
            by_m[str(m)] = {"weight_gbs": wbm / sm / 1e9, "tok_s": m / sm, "ms_per_step": sm * 1e3,
                            "frac_of_hbm_measured": wbm / sm / 1e9 / hbm,
                            "backend": int(stack.handles(m)[0].info().backend),
                            "runs": "independent (one persistent kernel per step)"}
            if not args.no_parity:
                last = len(stack.mats) - 1
                by_m[str(m)]["parity"] = sampled_parity(stack, m, matrices=[0, 1, 2, 3, last])

    # Greedy verification of the lm_head fused into its matmul (qmm_run_argmax) against the
    # plain run that writes y, per launch, on the step's lm_head handles and activations
    verify = None
    formats = None
    attention = None
    single = sweep = prefill = attention_verify = None
    if not args.no_extra:
        verify = {str(m): lm_head_verify(stack, m, stream) for m in sorted({*EXTRA_M, HEADLINE_M})}
        # the other block formats of a mixed-quant file, on the lm_head shape at M = 12
        formats = {name: format_line(torch, f, code, HEADLINE_M, stream, not args.no_parity)
                   for name, f, code in (("Q6_K", synth.Q6_K, 1), ("Q8_0", synth.Q8_0, 2))}
        attention = attention_line(torch, stream, hbm, not args.no_parity)
        attention_verify = attention_line(torch, stream, hbm, not args.no_parity, w=synth.ATTN_VERIFY)
        single = single_projection_line(torch, stream, hbm, not args.no_parity)
        sweep = m_sweep_line(torch, stream, hbm)
        prefill = prefill_line(torch, stream, peaks, not args.no_parity, layers=args.layers)

    cpu = None
    if rank == 0:
        c = cpu_oracle_sample(args.cpu_seconds)
        cpu = {"value": c["gbs"], "unit": "GB/s", "cores": c["cores"], "kind": "oracle",
               "sample": c["sample"]}

    info = stack.handles(HEADLINE_M)[0].info()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {**workload_config(args.layers, HEADLINE_M, wb),
                   "runs": "independent: every matrix has its own synthetic activations and no "
                           "run reads another's output (one persistent kernel per step)",
                   "backend": int(info.backend), "ctas": int(info.grid),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tok_s": HEADLINE_M * world / step_s,
        "frac_of_hbm": {"measured": value / world / hbm, "nominal_8TBs": value / world / NOMINAL_HBM_GBS},
        "by_m": by_m,
        "dependent_step": dependent,
        "lm_head_verify": verify,
        "formats": formats,
        "attention": attention,
        "attention_verify": attention_verify,
        "single_projection": single,
        "m_sweep": sweep,
        "chunked_prefill": prefill,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": measured_traffic(stack.handles(HEADLINE_M)),
                     "kernel": f"{KERNEL_NAME[head_backend]} (one persistent launch per step)",
                     "note": f"algorithmic bytes per step (weights + x + y of the 257 matrices) "
                             f"/ step time (the stream kernel plus, for mma.sync, its fragment "
                             f"pre-pass); peak is the {peak_kind} copy bandwidth"},
        "cpu_baseline": cpu,
        "e2e": {"value": wb * e2e_steps / te / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": xb, "d2h_bytes_per_step": yb,
                "ms_per_step": te / e2e_steps * 1e3, "outputs_match_device_run": e2e_ok,
                "steps": e2e_steps,
                "how": "C-ABI host-buffer call qmm_step_launch_host: every step's activations copied in "
                       "from pinned host memory and its outputs copied back, inside the timed region; "
                       "two steps over two device buffer sets called alternately, with the copies on two "
                       "more streams, so the copies of adjacent steps overlap the running step",
                "serialised": {"value": wb * e2e_steps / te_serial / 1e9,
                               "ms_per_step": te_serial / e2e_steps * 1e3,
                               "how": "qmm_step_launch_host with copy in, launch and copy out on one stream"}},
        # a persistent mma.sync step is two launches (the activation-fragment pre-pass, then the
        # stream); a tcgen05 step at M <= 64 is one
        "gpu_launches": args.steps * (2 if head_backend == 1 else 1),
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
    if args.single in ("attention", "attention_verify"):
        peaks, _ = measured_peaks()
        stream = torch.cuda.Stream()
        w = synth.ATTN_DECODE if args.single == "attention" else synth.ATTN_VERIFY
        line = attention_line(torch, stream, float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS)), not args.no_parity,
                              reps=max(args.steps, 1), w=w)
        print(json.dumps({"single": args.single, **line}), flush=True)
        return
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
