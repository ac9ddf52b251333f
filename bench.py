"""Benchmark of the fused attention forward pass (one JSON line on stdout).

A step is one forward pass (one kernel launch of the C-ABI library) over the
headline workload, the largest single-GPU configuration: long-sequence prefill,
B=1, H=8, N=16384, D=128, fp16, non-causal, Q and K drawn N(0,1) then scaled by
4 (exp(m_old - m_new) underflows), V ~ U(-1,1), inputs resident in HBM. The
steps cycle through enough copies of the inputs (and outputs) that their total
is more than twice the 126 MB L2, so no step finds its inputs in L2; the K timed
steps run back to back on one stream between two CUDA events (the mean step
time); a second pass of K steps with an event between consecutive steps gives
the median, p10 and p90.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fa|reference]
                    [--workload c1..c5] [--kernel-only] [--no-sweep]

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step). --kernel-only runs just the
warm-up and timed kernel steps (the form used under ncu); with --path splitkv
or naive it runs the split-KV forward or the unfused baseline instead.

Under torchrun each rank runs its own replica of the workload (the forward
pass has no exchange step); value = all ranks' FLOPs / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS and % of GB300 fp16/bf16 tensor peak; DRAM bytes vs min"
UNIT = "TFLOP/s"
HEADLINE = "c5"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 126 << 20
# The sources of the fused kernels whose DRAM traffic profiles/fa_fwd_dram_traffic.json records.
KERNEL_SOURCES = ["tiled_attention_prefill_gb300/csrc/" + f for f in
                  ("fa_kernel.cuh", "fa_kernel_f32.cuh", "ptx.cuh", "fa_launch.cuh", "fa_api.cu", "fa_inst_f32.cu")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fa_fwd_dram_traffic.json")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def measured_traffic(workload: str):
    """ncu DRAM bytes per launch for this workload, if taken on the current kernel sources."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get("workloads", {}).get(workload)
    if not e or e.get("kernel_sources_sha256_16") != kernel_source_hash():
        return None
    return e


class ClockSampler:
    """nvidia-smi sampling (200 ms) while the GPU is busy; median SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "fa_bench_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        busy = [r for r in rows if r[4].replace(".", "", 1).isdigit() and float(r[4]) > 0] or rows
        sm = [float(r[1]) for r in busy if r[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(busy[0][2]) if busy[0][2].replace(".", "", 1).isdigit() else None,
                "reasons": reasons, "samples": len(busy)}


def dist_setup(want_gpu: bool):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if (want_gpu and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_desc(w):
    return {"workload": "%s: %s" % (w.name, w.note), "B": w.B, "H": w.H, "N": w.N, "D": w.D,
            "dtype": w.dtype, "causal": w.causal, "scale": "1/sqrt(D)",
            "values": "Q,K x%g N(0,1); V %s" % (w.qk_mult, "U(-1,1)" if w.v_uniform else "N(0,1)")}


def traffic_fields(w, tr):
    """Traffic of one launch (ncu summary) against the minimum |Q|+|K|+|V|+|O|.

    traffic = DRAM bytes read + bytes the kernel stored. The stores (O, lse) are counted where
    they enter L2 (write sectors x 32 B): O of a small workload can still sit in the L2 when the
    kernel ends, so DRAM write counters taken over the launch alone miss it, but every stored
    byte is a distinct output byte and reaches DRAM exactly once."""
    from tiled_attention_prefill_gb300 import workloads
    eb = 4 if w.dtype == "fp32" else 2
    qkv = 3 * w.B * w.H * w.N * w.D * eb
    o = w.B * w.H * w.N * w.D * eb
    lse = 4 * w.B * w.H * w.N
    out = {"min_bytes": workloads.min_dram_bytes(w.B, w.H, w.N, w.D, elem_bytes=eb, with_lse=False),
           "traffic_bytes": None, "traffic_vs_min": None, "read_vs_qkv": None, "stored_vs_o": None}
    if not tr or tr.get("stored_bytes") is None:
        return out
    t = tr["read_bytes"] + tr["stored_bytes"]
    out.update(traffic_bytes=t, traffic_vs_min=t / out["min_bytes"], traffic_vs_min_with_lse=t / (qkv + o + lse),
               read_vs_qkv=tr["read_bytes"] / qkv, stored_vs_o=tr["stored_bytes"] / (o + lse),
               dram_write_in_launch=tr.get("write_bytes"))
    return out


def sample_rows(w, n_heads=4, seed=0):
    """(b*H + h, i) pairs: tile edges, first and last rows, and random rows of a few heads."""
    import numpy as np
    rng = np.random.default_rng(seed)
    BH, N = w.B * w.H, w.N
    heads = sorted(set([0, BH - 1] + rng.integers(0, BH, size=n_heads).tolist()))
    fixed = [0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = []
    for bh in heads:
        idx = set(i for i in fixed if 0 <= i < N) | set(rng.integers(0, N, size=24).tolist())
        rows += [(bh, i) for i in sorted(idx)]
    return np.array(rows, dtype=np.int64)


def sampled_errors(w, rows, go, gl):
    """Max abs errors of the CUDA path's sampled rows against the oracle on the same rows."""
    import numpy as np

    import oracle
    from tiled_attention_prefill_gb300 import workloads
    q, k, v = workloads.make_qkv(w)
    ro, rl = oracle.attention_rows(q, k, v, w.scale, w.causal, rows)
    return float(np.abs(go - ro).max()), float(np.abs(gl - rl).max())


# ----------------------------------------------------------------------------- CPU oracle arm
def cpu_oracle_rate(w, budget_s: float = 12.0, max_heads=None, gpu_out=None, parity=None):
    """Time the oracle on whole heads of the workload until ~budget_s; returns (TFLOP/s, sample, threads).

    gpu_out: optional (O [B*H, N, D], lse [B*H, N]) fp64 arrays of the CUDA path on the same
    inputs; the heads the oracle computed are then compared with them (untimed) and the
    largest errors are stored in the dict `parity`."""
    import numpy as np

    import oracle
    from tiled_attention_prefill_gb300 import workloads

    q, k, v = workloads.make_qkv(w)
    q64, k64, v64 = (oracle.to_f64(x) for x in (q, k, v))
    per_head = workloads.attention_flops(1, 1, w.N, w.D, w.causal)
    threads = oracle.max_threads()
    BH = w.B * w.H
    done_heads, elapsed = 0, 0.0
    h = 0
    while (done_heads < max_heads) if max_heads is not None else (done_heads == 0 or elapsed < budget_s):
        rows = np.stack([np.full(w.N, h % BH), np.arange(w.N)], axis=1)
        t0 = time.perf_counter()
        ro, rl = oracle.attention_rows(q64, k64, v64, w.scale, w.causal, rows)
        elapsed += time.perf_counter() - t0
        if gpu_out is not None and parity is not None:
            eo = float(np.abs(gpu_out[0][h % BH] - ro).max())
            el = float(np.abs(gpu_out[1][h % BH] - rl).max())
            parity["o_max_abs_err"] = max(parity.get("o_max_abs_err", 0.0), eo)
            parity["lse_max_abs_err"] = max(parity.get("lse_max_abs_err", 0.0), el)
            parity["heads_compared"] = parity.get("heads_compared", 0) + 1
        done_heads += 1
        h += 1
    rate = per_head * done_heads / elapsed / 1e12
    sample = "%d whole head(s) (all %d query rows each) of workload %s, fp64 oracle" % (done_heads, w.N, w.name)
    return rate, sample, threads, elapsed


def run_reference(args, w):
    """The reference arm: the fp64 oracle on the host cores, one bounded sample per step.

    A step is a block of `rows_per_step` consecutive query rows of one head (the blocks cycle
    through the heads and row ranges of the workload); its FLOPs are counted exactly (4*D per
    unmasked (query, key) pair)."""
    world, rank, _ = dist_setup(want_gpu=False)
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from tiled_attention_prefill_gb300 import workloads
    oracle.build()
    rows_per_step = min(w.N, 2048)
    q, k, v = workloads.make_qkv(w)
    q64, k64, v64 = (oracle.to_f64(x) for x in (q, k, v))
    BH = w.B * w.H
    blocks = [(bh, r0) for bh in range(BH) for r0 in range(0, w.N, rows_per_step)]

    def step(i):
        bh, r0 = blocks[i % len(blocks)]
        idx = np.arange(r0, min(r0 + rows_per_step, w.N))
        rows = np.stack([np.full(len(idx), bh), idx], axis=1)
        keys = (idx + 1).sum() if w.causal else len(idx) * w.N
        t0 = time.perf_counter()
        oracle.attention_rows(q64, k64, v64, w.scale, w.causal, rows)
        return time.perf_counter() - t0, 4.0 * w.D * float(keys)

    for i in range(args.warmup):
        step(i)
    times, flops = [], []
    for i in range(args.steps):
        t, f = step(args.warmup + i)
        times.append(t)
        flops.append(f)
    value = sum(flops) / sum(times) / 1e12
    # n_gpus is the launch's N (the same as the GPU arm's line); the work runs on rank 0's host cores
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": "%d consecutive query rows of one head per step of workload %s (fp64 "
                                       "oracle, %.3g FLOP per step on average)"
                                       % (rows_per_step, w.name, statistics.mean(flops))},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def time_steps(fwd, steps, warmup, stream, per_step=None):
    """Mean CUDA-event time (ms) of one step over `steps` back-to-back calls fwd(i) on `stream`.

    The timed region has one event before the first step and one after the last, so
    consecutive launches keep their overlap (programmatic dependent launch). If `per_step` is a
    list, a second pass of `steps` calls follows with an event between consecutive steps, and
    its step times (ms) are appended to it: an event between two launches removes that
    overlap, so these times are for the distribution (median, p10, p90), not the mean."""
    import torch
    for i in range(warmup):
        fwd(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        fwd(warmup + i)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = start.elapsed_time(end) / steps
    if per_step is not None:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            fwd(warmup + steps + i)
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        per_step.extend(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
    return ms


def step_stats(per_step):
    """Median, p10 and p90 (ms) of the step times."""
    xs = sorted(per_step)
    if not xs:
        return None

    def pct(p):
        i = p * (len(xs) - 1)
        lo = int(i)
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (i - lo)
    return {"median_ms": pct(0.5), "p10_ms": pct(0.1), "p90_ms": pct(0.9), "n": len(xs),
            "method": "a second pass of the same steps with a CUDA event between consecutive steps"}


def n_copies(bytes_per_set: int, cap_bytes: int = 4 << 30) -> int:
    """Input/output sets to cycle through so that their total exceeds twice the L2."""
    n = -(-2 * L2_BYTES // max(1, bytes_per_set))
    return int(max(2, min(n, max(2, cap_bytes // max(1, bytes_per_set)))))


def run_fa(args, w):
    import torch

    world, rank, local = dist_setup(want_gpu=True)
    from tiled_attention_prefill_gb300 import _build, fa, workloads

    if rank == 0 or world == 1:
        _build.build()
    barrier()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_kind = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # tf32 (the fp32-I/O kernel): the measured bf16 peak times the nominal dense ratio 1.1 / 2.25
    peak_of = {"fp16": peak_tf, "bf16": peak_tf, "fp32": peak_tf * 1.1 / 2.25}
    copies_used = {}

    def measure(wl, steps, warmup, splits=None, naive=False, per_step=None, rows=None, outputs=None):
        """Mean step time (ms) with the inputs cycled over enough copies to defeat L2.

        splits: None times fa_forward; an integer times fa_forward_splitkv with that many
        splits (one workspace, reused by every step in stream order). naive: times the
        unfused baseline fa_naive_forward (its S/P workspace reused likewise). per_step: a
        list that receives the step times. After the timed steps, one more (untimed) call on
        the first input set; `rows` (an int64 array of (b*H + h, i) pairs) selects output rows
        of it returned as fp64 host arrays (O [R, D], lse [R]) in outputs["rows"], and
        outputs["full"] receives the whole result (O [B*H, N, D], lse [B*H, N]) when present."""
        q0, k0, v0 = workloads.make_qkv(wl)
        set_bytes = 4 * q0.numel() * q0.element_size() + wl.B * wl.H * wl.N * 4
        n = n_copies(set_bytes)
        copies_used[wl.name] = (n, n * set_bytes)
        sets = []
        for _ in range(n):
            q, k, v = (x.to(dev) for x in (q0, k0, v0))
            sets.append((q, k, v, torch.empty_like(q), torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)))

        ws = None
        if splits is not None:
            ws = torch.empty(max(1, fa.splitkv_workspace_bytes(wl.B, wl.H, wl.N, wl.D, splits)), dtype=torch.uint8,
                             device=dev)
        if naive:
            ws = torch.empty(fa.naive_workspace_bytes(wl.B, wl.H, wl.N), dtype=torch.uint8, device=dev)

        def fwd(i):
            q, k, v, o, lse = sets[i % n]
            if naive:
                fa.naive_forward(q, k, v, causal=wl.causal, scale=wl.scale, workspace=ws, out=o, lse=lse)
            elif splits is None:
                fa.forward(q, k, v, causal=wl.causal, scale=wl.scale, out=o, lse=lse)
            else:
                fa.forward_splitkv(q, k, v, causal=wl.causal, scale=wl.scale, num_splits=splits, workspace=ws,
                                   out=o, lse=lse)

        ms = time_steps(fwd, steps, warmup, stream, per_step)
        fa.check_device_status()
        if outputs is not None:
            fwd(0)
            torch.cuda.synchronize()
            o_all = sets[0][3].reshape(wl.B * wl.H, wl.N, wl.D)
            l_all = sets[0][4].reshape(wl.B * wl.H, wl.N)
            if rows is not None:
                ri = torch.as_tensor(rows, device=dev)
                outputs["rows"] = (o_all[ri[:, 0], ri[:, 1]].double().cpu().numpy(),
                                   l_all[ri[:, 0], ri[:, 1]].double().cpu().numpy())
            if "full" in outputs:
                outputs["full"] = (o_all.double().cpu().numpy(), l_all.double().cpu().numpy())
        flops = workloads.attention_flops(wl.B, wl.H, wl.N, wl.D, wl.causal)
        del sets, ws
        return ms, flops

    def measure_merge(wl, splits, steps=20):
        """The merge kernel alone on partials of this workload's size (HBM-bound): ms, bytes."""
        P = splits
        op = torch.randn((P, wl.B, wl.H, wl.N, wl.D), device=dev)
        lp = torch.randn((P, wl.B, wl.H, wl.N), device=dev)
        o = torch.empty((wl.B, wl.H, wl.N, wl.D), dtype=torch.float16, device=dev)
        lo = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)
        ms = time_steps(lambda i: fa.merge_partials(op, lp, out=o, lse=lo), steps, 3, stream)
        nbytes = (op.numel() + lp.numel()) * 4 + o.numel() * 2 + lo.numel() * 4
        del op, lp, o, lo
        return ms, nbytes

    sampler = ClockSampler(local) if not args.kernel_only else None
    if sampler:
        sampler.start()
    per_step = []
    head_out = {}
    if args.kernel_only and args.path != "fused":
        # the split-KV (automatic split count) or the naive path alone, for ncu captures
        splits = fa.splitkv_num_splits(w.B, w.H, w.N, w.D, w.causal) if args.path == "splitkv" else None
        ms_local, flops = measure(w, args.steps, args.warmup, splits=splits, naive=args.path == "naive")
    else:
        head_out = {} if args.kernel_only or args.no_cpu else {"full": None}
        ms_local, flops = measure(w, args.steps, args.warmup, per_step=per_step, outputs=head_out)
    ms = max_over_ranks(ms_local)
    value = world * flops / (ms * 1e-3) / 1e12
    if args.kernel_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "ms_per_step": ms,
                              "config": workload_desc(w), "kernel_only": True}), flush=True)
        return 0

    # End to end through the public API: pinned host inputs -> device -> forward -> pinned host,
    # every step. q, k, v share one pinned buffer and o, lse another (one H2D and one D2H copy
    # per step). Steps are pipelined the way a server runs a stream of requests: the H2D copy,
    # the forward and the D2H copy run on three streams with two buffer sets, so the copies of
    # one step overlap the forward of its neighbours (events keep each buffer set in order).
    q_c, k_c, v_c = workloads.make_qkv(w)
    numel = q_c.numel()
    o_bytes = numel * q_c.element_size()
    l_bytes = w.B * w.H * w.N * 4
    in_h, in_d, out_d, out_h, views = [], [], [], [], []
    for b in range(2):
        ih = torch.empty(3 * numel, dtype=q_c.dtype).pin_memory()
        ih.view(3, -1).copy_(torch.stack([q_c.reshape(-1), k_c.reshape(-1), v_c.reshape(-1)]))
        idv = torch.empty_like(ih, device=dev)
        od = torch.empty(o_bytes + l_bytes, dtype=torch.uint8, device=dev)
        in_h.append(ih)
        in_d.append(idv)
        out_d.append(od)
        out_h.append(torch.empty(o_bytes + l_bytes, dtype=torch.uint8).pin_memory())
        views.append(tuple(x.view(q_c.shape) for x in idv.view(3, -1).unbind(0)) +
                     (od[:o_bytes].view(q_c.dtype).view(q_c.shape), od[o_bytes:].view(torch.float32).view(w.B, w.H, w.N)))
    s_in, s_fw, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer set b on the device
    ev_fw = [torch.cuda.Event() for _ in range(2)]    # forward on set b done (inputs free, output ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # output of set b copied to the host

    def e2e_steps(n, first):
        for i in range(first, first + n):
            b = i & 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_fw[b])
                in_d[b].copy_(in_h[b], non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_fw):
                s_fw.wait_event(ev_in[b])
                s_fw.wait_event(ev_out[b])
                q_d, k_d, v_d, o_d, l_d = views[b]
                fa.forward(q_d, k_d, v_d, causal=w.causal, scale=w.scale, out=o_d, lse=l_d)
                ev_fw[b].record(s_fw)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fw[b])
                out_h[b].copy_(out_d[b], non_blocking=True)
                ev_out[b].record(s_out)

    e2e_steps(args.warmup, 0)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for st_ in (s_in, s_fw, s_out):
        st_.wait_event(t0)
    e2e_steps(args.steps, args.warmup)
    for ev in ev_out:
        stream.wait_event(ev)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1) / args.steps)
    h2d = in_h[0].numel() * in_h[0].element_size()
    d2h = out_h[0].numel()

    sweep = {}
    sweep_rows = {}  # workload -> (sampled rows, GPU O rows, GPU lse rows), for the oracle leg
    if not args.no_sweep:
        for name, wl in workloads.WORKLOADS.items():
            st = 50 if wl.N <= 4096 else 20
            steps_ms = []
            rows = sample_rows(wl) if not args.no_cpu else None
            outs = {} if rows is not None else None
            m, f = measure(wl, st, 3, per_step=steps_ms, rows=rows, outputs=outs)
            if rows is not None:
                sweep_rows[name] = (rows,) + outs["rows"]
            tf = f / (m * 1e-3) / 1e12
            sweep[name] = {"ms_mean": m, "step_ms": step_stats(steps_ms), "tflops": tf,
                           "frac_of_peak": tf / peak_of[wl.dtype], "peak_tflops": peak_of[wl.dtype],
                           "input_copies": copies_used[name][0]}
            sweep[name].update(traffic_fields(wl, measured_traffic(name)))
            # the unfused baseline (S and P in memory) on the fp16 workloads whose S fits in 1 GiB
            if wl.dtype == "fp16" and wl.B * wl.H * wl.N * wl.N * 2 <= (1 << 30):
                m3, _ = measure(wl, st, 3, naive=True)
                sweep[name]["naive"] = {"ms_mean": m3, "tflops": f / (m3 * 1e-3) / 1e12, "fused_speedup": m3 / m,
                                        "s_bytes": wl.B * wl.H * wl.N * wl.N * 2}
            # split-KV forward where its automatic split count is above one
            S = fa.splitkv_num_splits(wl.B, wl.H, wl.N, wl.D, wl.causal)
            if S > 1:
                m2, _ = measure(wl, st, 3, splits=S)
                mm, mb = measure_merge(wl, S)
                hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
                sweep[name]["splitkv"] = {
                    "splits": S, "ms_mean": m2, "tflops": f / (m2 * 1e-3) / 1e12,
                    "frac_of_peak": f / (m2 * 1e-3) / 1e12 / peak_tf, "speedup_vs_fused": m / m2,
                    "merge_alone": {"ms": mm, "bytes": mb, "gbs": mb / (mm * 1e-3) / 1e9,
                                    "frac_of_hbm": mb / (mm * 1e-3) / 1e9 / hbm}}
    clocks = sampler.stop() if sampler else None

    if rank != 0:
        return 0
    achieved = flops / (ms_local * 1e-3) / 1e12
    tf_fields = traffic_fields(w, measured_traffic(w.name))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(workload_desc(w),
                       l2="inputs larger than L2: steps cycle over %d copies of q/k/v/o/lse (%.0f MiB in total, "
                          "> 2 x 126 MB L2); timed steps back to back on one stream between two CUDA events"
                          % (copies_used[w.name][0], copies_used[w.name][1] / 2**20),
                       parallelism="replicas" if world > 1 else "single GPU"),
        "step_ms": step_stats(per_step),
        "pct_of_peak": 100.0 * achieved / peak_tf,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf,
                     "peak_source": "%s bf16_tflops (burst: the kernel is timed alone; fp16 dense rate equal)"
                                    % peak_kind,
                     "peak_sustained": peak_sus, "frac_of_sustained": achieved / peak_sus,
                     "traffic": tf_fields["traffic_bytes"],
                     "traffic_vs_min": tf_fields["traffic_vs_min"],
                     "read_vs_qkv": tf_fields["read_vs_qkv"], "stored_vs_o": tf_fields["stored_vs_o"],
                     "min_bytes": tf_fields["min_bytes"],
                     "traffic_def": "ncu, one launch: dram__bytes_read.sum + bytes the kernel stored "
                                    "(lts__t_sectors_srcunit_tex_op_write.sum x 32: O and lse, every byte of which "
                                    "reaches DRAM once, whether before or after the kernel ends)"},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "method": "every step copies its q, k, v in (one pinned H2D copy) and o, lse out (one D2H "
                          "copy); H2D, forward and D2H run on three streams with two buffer sets, so the "
                          "copies of a step overlap the forward of its neighbours"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if sweep:
        line["workloads"] = sweep
    if not args.no_cpu and world >= 1:
        # The oracle leg: the oracle timed on whole heads of the headline workload (the CPU
        # baseline); untimed, the same heads and sampled rows of every swept workload are
        # compared with the CUDA path's outputs (max abs errors).
        par = {}
        rate, sample, threads, el = cpu_oracle_rate(w, gpu_out=head_out.get("full"), parity=par)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                                "seconds": el}
        line["max_abs_err"] = dict(par, tol_o=2e-3 if w.dtype == "fp16" else 1e-2, tol_lse=1e-3,
                                   what="whole heads the oracle computed for the CPU baseline")
        for name, (rows, go, gl) in sweep_rows.items():
            eo, el_ = sampled_errors(workloads.WORKLOADS[name], rows, go, gl)
            sweep[name]["max_abs_err"] = {"o": eo, "lse": el_, "rows_compared": int(len(rows))}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 20 timed steps of the 0.7 ms headline forward (14 ms): the burst regime the kernel-alone peak
    # is measured in. Runs of several hundred steps settle under the power cap (sw_power_cap) about
    # 5% slower; the line reports the fraction of both the burst and the sustained peak.
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fa", "reference"], default="fa")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--kernel-only", action="store_true")
    ap.add_argument("--path", choices=["fused", "splitkv", "naive"], default="fused",
                    help="with --kernel-only: which forward to run")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warmup raised to 3 (timing rule)")
        args.warmup = 3
    from tiled_attention_prefill_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_fa(args, w)


if __name__ == "__main__":
    sys.exit(main())
