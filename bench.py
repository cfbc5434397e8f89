#!/usr/bin/env python3
"""Benchmark of the block-quantized weight-row hot path on GB300.

Headline (one JSON line on rank 0): Q4_0 decode GEMV weight GB/s over the
7B-shaped decode step (32 layers x {q,k,v,o 4096x4096, gate/up 11008x4096,
down 4096x11008}, batch 1, 224 GEMVs, 3.643 GB of Q4_0 weights), inputs
resident in HBM, the step replayed as one CUDA graph. A "step" is one decode
token: every weight read once, each activation quantized to Q8_0 inside the
GEMV kernel. The step's weights are far larger than L2 (3.6 GB vs 129 MB), so
no flush is needed between steps.

Also measured in the same run (keys of the JSON line):
  roofline      the dominant kernel (Q4_0 GEMV) timed alone over back-to-back
                launches on distinct 11008x4096 matrices, against the measured
                HBM copy bandwidth;
  e2e           the same metric through the C ABI with host buffers: per step
                the activations are copied from pinned host memory, the 224
                GEMVs are issued as direct C-ABI calls, and all outputs are read
                back to the host, then the host waits;
  secondary     the prefill GEMM (512 tokens, Q8_0, TOPS), the KV-cache write
                (28 layers x 32768 tokens x 8 x 128, K to Q4_0 with the
                mean-centering bias and V to Q8_0, GB/s) and the Qwen3-0.6B-shaped
                decode step (GB/s, L2 flushed between steps);
  cpu_baseline  the plain-C oracle's GEMV timed on this host's cores over a
                bounded sample of the same workload.

--impl reference times the oracle itself as the reference arm.
Under torchrun (N > 1) every rank runs an independent replica (the path has
no data exchange); time is the max over ranks and value sums all ranks' bytes.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4_0/Q8_0 decode GEMV weight GB/s (% of HBM peak); prefill GEMM int8 TOPS"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------ distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(value: float, dist) -> float:
    """Max of a float over all ranks (the slowest rank sets the time)."""
    if dist is None:
        return value
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() and \
        dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(bytes_per_rank_step: float, world: int, max_seconds_per_step: float) -> float:
    """Whole-job rate: all ranks' units over the slowest rank's time."""
    return bytes_per_rank_step * world / max_seconds_per_step


# ------------------------------------------------------------------ peaks --

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path, encoding="utf-8") as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_traffic(key: str):
    """DRAM bytes per launch from a committed ncu capture, or None if the
    kernel source changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path, encoding="utf-8") as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("sha256"):
        return None
    return float(rec["bytes_per_launch"])


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """SM clock, its maximum, power and the clock-event reasons, sampled every
    ~2 ms through NVML (read-only queries of libnvidia-ml via ctypes) by a
    background thread and kept only inside [t0, t1], so that even a timed
    region of a few milliseconds carries samples. Falls back to nvidia-smi at
    its finest period when NVML cannot be loaded."""
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}
    SMI_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.rows = []  # (time, sm_mhz, max_mhz, power_w, set of reasons)
        self.t0 = self.t1 = None
        self.source = None
        self.stop_evt = threading.Event()
        self.proc = None
        self.th = None
        nv = self._nvml(device_index)
        if nv is not None:
            self.source = "nvml"
            self.th = threading.Thread(target=self._poll_nvml, args=(nv, period_s), daemon=True)
            self.th.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.source = "nvidia-smi"
        first = threading.Event()
        self.th = threading.Thread(target=self._read_smi, args=(first,), daemon=True)
        self.th.start()
        first.wait(timeout=10)

    @staticmethod
    def _nvml(device_index):
        """(library, handle) of this process's GPU, or None."""
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            ok = False
            try:
                import torch
                uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
                ok = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(h)) == 0
            if not ok:
                return None
            reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            return nv, h, reasons
        except (OSError, AttributeError):
            return None

    def _poll_nvml(self, nvh, period_s):
        nv, h, reasons = nvh
        sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_evt.is_set():
            t = time.time()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and \
                    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                power = pw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                bits = rs.value if reasons(h, ctypes.byref(rs)) == 0 else 0
                names = {n for n, b in self.REASON_BITS.items() if bits & b}
                self.rows.append((t, float(sm.value), float(mx.value), power, names))
            time.sleep(period_s)

    def _read_smi(self, first):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            first.set()
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                power = float(parts[3])
            except ValueError:
                power = None
            self.rows.append((time.time(), sm, mx, power,
                              {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()

    def close(self):
        self.stop_evt.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.th:
            self.th.join(timeout=5)

    def summary(self):
        if self.t0 is None or self.t1 is None:
            return {"samples": 0, "source": self.source}
        allrows = list(self.rows)
        rows = [r for r in allrows if self.t0 <= r[0] <= self.t1]
        window = "timed region"
        if not rows:  # a region shorter than the sampling period: the samples just around it
            before = [r for r in allrows if r[0] < self.t0][-1:]
            after = [r for r in allrows if r[0] > self.t1][:1]
            rows = before + after
            window = "samples just before and after the timed region (shorter than the period)"
        if not rows:
            return {"samples": 0, "source": self.source}
        reasons = set()
        for r in rows:
            reasons |= r[4]
        powers = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "source": self.source,
                "power_w_max": round(max(powers), 1) if powers else None,
                "window_s": round(self.t1 - self.t0, 4), "window": window}


# -------------------------------------------------------------- workloads --

def build_decode_step(workload, dev, bq, inputs, chain=False):
    """Resident Q4_0 weights of every matrix of the step, one fp32 input per
    distinct activation (in one contiguous buffer) and one output per matrix
    (in one contiguous buffer). Matrices reading the same activation (q/k/v,
    gate/up) form one batch.

    chain: every batch after the first reads an output of the batch before it
    (o reads q's output, gate/up read o's, down reads gate's, the next layer's
    q/k/v read down's), so each batch depends on the previous one through
    memory; the weights are then ~N(0, 1/K) so that the values stay in range
    along the chain, and x_all holds only the first batch's input."""
    import torch
    plan = inputs.decode_plan(workload)
    keys = []
    for e in plan:
        if e.x_key not in keys:
            keys.append(e.x_key)
    if chain:
        keys = keys[:1]
    x_len = {e.x_key: e.K for e in plan}
    x_off, off = {}, 0
    for k in keys:
        x_off[k] = off
        off += (x_len[k] + 3) // 4 * 4  # keep every x 16-byte aligned
    x_all = torch.empty(off, dtype=torch.float32, device=dev)
    for k in keys:
        e = next(e for e in plan if e.x_key == k)
        x_all[x_off[k]:x_off[k] + e.K].copy_(inputs.activation(e.K, e.x_seed, device=dev))
    y_off, off = [], 0
    for e in plan:
        y_off.append(off)
        off += (e.M + 3) // 4 * 4
    y_all = torch.empty(off, dtype=torch.float32, device=dev)
    mats = []
    for i, e in enumerate(plan):
        W = inputs.chain_weight(e.M, e.K, e.w_seed + 100000, device=dev) if chain else \
            inputs.weight(e.M, e.K, e.w_seed, device=dev)
        wq = bq.quantize_rows(bq.Q4_0, W)
        del W
        mats.append([wq, None, y_all[y_off[i]:y_off[i] + e.M], e.M, e.K])
    groups = []
    for m, e in zip(mats, plan):
        if groups and groups[-1]["key"] == e.x_key:
            g = groups[-1]
        else:
            if chain and groups:
                x = groups[-1]["y"][0][:e.K]
                assert x.numel() == e.K, "chain: an output of the previous batch is this batch's input"
            else:
                x = x_all[x_off[e.x_key]:x_off[e.x_key] + e.K]
            g = {"key": e.x_key, "x": x, "K": e.K, "w": [], "y": [], "M": []}
            groups.append(g)
        m[1] = g["x"]
        g["w"].append(m[0])
        g["y"].append(m[2])
        g["M"].append(m[3])
    torch.cuda.synchronize(dev)
    wbytes = sum(e.M * (e.K // 32) * 18 for e in plan)
    return {"plan": plan, "mats": [tuple(m) for m in mats], "groups": groups, "x_all": x_all, "y_all": y_all,
            "weight_bytes": wbytes, "chain": chain}


def seq_groups(step):
    """The step's batches in the form bq_gemv_sequence takes."""
    return [(g["w"], g["x"], g["M"], g["K"], g["y"]) for g in step["groups"]]


def run_step(step, bq, batched=True):
    """One decode token, one launch per batch: every matrix once, in layer
    order. batched: one launch per group of matrices sharing an input; else
    one per matrix."""
    if batched:
        for g in step["groups"]:
            bq.gemv_multi(bq.Q4_0, g["w"], g["x"], g["M"], g["K"], outs=g["y"])
    else:
        for wq, x, y, M, K in step["mats"]:
            bq.gemv(bq.Q4_0, wq, x, M, K, out=y)


def capture(fn, stream):
    import torch
    with torch.cuda.stream(stream):
        fn()  # uncaptured first call: kernel attributes, device info
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def capture_or_direct(fn, stream):
    """(callable replaying one step, how): a CUDA graph of fn when its launches
    can be captured, else fn itself issued on `stream` each step."""
    import torch
    try:
        g = capture(fn, stream)
        return g.replay, "cuda graph"
    except Exception as e:  # a launch kind the capture does not take
        torch.cuda.synchronize()
        return fn, f"direct calls ({type(e).__name__} in capture)"


def time_graph(g, stream, steps, warmup, dist=None, clocks=None, between=None):
    """Per-step device time (ms) of graph replays (see time_steps)."""
    return time_steps(g.replay, stream, steps, warmup, dist, clocks, between)


def time_steps(run, stream, steps, warmup, dist=None, clocks=None, between=None):
    """Per-step device time (ms): events on the launching stream around each
    step run(); `between` (e.g. an L2 flush) runs outside the timed spans."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
            if between:
                between()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    if between is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                run()
            e1.record(stream)
        e1.synchronize()
        total = e0.elapsed_time(e1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                a.record(stream)
                run()
                b.record(stream)
                between()
        torch.cuda.synchronize()
        total = sum(a.elapsed_time(b) for a, b in evs)
    if clocks:
        clocks.stop()
    torch.cuda.synchronize()
    barrier(dist)
    return total / steps


# ------------------------------------------------------------ CPU oracle ---

def oracle_layer0(workload="7b-decode"):
    """Layer 0 of the decode step for the oracle: (Q4_0 blocks, x, M, K) per matrix."""
    import oracle
    from block_quantized_weight_row_gb300 import inputs
    plan = [e for e in inputs.decode_plan(workload) if e.layer == 0]
    mats = []
    for e in plan:
        W = inputs.weight(e.M, e.K, e.w_seed).numpy()
        mats.append((oracle.quantize_rows(oracle.Q4_0, W), inputs.activation(e.K, e.x_seed).numpy(), e.M, e.K))
        del W
    return mats


def oracle_decode_sample(seconds: float, mats, label="single thread", workload="7b-decode"):
    """The oracle GEMV over layer 0 of the decode step, repeated until at
    least `seconds` of oracle time; returns (GB/s, description)."""
    import oracle
    done_bytes, spent, passes = 0, 0.0, 0
    while spent < seconds:
        for wq, x, M, K in mats:
            t = time.perf_counter()
            oracle.gemv(oracle.Q4_0, wq, x, M, K)
            spent += time.perf_counter() - t
            done_bytes += wq.nbytes
        passes += 1
    mb = sum(m[0].nbytes for m in mats) / 1e6
    return done_bytes / spent / 1e9, (f"oracle GEMV ({label}) over layer 0 of the {workload} step "
                                      f"({len(mats)} matrices, {mb:.1f} MB Q4_0), {passes} passes, {spent:.1f} s")


# ------------------------------------------------------------------ main ---

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--path", choices=("sequence", "per-launch"), default="sequence",
                    help="the whole step in one persistent launch, or one launch per batch")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-prefetch", action="store_true",
                    help="per-launch path: launch each GEMV only after the previous kernel completed")
    ap.add_argument("--no-batch", action="store_true",
                    help="per-launch path: one launch per matrix instead of one per batch sharing an input")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--kernel-case", choices=("gemv", "gemv-q8", "gemv-unaligned", "seq", "gemm", "kv", "attn"),
                    default=None,
                    help="run one kernel case a few times and exit (for profiler captures)")
    ap.add_argument("--case-launches", type=int, default=16)
    ap.add_argument("--probe", choices=("bulk", "rates"), default=None,
                    help="print a hardware probe's numbers and exit: bulk-copy read rate by copy size, or the "
                         "tensor-op and dp4a rates")
    args = ap.parse_args()
    if args.kernel_case:
        return kernel_case(args.kernel_case, args.case_launches)
    if args.probe:
        return hardware_probe(args.probe)
    if args.warmup < 3:
        args.warmup = 3

    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    import block_quantized_weight_row_gb300 as bq
    from block_quantized_weight_row_gb300 import binding, inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    clocks = ClockSampler(local) if rank == 0 else None

    # ---- headline: 7B decode step, every weight read once per token
    step = build_decode_step("7b-decode", dev, bq, inputs)
    binding.set_weight_prefetch(not args.no_prefetch)
    Lb = binding.lib()
    if args.path == "sequence":
        sargs = binding.gemv_sequence_args(seq_groups(step))
        run, how = capture_or_direct(lambda: binding.gemv_sequence_call(bq.Q4_0, sargs, dev), stream)
        launches_per_step = 1
        kernel = "k_gemv_seq<Q4_0>"
    else:
        batched = not args.no_batch
        run, how = capture_or_direct(lambda: run_step(step, bq, batched), stream)
        calls = [g["K"] for g in step["groups"]] if batched else [m[4] for m in step["mats"]]
        launches_per_step = sum(2 if Lb.bq_gemv_workspace_size(bq.Q4_0, K) > 0 else 1 for K in calls)
        kernel = "k_gemv_tma<Q4_0> (+ k_gemv_prep)"
    ms = time_steps(run, stream, args.steps, args.warmup, dist, clocks)
    ms_max = max_over_ranks(ms, dist)
    value = aggregate_rate(step["weight_bytes"], world, ms_max * 1e-3) / 1e9
    launches = launches_per_step * args.steps

    # ---- roofline of the dominant kernel
    if args.path == "sequence":
        # one launch is the whole step: weights, every x once, every y once
        x_bytes = sum(4 * g["K"] for g in step["groups"])
        y_bytes = sum(4 * M for g in step["groups"] for M in g["M"])
        alg_bytes = step["weight_bytes"] + x_bytes + y_bytes
        launch_ms = ms
        roofline = {"bound": "hbm", "kernel": "k_gemv_seq<Q4_0>, the whole 7B decode step in one launch",
                    "traffic": kernel_traffic("gemv_seq_q4_0_7b_step"),
                    "duration_note": "launch duration = step time on its stream (the step is this one "
                                     "launch after a counter reset of 1 KB)"}
    else:
        # the 11008 x 4096 launch alone, back to back on distinct matrices
        gate_up = [m for m, e in zip(step["mats"], step["plan"]) if e.name in ("gate", "up")]
        rg = capture(lambda: [bq.gemv(bq.Q4_0, wq, x, M, K, out=y) for wq, x, y, M, K in gate_up], stream)
        launch_ms = time_graph(rg, stream, 20, 3) / len(gate_up)
        M_, K_ = 11008, 4096
        alg_bytes = M_ * (K_ // 32) * 18 + K_ * 4 + M_ * 4
        roofline = {"bound": "hbm", "kernel": "k_gemv_tma<Q4_0> 11008x4096",
                    "traffic": kernel_traffic("gemv_q4_0_11008x4096")}
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    roofline.update({"achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                     "algorithmic_bytes_per_launch": alg_bytes, "avg_launch_us": round(launch_ms * 1e3, 3)})

    # ---- e2e: direct C-ABI calls, host buffers, copies inside the timed region
    e2e = e2e_decode(step, stream, dev, args, dist, world)

    secondary = {}
    if not args.no_secondary:
        secondary = secondary_rows(bq, binding, inputs, dev, stream, peaks, dist, world, step, args)

    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "q4_0xq8_0->f32",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
            "config": {"workload": "7b-decode: 32 layers x {q,k,v,o 4096x4096, gate/up 11008x4096, "
                                   "down 4096x11008}, batch 1, Q4_0 weights, 224 GEMVs per step",
                       "weight_bytes_per_step": step["weight_bytes"],
                       "l2": "inputs larger than L2 (3.64 GB of weights per step)",
                       "parallelism": f"replicas x{world}", "issue": how, "path": args.path,
                       "kernel": kernel, "launches_per_step": launches_per_step,
                       "inputs": "one fp32 x per distinct activation (q/k/v share one, gate/up share one); no "
                                 "batch reads another's output, so no batch waits (secondary.decode_chain "
                                 "times the step with every batch reading the previous batch's output)"},
            "hbm_frac_of_measured": round(value / world / peaks["hbm_gbs"], 4),
            "tokens_per_s_equiv": round(1e3 / ms_max, 1),
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks.summary() if clocks else None,
            "cpu_baseline": cpu, "secondary": secondary,
        }
        print(json.dumps(out))
    if clocks:
        clocks.close()
    if dist is not None:
        dist.destroy_process_group()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return None


def cpu_baseline(seconds):
    """The oracle's GEMV on this host: single-threaded, and the same source
    built with OpenMP over rows on every core this process may use."""
    mats = oracle_layer0()
    v1, desc1 = oracle_decode_sample(seconds, mats)
    cores = len(os.sched_getaffinity(0))
    out = {"value": round(v1, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc1,
           "cpu_model": cpu_model()}
    try:
        import oracle
        from oracle import build as obuild
        os.environ["OMP_NUM_THREADS"] = str(cores)
        with oracle.use_library(obuild.build_omp()):
            vn, descn = oracle_decode_sample(seconds, mats, f"OpenMP over rows, {cores} threads")
        out["all_cores"] = {"value": round(vn, 4), "unit": "GB/s", "cores": cores, "kind": "oracle (OpenMP rows)",
                            "sample": descn}
    except Exception as e:  # no OpenMP runtime on this host
        out["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"}
    return out


def e2e_decode(step, stream, dev, args, dist, world):
    """Per step: pinned host -> device copy of every activation, the whole step
    as one bq_gemv_sequence C-ABI call (argument arrays built once), device ->
    pinned host copy of every output, and a host wait."""
    import torch
    from block_quantized_weight_row_gb300 import binding
    L = binding.lib()
    x_host = step["x_all"].cpu().pin_memory()
    y_host = torch.empty(step["y_all"].numel(), dtype=torch.float32).pin_memory()
    sargs = binding.gemv_sequence_args(seq_groups(step))
    binding._workspace(dev, int(L.bq_gemv_sequence_workspace_size()))
    f = L.bq_gemv_sequence

    def one():
        step["x_all"].copy_(x_host, non_blocking=True)
        rc = f(2, *sargs)
        if rc:
            raise binding.BQError(rc, L.bq_last_error().decode())
        y_host.copy_(step["y_all"], non_blocking=True)
        stream.synchronize()

    n = max(3, min(args.steps, 200))
    with torch.cuda.stream(stream):
        assert L.bq_set_stream(ctypes.c_void_p(stream.cuda_stream)) == 0
        for _ in range(args.warmup):
            one()
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            one()
        e1.record(stream)
        e1.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(y_host, step["y_all"].cpu()), "the read-back must cover every output"
    ms = max_over_ranks(e0.elapsed_time(e1) / n, dist)
    return {"value": round(aggregate_rate(step["weight_bytes"], world, ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(step["x_all"].numel() * 4), "d2h_bytes_per_step": int(y_host.numel() * 4),
            "ms_per_step": round(ms, 4), "steps": n,
            "path": "per step: pinned H2D copy of the inputs, one bq_gemv_sequence C-ABI call, pinned D2H copy "
                    "of every output, host wait"}


def tensor_rates(dev):
    """Measured int8 (and, beside it, f16) tensor-op rates this GPU offers,
    the denominators of the prefill GEMM's fractions: mma.sync throughput from
    the probe library (register operands, 8 independent chains per warp, 4
    CTAs of 8 warps per SM, best of 3) and torch._int_mm (cuBLAS int8 GEMM,
    8192^3, best of 5 after 2 warm-ups). No clock or other setting is changed."""
    import torch
    from block_quantized_weight_row_gb300 import build as bbuild
    out = {}
    try:
        P = ctypes.CDLL(bbuild.PROBE_LIB)
        P.bq_probe_mma_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        P.bq_probe_mma_rate.restype = ctypes.c_int
        for kind, name in ((0, "mma_sync_s8_tops"), (1, "mma_sync_f16_tflops")):
            best = 0.0
            for _ in range(3):
                v = ctypes.c_double()
                if P.bq_probe_mma_rate(kind, 16384, 4, ctypes.byref(v)) == 0:
                    best = max(best, v.value)
            out[name] = round(best, 1)
    except OSError as e:
        out["probe"] = f"unavailable: {e}"
    try:
        n = 8192
        A = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
        B = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
        for _ in range(2):
            torch._int_mm(A, B)
        torch.cuda.synchronize()
        best = None
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._int_mm(A, B)
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out["torch_int_mm_tops"] = round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
        del A, B
    except Exception as e:  # no int8 GEMM in this torch build for this GPU
        out["torch_int_mm"] = f"unavailable: {type(e).__name__}: {str(e)[:120]}"
    i8 = [v for k, v in out.items() if k in ("mma_sync_s8_tops", "torch_int_mm_tops") and v]
    out["int8_tops_measured"] = max(i8) if i8 else None
    out["note"] = ("sm_103a has no int8 tcgen05.mma; the int8 tensor path is mma.sync s8 (and whatever cuBLAS "
                   "runs for torch._int_mm); int8_tops_measured is the larger of the two")
    torch.cuda.empty_cache()
    return out


def l2_flusher(dev):
    """Evict every line of L2 between timed steps: write a buffer twice the
    size of L2, then read another one (so that the write-backs of the flush's
    own dirty lines happen inside the flush, not inside the next timed step)."""
    import torch
    wbuf = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(64 * 2**20, dtype=torch.float32, device=dev)

    def flush():
        wbuf.fill_(1)
        rbuf.sum()
    return flush


def secondary_rows(bq, binding, inputs, dev, stream, peaks, dist, world, step, args):
    import torch
    out = {}
    flush = l2_flusher(dev)

    # the 7B step issued one launch per batch (the previous path), and the
    # step as a dependency chain on both paths
    def rate(st, ms_):
        return round(aggregate_rate(st["weight_bytes"], world, ms_ * 1e-3) / 1e9, 1)

    if args.path == "sequence":
        g = capture(lambda: run_step(step, bq, True), stream)
        ms = max_over_ranks(time_graph(g, stream, 50, 5), dist)
        out["decode_per_launch"] = {"metric": "Q4_0 decode GEMV weight GB/s, 7B step, one launch per batch "
                                              "(prep + GEMV kernel pairs with dependent launch, one CUDA graph)",
                                    "value": rate(step, ms), "unit": "GB/s", "ms_per_step": round(ms, 4),
                                    "launches_per_step": 2 * len(step["groups"])}
        del g
    chain = build_decode_step("7b-decode", dev, bq, inputs, chain=True)
    sargs = binding.gemv_sequence_args(seq_groups(chain))
    run, how = capture_or_direct(lambda: binding.gemv_sequence_call(bq.Q4_0, sargs, dev), stream)
    ms_seq = max_over_ranks(time_steps(run, stream, 50, 5), dist)
    g = capture(lambda: run_step(chain, bq, True), stream)
    ms_pl = max_over_ranks(time_graph(g, stream, 50, 5), dist)
    out["decode_chain"] = {"metric": "Q4_0 decode GEMV weight GB/s, 7B step as a chain: every batch reads the "
                                     "previous batch's output (o <- q, gate/up <- o, down <- gate, next q/k/v <- "
                                     "down), weights ~N(0, 1/K)",
                           "value": rate(chain, ms_seq), "unit": "GB/s", "ms_per_step": round(ms_seq, 4),
                           "issue": how, "waits_per_step": len(chain["groups"]) - 1,
                           "per_launch": {"value": rate(chain, ms_pl), "ms_per_step": round(ms_pl, 4)},
                           "hbm_frac_of_measured": round(chain["weight_bytes"] / (ms_seq * 1e-3) / 1e9 /
                                                         peaks["hbm_gbs"], 4)}
    del chain, g, run
    torch.cuda.empty_cache()

    # prefill GEMM, 512 tokens, Q8_0 weights
    rates = tensor_rates(dev)
    out["tensor_rates"] = rates
    cfg = inputs.WORKLOADS["prefill-q8_0"]
    N = cfg["tokens"]
    rows = []
    for i, (M, K) in enumerate(cfg["shapes"]):
        W = inputs.weight(M, K, inputs.seed_of("prefill-q8_0", 0, i), device=dev)
        wq = bq.quantize_rows(bq.Q8_0, W)
        del W
        X = inputs.activation(K, inputs.seed_of("prefill-q8_0", 1, i), device=dev, rows=N)
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
        g = capture(lambda: bq.gemm(bq.Q8_0, wq, X, M, N, K, out=Y), stream)
        ms = max_over_ranks(time_graph(g, stream, 20, 3, between=flush), dist)
        ops = 2.0 * N * M * K
        tops = ops / (ms * 1e-3) / 1e12
        rows.append({"M": M, "K": K, "N": N, "ms": round(ms, 4), "tops": round(tops, 1)})
    tot_ops = sum(2.0 * r["N"] * r["M"] * r["K"] for r in rows)
    tot_ms = sum(r["ms"] for r in rows)
    tops = tot_ops / (tot_ms * 1e-3) / 1e12 * world
    out["prefill_gemm"] = {"metric": "prefill GEMM int8-equivalent TOPS (2*N*M*K per GEMM, X quantize included)",
                           "value": round(tops, 1), "unit": "TOPS", "shapes": rows,
                           "tensor_frac_of_measured": round(tops / peaks["bf16_tflops"], 4),
                           "tensor_frac_of_int8_peak": (round(tops / rates["int8_tops_measured"], 4)
                                                        if rates.get("int8_tops_measured") else None),
                           "int8_peak_tops": rates.get("int8_tops_measured"),
                           "tensor_peak_note": "integer codes run as binary16 operands, so the peak is the measured "
                                               "dense bf16/f16 rate",
                           "kernel": "k_gemm_q8_tc (tcgen05.mma kind::f16, exact integer codes) + k_quantize_x_tc",
                           "l2": "flushed between iterations"}

    # KV-cache write: 28 layers x (K -> Q4_0 with bias, V -> Q8_0)
    kv = inputs.WORKLOADS["kv-write"]
    T, H, D = kv["tokens"], kv["kv_heads"], kv["head_dim"]
    layers = []
    for layer in range(kv["layers"]):
        Lr = inputs.kv_layer(layer, T, H, D, kv["calib_tokens"], device=dev)
        bias = Lr.K_calib.double().mean(dim=0).float().contiguous()
        kq = torch.empty((T, H, D // 32 * 18), dtype=torch.uint8, device=dev)
        vq = torch.empty((T, H, D // 32 * 34), dtype=torch.uint8, device=dev)
        layers.append((Lr.K, Lr.V, bias, kq, vq))
        del Lr

    def kv_step():  # one bq_kv_write launch per layer (K and V)
        for K_, V_, b, kq, vq in layers:
            bq.kv_write(bq.Q4_0, K_, b, bq.Q8_0, V_, out_k=kq, out_v=vq)

    def kv_step_per_tensor():  # one bq_kv_quantize launch per tensor
        for K_, V_, b, kq, vq in layers:
            bq.kv_quantize(bq.Q4_0, K_, b, out=kq)
            bq.kv_quantize(bq.Q8_0, V_, None, out=vq)
    g = capture(kv_step, stream)
    ms = max_over_ranks(time_graph(g, stream, 10, 3), dist)
    gp = capture(kv_step_per_tensor, stream)
    ms_pt = max_over_ranks(time_graph(gp, stream, 10, 3), dist)
    del gp
    kv_bytes = kv["layers"] * (2 * T * H * D * 4 + H * D * 4 + T * H * (D // 32) * (18 + 34))
    out["kv_write"] = {"metric": "KV-cache write GB/s (fp32 K,V read + Q4_0 K / Q8_0 V written)",
                       "value": round(aggregate_rate(kv_bytes, world, ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                       "ms_per_step": round(ms, 4), "bytes_per_step": kv_bytes,
                       "hbm_frac_of_measured": round(kv_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                       "kernel": "k_quantize_rows x 2 (bq_kv_write: V a programmatic dependent of K that does not wait)",
                       "per_tensor_calls": {"ms_per_step": round(ms_pt, 4),
                                            "value": round(aggregate_rate(kv_bytes, world, ms_pt * 1e-3) / 1e9, 1),
                                            "kernel": "k_quantize_rows, one bq_kv_quantize launch per tensor"},
                       "l2": "inputs larger than L2 (7.5 GB read per step)"}

    # decode attention of one token over every layer's quantized cache: the
    # caches the KV write above produced (mean-centered Q4_0 K, Q8_0 V), 16
    # query heads over 8 kv heads
    HQ = 2 * H
    qs = [inputs.activation(D, inputs.seed_of("kv-write", layer, 9), device=dev, rows=HQ)
          for layer in range(kv["layers"])]
    outs = [torch.empty((HQ, D), dtype=torch.float32, device=dev) for _ in qs]
    scale = 1.0 / (D ** 0.5)

    def attn_step():
        for (_K, _V, _b, kq, vq), qv, ov in zip(layers, qs, outs):
            bq.attn_decode(bq.Q4_0, bq.Q8_0, qv, kq, vq, H, scale, out=ov)
    g2 = capture(attn_step, stream)
    ms2 = max_over_ranks(time_graph(g2, stream, 20, 3), dist)
    cache_bytes = kv["layers"] * T * H * (D // 32) * (18 + 34)
    out["attn_decode"] = {"metric": "decode attention GB/s of quantized KV cache read (one token, every layer)",
                          "value": round(aggregate_rate(cache_bytes, world, ms2 * 1e-3) / 1e9, 1), "unit": "GB/s",
                          "ms_per_step": round(ms2, 4), "bytes_per_step": cache_bytes,
                          "hbm_frac_of_measured": round(cache_bytes / (ms2 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                          "config": f"{kv['layers']} layers x {T} tokens x {H} kv heads x {D}, {HQ} query heads, "
                                    "Q4_0 K (mean-centered) + Q8_0 V",
                          "kernel": "k_attn_warp + k_attn_combine",
                          "l2": "inputs larger than L2 (1.5 GB of cache per step)"}
    # the same write and attention with K Hadamard-rotated per 64 channels and
    # the bias calibrated in the rotated basis (bq_kv_bias)
    for i, (K_, V_, b, kq, vq) in enumerate(layers):
        layers[i] = (K_, V_, bq.kv_bias(inputs.kv_layer(i, 1, H, D, kv["calib_tokens"], device=dev).K_calib,
                                        bq.BASIS_HADAMARD64), kq, vq)

    def kv_step_rot():
        for K_, V_, b, kq, vq in layers:
            bq.kv_write(bq.Q4_0, K_, b, bq.Q8_0, V_, out_k=kq, out_v=vq, basis=bq.BASIS_HADAMARD64)
    g3 = capture(kv_step_rot, stream)
    ms3 = max_over_ranks(time_graph(g3, stream, 10, 3), dist)
    out["kv_write_rotated"] = {"metric": "KV-cache write GB/s, K Hadamard-rotated per 64 channels",
                               "value": round(aggregate_rate(kv_bytes, world, ms3 * 1e-3) / 1e9, 1), "unit": "GB/s",
                               "ms_per_step": round(ms3, 4), "bytes_per_step": kv_bytes,
                               "hbm_frac_of_measured": round(kv_bytes / (ms3 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                               "kernel": "k_quantize_rows x 2 (bq_kv_write, K in the rotated basis)",
                               "l2": "inputs larger than L2 (7.5 GB read per step)"}

    def attn_step_rot():
        for (_K, _V, _b, kq, vq), qv, ov in zip(layers, qs, outs):
            bq.attn_decode(bq.Q4_0, bq.Q8_0, qv, kq, vq, H, scale, out=ov, k_basis=bq.BASIS_HADAMARD64)
    g4 = capture(attn_step_rot, stream)
    ms4 = max_over_ranks(time_graph(g4, stream, 20, 3), dist)
    out["attn_decode_rotated"] = {"metric": "decode attention GB/s over the rotated K cache (q rotated alike)",
                                  "value": round(aggregate_rate(cache_bytes, world, ms4 * 1e-3) / 1e9, 1),
                                  "unit": "GB/s", "ms_per_step": round(ms4, 4), "bytes_per_step": cache_bytes,
                                  "hbm_frac_of_measured": round(cache_bytes / (ms4 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                  "l2": "inputs larger than L2 (1.5 GB of cache per step)"}
    del layers, g, g2, g3, g4, qs, outs
    torch.cuda.empty_cache()

    # legacy weight types: GEMV on 11008 x 4096 matrices, 8 distinct matrices
    # per type (beyond L2) launched back to back in one graph
    M_, K_ = 11008, 4096
    x_ = inputs.activation(K_, inputs.seed_of("legacy-gemv", 0, 0), device=dev)
    y_ = torch.empty(M_, dtype=torch.float32, device=dev)
    leg = {}
    for name, t in (("Q4_0", bq.Q4_0), ("Q4_1", bq.Q4_1), ("Q5_0", bq.Q5_0), ("Q5_1", bq.Q5_1),
                    ("Q4_K", bq.Q4_K), ("Q6_K", bq.Q6_K)):
        mats = [bq.quantize_rows(t, inputs.weight(M_, K_, inputs.seed_of("legacy-gemv", 1, i), device=dev))
                for i in range(8)]

        def leg_step():
            for w in mats:
                bq.gemv(t, w, x_, M_, K_, out=y_)
        gl = capture(leg_step, stream)
        msl = max_over_ranks(time_graph(gl, stream, 20, 3), dist)
        byts = 8 * mats[0].numel()
        leg[name] = {"GB/s": round(aggregate_rate(byts, world, msl * 1e-3) / 1e9, 1),
                     "us_per_launch": round(msl * 1e3 / 8, 2),
                     "hbm_frac_of_measured": round(byts / (msl * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        del mats, gl
    out["gemv_legacy_types"] = {"metric": "decode GEMV GB/s of weights per type (11008 x 4096, back to back)",
                                "value": leg["Q5_0"]["GB/s"], "unit": "GB/s", "per_type": leg,
                                "kernel": "k_gemv_tma (+ k_gemv_prep) for every type (Q6_K: K % 2048 == 0); "
                                          "Q4_0 for comparison",
                                "l2": "8 distinct matrices per type, 203-370 MB: beyond L2"}
    torch.cuda.empty_cache()

    # shapes whose rows are not whole multiples of 16 bytes: Q6_K down-projection
    # rows (K = 11008: bulk copies of whole 8-row quanta) and Q4_0 / Q8_0 and
    # the legacy types with K = 4128, not a multiple of 256 (rows staged in
    # shared memory, x quantized once into the workspace)
    gen = {}
    for name, t, M_, K_ in (("Q6_K_4096x11008", bq.Q6_K, 4096, 11008), ("Q4_0_11008x4128", bq.Q4_0, 11008, 4128),
                            ("Q8_0_11008x4128", bq.Q8_0, 11008, 4128), ("Q4_1_11008x4128", bq.Q4_1, 11008, 4128),
                            ("Q5_0_11008x4128", bq.Q5_0, 11008, 4128), ("Q5_1_11008x4128", bq.Q5_1, 11008, 4128)):
        x_ = inputs.activation(K_, inputs.seed_of("legacy-gemv", 2, 0), device=dev)
        y_ = torch.empty(M_, dtype=torch.float32, device=dev)
        mats = [bq.quantize_rows(t, inputs.weight(M_, K_, inputs.seed_of("legacy-gemv", 3, i), device=dev))
                for i in range(8)]

        def gen_step():
            for w in mats:
                bq.gemv(t, w, x_, M_, K_, out=y_)
        gg = capture(gen_step, stream)
        msg = max_over_ranks(time_graph(gg, stream, 20, 3), dist)
        byts = 8 * mats[0].numel()
        gen[name] = {"GB/s": round(aggregate_rate(byts, world, msg * 1e-3) / 1e9, 1),
                     "us_per_launch": round(msg * 1e3 / 8, 2),
                     "hbm_frac_of_measured": round(byts / (msg * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        del mats, gg
    out["gemv_unaligned_rows"] = {"metric": "decode GEMV GB/s of weights, rows not multiples of 16 bytes (back to back)",
                                "value": gen["Q6_K_4096x11008"]["GB/s"], "unit": "GB/s", "per_shape": gen,
                                "kernel": "Q6_K: k_gemv_tma in 8-row quanta (+ k_gemv_prep); K % 256 != 0: "
                                          "k_gemv_generic_prep + k_gemv_staged (rows staged in shared memory by "
                                          "async copies, a dependent launch of the prep)",
                                "l2": "8 distinct matrices per shape, 204-384 MB: beyond L2"}
    torch.cuda.empty_cache()

    # Qwen3-0.6B-shaped decode step (247.7 MB of Q4_0), L2 flushed between steps
    q = build_decode_step("qwen3-0.6b-decode", dev, bq, inputs)
    qargs = binding.gemv_sequence_args(seq_groups(q))
    run, how = capture_or_direct(lambda: binding.gemv_sequence_call(bq.Q4_0, qargs, dev), stream)
    ms = max_over_ranks(time_steps(run, stream, 50, 5, between=flush), dist)
    g = capture(lambda: run_step(q, bq, True), stream)
    ms_pl = max_over_ranks(time_graph(g, stream, 50, 5, between=flush), dist)
    out["qwen3_0_6b_decode"] = {"metric": "Q4_0 decode GEMV weight GB/s", "unit": "GB/s",
                                "value": round(aggregate_rate(q["weight_bytes"], world, ms * 1e-3) / 1e9, 1),
                                "ms_per_step": round(ms, 4), "weight_bytes_per_step": q["weight_bytes"],
                                "gemvs_per_step": len(q["mats"]), "launches_per_step": 1, "issue": how,
                                "path": "bq_gemv_sequence (one persistent launch)",
                                "per_launch": {"value": round(aggregate_rate(q["weight_bytes"], world,
                                                                             ms_pl * 1e-3) / 1e9, 1),
                                               "ms_per_step": round(ms_pl, 4),
                                               "launches_per_step": 2 * len(q["groups"])},
                                "hbm_frac_of_measured": round(q["weight_bytes"] / (ms * 1e-3) / 1e9 /
                                                              peaks["hbm_gbs"], 4),
                                "l2": "flushed between steps"}
    return out


def hardware_probe(name):
    """Probe numbers behind design choices (libbq_probe.so), one JSON line."""
    import torch
    from block_quantized_weight_row_gb300 import build as bbuild
    torch.cuda.set_device(0)
    torch.zeros(1, device="cuda")
    P = ctypes.CDLL(bbuild.PROBE_LIB)
    dbl = ctypes.POINTER(ctypes.c_double)
    out = {"probe": name}
    if name == "bulk":
        P.bq_probe_bulk_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_size_t, dbl]
        rates = {}
        for sz in (4096, 8192, 12288, 16384, 24576, 32768, 49152, 98304):
            for depth in (1, 2, 4, 8):
                if sz * depth > 200 * 1024:
                    continue
                v = ctypes.c_double()
                rc = P.bq_probe_bulk_rate(sz, depth, 4 << 30, ctypes.byref(v))
                rates[f"{sz}x{depth}"] = round(v.value, 1) if rc == 0 else f"rc {rc}"
        out.update({"unit": "GB/s read", "key": "copy bytes x copies in flight per SM", "rates": rates})
    else:
        P.bq_probe_int_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dbl]
        P.bq_probe_mma_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dbl]
        for kind, key, f in ((2, "dp4a_tera_lane_ops", P.bq_probe_int_rate), (3, "imad_tera_lane_ops", P.bq_probe_int_rate),
                             (0, "mma_sync_s8_tops", P.bq_probe_mma_rate), (1, "mma_sync_f16_tflops", P.bq_probe_mma_rate)):
            v = ctypes.c_double()
            rc = f(kind, 16384 if kind < 2 else 20000, 4, ctypes.byref(v))
            out[key] = round(v.value, 2) if rc == 0 else f"rc {rc}"
    print(json.dumps(out))


def kernel_case(name, launches):
    """A small, self-contained case of one kernel for profiler captures:
    inputs larger than L2 (rotated over distinct buffers) but well under a
    few GB on the device."""
    import torch
    import block_quantized_weight_row_gb300 as bq
    from block_quantized_weight_row_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if name in ("gemv", "gemv-q8", "gemv-unaligned"):
        t = bq.Q8_0 if name == "gemv-q8" else bq.Q4_0
        M, K = 11008, 4128 if name == "gemv-unaligned" else 4096
        mats = []
        for i in range(8):  # 8 x 25.4 MB (Q4_0) or 48 MB (Q8_0): beyond L2
            mats.append(bq.quantize_rows(t, inputs.weight(M, K, 7000 + i, device=dev)))
        x = inputs.activation(K, 7100, device=dev)
        y = torch.empty(M, device=dev)
        for i in range(launches):
            bq.gemv(t, mats[i % len(mats)], x, M, K, out=y)
    elif name == "seq":
        from block_quantized_weight_row_gb300 import binding
        # the first 4 layers of the 7B step (455 MB of weights: beyond L2) in
        # one bq_gemv_sequence launch, on two copies of the weights in turn
        plan = [e for e in inputs.decode_plan("7b-decode") if e.layer < 4]
        steps, keep = [], []  # keep: the tensors the argument arrays point to
        for c in range(2):
            groups, cur = [], None
            for e in plan:
                if cur is None or cur[5] != e.x_key:
                    cur = ([], inputs.activation(e.K, e.x_seed + c, device=dev), [], e.K, [], e.x_key)
                    groups.append(cur)
                cur[0].append(bq.quantize_rows(bq.Q4_0, inputs.weight(e.M, e.K, e.w_seed + 7 * c, device=dev)))
                cur[2].append(e.M)
                cur[4].append(torch.empty(e.M, device=dev))
            keep.append(groups)
            steps.append(binding.gemv_sequence_args([g[:5] for g in groups]))
        for i in range(launches):
            binding.gemv_sequence_call(bq.Q4_0, steps[i % 2], dev)
    elif name == "gemm":
        M, N, K = 4096, 512, 4096
        wq = bq.quantize_rows(bq.Q8_0, inputs.weight(M, K, 7200, device=dev))
        X = inputs.activation(K, 7201, device=dev, rows=N)
        Y = torch.empty((N, M), device=dev)
        for _ in range(launches):
            bq.gemm(bq.Q8_0, wq, X, M, N, K, out=Y)
    elif name == "kv":
        kv = inputs.WORKLOADS["kv-write"]
        L_ = inputs.kv_layer(0, kv["tokens"], kv["kv_heads"], kv["head_dim"], kv["calib_tokens"], device=dev)
        bias = L_.K_calib.double().mean(dim=0).float().contiguous()
        kq, vq = bq.kv_write(bq.Q4_0, L_.K, bias, bq.Q8_0, L_.V)
        for _ in range(launches):
            bq.kv_write(bq.Q4_0, L_.K, bias, bq.Q8_0, L_.V, out_k=kq, out_v=vq)
    elif name == "attn":
        kv = inputs.WORKLOADS["kv-write"]
        T, H, D = kv["tokens"], kv["kv_heads"], kv["head_dim"]
        caches = []
        for layer in range(4):  # 4 x 54.5 MB of cache: beyond L2
            L_ = inputs.kv_layer(layer, T, H, D, kv["calib_tokens"], device=dev)
            caches.append((bq.kv_quantize(bq.Q4_0, L_.K, None), bq.kv_quantize(bq.Q8_0, L_.V, None)))
            del L_
        q = inputs.activation(D, 7300, device=dev, rows=2 * H)
        o = torch.empty((2 * H, D), device=dev)
        for i in range(launches):
            kq, vq = caches[i % len(caches)]
            bq.attn_decode(bq.Q4_0, bq.Q8_0, q, kq, vq, H, 1.0 / D ** 0.5, out=o)
    torch.cuda.synchronize()
    print(json.dumps({"kernel_case": name, "launches": launches, "ok": True}))


def reference_arm(args, world, rank):
    """The CPU oracle as the reference arm, on the host cores: each step is
    the oracle GEMV over a fixed slice of rows of every matrix of layer 0 of
    the 7B decode step, the slice sized so that warm-up plus timed steps take
    about a minute of oracle time."""
    if world > 1 and rank != 0:
        return
    import oracle
    from block_quantized_weight_row_gb300 import inputs
    plan = [e for e in inputs.decode_plan("7b-decode") if e.layer == 0]
    mats = []
    for e in plan:
        W = inputs.weight(e.M, e.K, e.w_seed).numpy()
        mats.append((oracle.quantize_rows(oracle.Q4_0, W), inputs.activation(e.K, e.x_seed).numpy(), e.M, e.K))
        del W
    # calibrate: oracle seconds per weight byte on one full matrix
    wq, x, M, K = mats[0]
    t = time.perf_counter()
    oracle.gemv(oracle.Q4_0, wq, x, M, K)
    s_per_byte = (time.perf_counter() - t) / wq.nbytes
    layer_bytes = sum(m[0].nbytes for m in mats)
    budget = 60.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, budget / (s_per_byte * layer_bytes))
    sample = [(wq[:max(1, int(M * frac))], x, max(1, int(M * frac)), K) for wq, x, M, K in mats]
    step_bytes = sum(m[0].nbytes for m in sample)

    def one():
        for wq_, x_, M_, K_ in sample:
            oracle.gemv(oracle.Q4_0, wq_, x_, M_, K_)

    for _ in range(args.warmup):
        one()
    t = time.perf_counter()
    for _ in range(args.steps):
        one()
    spent = time.perf_counter() - t
    ms = spent / args.steps * 1e3
    value = step_bytes / (ms * 1e-3) / 1e9
    desc = (f"oracle GEMV (single thread) per step over the first {frac:.2%} of the rows of each of the "
            f"7 matrices of layer 0 of the 7b-decode step ({step_bytes / 1e6:.2f} MB Q4_0 per step)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "q4_0xq8_0->f64", "data": "synthetic",
        "config": {"workload": "7b-decode (layer-0 row sample per step), oracle on host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    main()
