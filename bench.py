#!/usr/bin/env python
"""Benchmark of the mixed-batch multi-adapter LoRA layer: one forward + backward step per iteration.

Default workload (the large heterogeneous co-serving batch): Llama-70B-like MLP projection K=8192 -> N=28672, bf16,
an adapter pool of 320 adapters with ranks drawn from {8,16,32,64,128}, a batch of 2048 decode tokens (one per
segment, Zipf(1.1) adapter popularity) + 4096 prefill tokens (segments of 64..1024) + 2048 fine-tuning tokens
(2 segments on one adapter).  A step is the forward over all 8192 tokens followed by the LoRA backward of the 2048
fine-tuning tokens (xA recomputed), i.e. every step of the layer's hot path.

Prints one JSON line (rank 0).  `value` is forward tokens per second over all ranks, timed with CUDA events on the
launching stream after warm-up; the step's inputs (W 470 MB, the adapter pool, x, dY) exceed the 129 MB L2, so L2 is
not flushed.  `--impl reference` times the float64 CPU oracle on a bounded sample of the same workload instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "mixed-batch multi-LoRA fwd+bwd tokens/s; TFLOP/s and HBM GB/s vs GB300 peak"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, choices=[2, 3, 4, 5])
    ap.add_argument("--workload", choices=["config", "layer", "sweep", "gemm"], default="config",
                    help="layer: the LoRA projections of one Llama-3-8B decoder layer (q|k|v, o, gate|up, down) "
                         "on a co-serving batch, chained on one stream; sweep: that layer step over a grid of batch "
                         "compositions, with the step-latency model (Eq. I / II) fitted to the timings; gemm: the "
                         "main pass alone (one base-only segment) beside cuBLAS (torch.matmul) on the shape "
                         "--set M=.. --set K=.. --set N=.. (default 4096 x 4096 x 4864)")
    ap.add_argument("--out", default=None, help="sweep: also write the fitted coefficients to this JSON file")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' summaries (20 timed steps each) in the headline line")
    ap.add_argument("--selftest-ranks", action="store_true",
                    help="start the ranks as --gpus asks and only check that they meet (gloo, no GPU)")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=VALUE",
                    help="override a workload parameter (e.g. N=4096) for profiling a reduced case")
    return ap.parse_args()


# ----------------------------------------------------------------------------------------------- workload accounting
def make_workload(cfg, rank=0, overrides=()):
    seed = 1000 + cfg + 7919 * rank      # each rank draws its own batch (weak scaling)
    kw = {}
    for item in overrides:
        k, v = item.split("=", 1)
        kw[k] = int(v)
    return workloads.config(cfg, seed=seed, **kw)


def accounting(wl):
    """Algorithmic FLOPs and bytes of one step, split by launch group (no padding, no redundant work)."""
    T, K, N = wl.T, wl.K, wl.N
    S = wl.n_slices                      # a sliced layer: S down factors per adapter, one up factor over N
    segs = wl.segs.tolist()
    r_of = lambda a: int(wl.rank[a]) if a >= 0 else 0
    fwd = wl.forward
    bwd = wl.backward
    out = {}
    if fwd:
        shrink = sum(2 * ln * S * K * r_of(a) for _, ln, a, _ in segs)
        expand = sum(2 * ln * N * r_of(a) for _, ln, a, _ in segs)
        out["fwd_main_flops"] = 2 * T * K * N + expand
        out["fwd_flops"] = 2 * T * K * N + expand + shrink
        used = sorted(set(a for _, ln, a, _ in segs if a >= 0 and ln > 0))
        save = sum(ln * S * r_of(a) for _, ln, a, tr in segs if tr) * 2 if wl.xa_mode == "save" else 0
        out["fwd_bytes"] = 2 * (T * K + K * N + T * N) + sum(2 * r_of(a) * (S * K + N) for a in used) + save
        # main launch: x, W, adapters' B blocks and y
        out["fwd_main_bytes"] = 2 * (T * K + K * N + T * N) + sum(2 * r_of(a) * N for a in used)
    if bwd:
        tr = [(st, ln, a) for st, ln, a, t in segs if t and ln > 0]
        Tt = sum(ln for _, ln, _ in tr)
        lora = sum(2 * ln * r_of(a) * (2 * S * K + 2 * N) for _, ln, a in tr)
        recompute = sum(2 * ln * S * K * r_of(a) for _, ln, a in tr) if wl.xa_mode != "save" else 0
        out["bwd_flops"] = 2 * Tt * K * N + lora + recompute
        # the backward main pass: dX (dense + its LoRA K-steps) and dA, dB (the backward shrink dY B^T and the x A
        # recompute run before it)
        out["bwd_main_flops"] = 2 * Tt * K * N + sum(2 * ln * r_of(a) * (2 * S * K + N) for _, ln, a in tr)
        tads = sorted(set(a for _, _, a in tr))
        out["bwd_bytes"] = 2 * (Tt * N + K * N + 2 * Tt * K) + sum(6 * r_of(a) * (S * K + N) for a in tads)
        out["train_tokens"] = Tt
    out["flops"] = out.get("fwd_flops", 0) + out.get("bwd_flops", 0)
    out["bytes"] = out.get("fwd_bytes", 0) + out.get("bwd_bytes", 0)
    out["tokens"] = T if fwd else out.get("train_tokens", 0)
    return out


def launches_per_step(wl, fwd_info=None):
    """Kernel launches of one step.  fwd_info: the forward tile plan (info rows of lora_plan_describe: gathered,
    adapters, LoRA columns, x row).  Gathered decode tiles of up to 1024 rows are shrunk on CUDA cores (one launch,
    which also gathers the rows) and leave the tensor-core shrink; a main pass with fewer output tiles than kMainTargetItems (96) is split and
    adds a reduce launch."""
    segs = wl.segs.tolist()
    n_nt = lambda cols: -(-cols // 256)
    n = 0
    if wl.forward:
        info = np.asarray(fwd_info) if fwd_info is not None else np.zeros((0, 4), np.int64)
        n_g = int(info[:, 0].sum()) if len(info) else 0
        bgmv = 0 < n_g * 128 <= 1024
        n += 1 if bgmv else (1 if n_g > 0 else 0)            # CUDA-core shrink (gathers the rows) or row gather
        tc_shrink = [(g, ext) for g, _, ext, _ in info.tolist() if ext > 0 and not (g and bgmv)]
        n += 1 if tc_shrink else 0                                                          # tensor-core shrink
        n += 1                                                                              # main pass
        if 0 < (len(info) // 2) * n_nt(wl.N) < 96:
            n += 1                                                                          # split reduce
    if wl.backward and any(tr for *_, tr in segs):
        n += 3                                                                              # shrink, dX, dA/dB
        pairs = sum(-(-ln // 256) for _, ln, _, tr in segs if tr and ln > 0)
        tiles, nk = pairs * n_nt(wl.K), -(-wl.N // 64)
        if (tiles < 96 and nk // 4 >= 2) or (tiles >= 96 and 0 < tiles % 76 <= 38 and nk // 4 >= 2):
            n += 1                                                                          # split reduce
    return n


L2_NOMINAL = 129 * 2 ** 20          # GB300 L2 size used for the flush decision (both arms decide alike)


def input_bytes(wl):
    """Bytes of the step's inputs (x, W, adapter pool, dY) in the layer's element type."""
    es = 2 if wl.dtype == "bf16" else 4
    return es * sum(int(a.size) for a in (wl.x, wl.Wt, wl.A, wl.B, wl.dY) if a is not None)


def needs_flush(in_bytes):
    """Inputs not well above the L2 size would largely stay resident from one step to the next: flush unless they
    exceed twice the L2 size."""
    return in_bytes <= 2 * L2_NOMINAL


def l2_note(in_bytes):
    if needs_flush(in_bytes):
        return ("inputs (x, W, adapter pool, dY: %.0f MB) within twice the L2 size: L2 flushed before every step "
                "by a write of twice its size, outside the step's events" % (in_bytes / 1e6))
    return "inputs larger than twice the L2 size (x, W, adapter pool, dY: %.0f MB); no flush" % (in_bytes / 1e6)


def config_dict(wl, acc, world):
    """The `config` object of a line (identical in both arms for one workload)."""
    return {"workload": wl.name, "T": wl.T, "K": wl.K, "N": wl.N, "adapters": wl.n_adapters,
            "train_tokens": acc.get("train_tokens", 0), "xa": wl.xa_mode, "l2": l2_note(input_bytes(wl)),
            "parallelism": "replicas" if world == 1 else "dp%d (independent batches)" % world}


def layer_config_dict(L, acc, world):
    q = L["qkv"]
    return {"workload": layer_name(L), "T": q.T, "hidden": q.K, "kv": (q.N - q.K) // 2,
            "intermediate": L["down"].K, "adapters": q.n_adapters,
            "train_tokens": acc["qkv"].get("train_tokens", 0), "xa": "recompute",
            "projections": "q|k|v (3 slices), o, gate|up (2 slices), down",
            "l2": "inputs larger than L2 (weights %.0f MB); no flush"
                  % (sum(2 * L[n].K * L[n].N for n in LAYER_ORDER) / 1e6),
            "parallelism": "replicas" if world == 1 else "dp%d (independent batches)" % world}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_hash():
    h = hashlib.sha256()
    for f in ("tc_kernel.cu", "tc_kernel.h", "common.h"):
        h.update(open(os.path.join(ROOT, "lora_co_serving_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(cfg):
    """DRAM bytes per launch of the forward main pass from a committed ncu summary, if it matches this kernel."""
    p = os.path.join(ROOT, "profiles", "fwd_main_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_sha") != kernel_hash() or d.get("config") != cfg:
        return None
    return d.get("bytes_per_launch")


# ----------------------------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self, t0=None, t1=None):
        """Summary of the samples taken between host times t0 and t1 (the timed region)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if t0 is not None:
            import datetime
            keep = []
            for r in rows:
                try:
                    ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if t0 - 0.05 <= ts <= t1 + 0.05:
                    keep.append(r)
            rows = keep
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max([float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()] or [0])}


class NvmlSampler:
    """Clock, power and clock-event samples every ~2 ms from the driver's NVML library (read-only queries), so that
    a timed region of tens of milliseconds still gets tens of samples; falls back to nvidia-smi when NVML is
    unavailable."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.samples = []
        self.fallback = None
        self.thread = None
        self.stop_flag = False
        try:
            import ctypes
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))        # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self.reasons_fn = None
            for name in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
                try:
                    self.reasons_fn = getattr(self.nv, name)
                    break
                except AttributeError:
                    pass
        except (OSError, AttributeError):
            self.nv = None
            self.fallback = ClockSampler(gpu_index)

    def _poll(self):
        import ctypes
        mhz, reasons, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self.stop_flag:
            t = time.time()
            ok = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0
            if self.reasons_fn is not None:
                self.reasons_fn(self.h, ctypes.byref(reasons))
            self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw))
            if ok:
                self.samples.append((t, float(mhz.value), int(reasons.value), mw.value / 1e3))
            time.sleep(0.002)

    def start(self):
        if self.fallback is not None:
            return self.fallback.start()
        import threading
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        time.sleep(0.01)

    def stop(self, t0=None, t1=None):
        if self.fallback is not None:
            return self.fallback.stop(t0, t1)
        self.stop_flag = True
        self.thread.join()
        rows = [r for r in self.samples if t0 is None or t0 <= r[0] <= t1]
        reasons = sorted(set(name for r in rows for bit, name in self.REASONS.items() if r[2] & bit))
        return {"sm_mhz": statistics.median(r[1] for r in rows) if rows else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(rows), "source": "NVML, every ~2 ms",
                "power_w_max": max((r[3] for r in rows), default=0.0)}


# ----------------------------------------------------------------------------------------------- CPU oracle sample
def pk_clock_mhz():
    """SM clock (MHz) used to turn a pause into spin-kernel cycles: the device's maximum (a lower clock only
    lengthens the pause)."""
    import torch
    rate = getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "clock_rate", 0)
    return rate / 1e3 if rate else 2070.0


def oracle_threads():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def sample_size():
    """The oracle sample of one step, the same in the reference arm and the cpu_baseline leg: at least one forward
    row per host thread (so that every thread has work), 16 dX rows, 32 + 32 gradient columns."""
    return {"fwd_rows": max(32, oracle_threads()), "dx_rows": 16, "cols": 32}


def oracle_sample(wl, fwd_rows=32, dx_rows=16, cols=32, seed=0):
    """Time the float64 oracle on a bounded, stratified sample of one step and extrapolate to the full step.

    Returns (seconds per full step, description, threads, seconds the sample took)."""
    import oracle
    t_start = time.perf_counter()
    rng = np.random.default_rng(seed)
    T, K, N = wl.T, wl.K, wl.N
    t_total = 0.0
    desc = []
    if wl.forward:
        segs = sorted(wl.segs.tolist())
        kinds = {"decode": [], "prefill": [], "train": []}
        for st, ln, a, tr in segs:
            kinds["train" if tr else ("decode" if ln < 16 else "prefill")].append((st, ln))
        rows = []
        per = max(1, fwd_rows // max(1, sum(1 for v in kinds.values() if v)))
        for v in kinds.values():
            if v:
                for i in rng.integers(0, len(v), per):
                    st, ln = v[i]
                    rows.append(st + int(rng.integers(0, ln)))
        rows = np.array(rows[:fwd_rows])
        t0 = time.perf_counter()
        oracle.forward_wl(wl, rows=rows)
        dt = time.perf_counter() - t0
        t_total += dt * T / rows.shape[0]
        desc.append("%d forward rows (stratified over decode/prefill/fine-tuning) x %d/%d" % (rows.shape[0], T,
                                                                                               rows.shape[0]))
    if wl.backward:
        trows = wl.train_rows()
        pick = trows[rng.integers(0, trows.shape[0], dx_rows)]
        t0 = time.perf_counter()
        oracle.backward_wl(wl, dx_rows=pick, want_grads=False)
        dt = time.perf_counter() - t0
        t_total += dt * trows.shape[0] / dx_rows
        cb1, ca1 = np.array([0]), np.array([0])
        t0 = time.perf_counter()
        oracle.backward_wl(wl, want_dx=False, cols_b=cb1, cols_a=ca1)
        t1 = time.perf_counter() - t0
        cb = rng.choice(N, cols, replace=False)
        ca = rng.choice(K, cols, replace=False)
        t0 = time.perf_counter()
        oracle.backward_wl(wl, want_dx=False, cols_b=cb, cols_a=ca)
        tc = time.perf_counter() - t0
        per_col = max(0.0, (tc - t1) / (2 * (cols - 1)))
        t_total += t1 + per_col * (N + K)
        desc.append("%d dX rows x %d/%d; dA/dB: shrink of all fine-tuning rows + %d+%d gradient columns "
                    "extrapolated to %d+%d" % (dx_rows, trows.shape[0], dx_rows, cols, cols, K, N))
    return (t_total, "; ".join(desc) + "; linear extrapolation to one full step", oracle_threads(),
            time.perf_counter() - t_start)


LAYER_ORDER = ["qkv", "o", "gate_up", "down"]


def make_layer(rank=0, overrides=()):
    kw = {}
    for item in overrides:
        k, v = item.split("=", 1)
        kw[k] = int(v)
    return workloads.llama_layer(seed=1006 + 7919 * rank, **kw)


def layer_oracle_sample(L, seed=0, fwd_rows=8, dx_rows=4, cols=8):
    """The oracle on a bounded sample of one layer step: every projection, a sliced one slice by slice (each slice
    is a plain LoRA layer on the shared input)."""
    t = spent = 0.0
    desc = threads = None
    for n in LAYER_ORDER:
        wl = L[n]
        parts = [workloads.slice_of(wl, i) for i in range(wl.n_slices)] if wl.bounds is not None else [wl]
        for part in parts:
            dt, desc, threads, sp = oracle_sample(part, fwd_rows=fwd_rows, dx_rows=dx_rows, cols=cols, seed=seed)
            t += dt
            spent += sp
    return t, "per projection (a sliced one per slice): " + desc, threads, spent


def layer_name(L):
    q = L["qkv"]
    return "llama3_8b_layer_h%d_kv%d_i%d_T%d_P%d" % (q.K, (q.N - q.K) // 2, L["down"].K, q.T, q.n_adapters)


def reference_line(args, tokens, config, steps_fn):
    """The reference arm's line.  Each step is one bounded oracle sample (sample_size()) of the workload: its
    wall time is ms_per_step; value is the workload's tokens over the sample's linear extrapolation to a whole
    step, the same figure the GPU arm's cpu_baseline leg reports."""
    full, spent = [], []
    desc = threads = None
    for i in range(args.warmup + args.steps):
        t, desc, threads, sp = steps_fn(i)
        if i >= args.warmup:
            full.append(t)
            spent.append(sp)
    t = statistics.mean(full) if full else float("nan")
    v = tokens / t
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(spent) * 1e3 if spent else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "step": "one bounded oracle sample of the workload per step (ms_per_step is its measured wall time); "
                    "value extrapolates the sample linearly to whole steps (%.1f s per step)" % t,
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if "WORLD_SIZE" in os.environ:
        # rank 0 alone does the work; the launcher's one-thread-per-rank default would idle the other host cores
        # (the oracle's OpenMP runtime reads this when the oracle library is first loaded, below)
        os.environ["OMP_NUM_THREADS"] = str(os.cpu_count() or 1)
    sz = sample_size()
    if args.workload == "layer":
        L = make_layer(0, args.set)
        acc = {n: accounting(L[n]) for n in LAYER_ORDER}
        line = reference_line(args, L["qkv"].T, layer_config_dict(L, acc, args.gpus),
                              lambda i: layer_oracle_sample(L, seed=i, fwd_rows=16, dx_rows=8, cols=16))
    else:
        wl = make_workload(args.config, 0, args.set)
        acc = accounting(wl)
        line = reference_line(args, acc["tokens"], config_dict(wl, acc, args.gpus),
                              lambda i: oracle_sample(wl, seed=i, **sz))
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------------------- GPU arm
def to_dev(a, torch):
    return torch.from_numpy(workloads.bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def init_ranks():
    """(rank, world, local rank, torch.distributed or None); rank 0 builds the library, the others wait for it."""
    import torch
    import lora_co_serving_gb300 as lm

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        lm.build()                   # one rank compiles (if anything is stale); the others wait, then load it
    if dist:
        dist.barrier()
    return rank, world, local, dist


def kernel_roofline(kernel, flops, nbytes, ms, pk, traffic=None):
    """Roofline of one launch group: bound by whichever of its FLOPs at the bf16 peak and its bytes at the HBM peak
    takes longer.  The launches run for milliseconds at most inside a short timed region, so the peak is the burst
    figure (frac_of_sustained: against the seconds-long figure, for reference)."""
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_tc >= t_hbm:
        achieved = flops / (ms / 1e3) / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                "peak_source": pk["source"] + " (burst bf16)",
                "frac_of_sustained": achieved / pk["bf16_tflops_sustained"], "ms_per_launch": ms,
                "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes}
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic, "peak_source": pk["source"] + " (HBM copy)",
            "ms_per_launch": ms, "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes}


def step_roofline(flops, nbytes, ms, pk):
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_roof = max(t_tc, t_hbm)
    return {"tflops": flops / (ms / 1e3) / 1e12, "hbm_gbs": nbytes / (ms / 1e3) / 1e9,
            "bound": "tensor" if t_tc >= t_hbm else "hbm", "roofline_ms": t_roof * 1e3,
            "roofline_frac": t_roof * 1e3 / ms, "peak_source": pk["source"] + " (burst bf16, HBM copy)",
            "roofline_frac_of_sustained": max(flops / (pk["bf16_tflops_sustained"] * 1e12), t_hbm) * 1e3 / ms,
            "algorithmic_flops": flops, "algorithmic_bytes": nbytes}


def compact(line):
    """The per-workload summary carried in the headline line's `configs` object."""
    if line is None:
        return None
    out = {"workload": line["config"]["workload"], "ms_per_step": line["ms_per_step"], "tokens_per_s": line["value"],
           "steps": line["steps"], "warmup": line["warmup"], "l2": line["config"]["l2"],
           "dominant": {k: line["roofline"][k] for k in ("kernel", "bound", "achieved", "unit", "frac")},
           "step_roofline_frac": line["step"]["roofline_frac"], "step_bound": line["step"]["bound"],
           "tflops": line["step"]["tflops"], "hbm_gbs": line["step"]["hbm_gbs"],
           "hbm_frac": line["step"]["hbm_gbs"] / peaks()["hbm_gbs"], "clocks": line["clocks"],
           "gpu_launches": line["gpu_launches"]}
    if line.get("graph_replay"):
        out["graph_replay_ms_per_step"] = line["graph_replay"]["ms_per_step"]
    return out


def measure(args, cfg, rank, world, dist, steps, warmup, extras=True):
    """Time `steps` steps of workload `cfg` after `warmup` steps; returns rank 0's line (None elsewhere).  extras:
    also the flagged backward, AdamW, end-to-end and oracle legs (the headline); otherwise the step, its launch
    groups and its graph replay only."""
    import torch
    import lora_co_serving_gb300 as lm

    local = torch.cuda.current_device()
    wl = make_workload(cfg, rank, args.set if cfg == args.config else ())
    acc = accounting(wl)
    x, Wt, A, B = to_dev(wl.x, torch), to_dev(wl.Wt, torch), to_dev(wl.A, torch), to_dev(wl.B, torch)
    dY = to_dev(wl.dY, torch) if wl.dY is not None else None
    pool = lm.Pool(A, B, wl.a_off, wl.b_off, wl.rank, wl.scale)
    segs = lm.segments(wl.segs)
    T, K, N = wl.T, wl.K, wl.N
    ws = torch.empty(lm.workspace_size(T, K, N, 0, pool, segs), dtype=torch.uint8, device="cuda")
    fwd_info = lm.plan_describe(T, K, N, pool, segs)[1] if wl.forward else None
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    save = wl.xa_mode == "save"
    xs = torch.empty(max(1, lm.xa_size(0, pool, segs) // 2), dtype=torch.bfloat16, device="cuda") if save else None
    dX = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda") if wl.backward else None
    dA = torch.zeros(A.numel(), dtype=torch.float32, device="cuda") if wl.backward else None
    dB = torch.zeros(B.numel(), dtype=torch.float32, device="cuda") if wl.backward else None
    stream = torch.cuda.current_stream()

    def step_on(st):
        if wl.forward:
            lm.forward(x, Wt, pool, segs, y=y, xa_save=xs, save_xa=save, workspace=ws, stream=st)
        if wl.backward:
            lm.backward(x, Wt, pool, segs, dY, dX=dX, dA=dA, dB=dB, workspace=ws, stream=st)

    def step():
        step_on(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    lm.workspace_status(ws)

    # ---- L2: unless the inputs exceed twice the L2 size, L2 is flushed (a write of twice its size) before every
    # step, outside that step's own events
    l2_bytes = max(L2_NOMINAL, int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0) or 0))
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda") if needs_flush(input_bytes(wl)) else None

    # ---- device-timed region: K steps, per-step trace events around each launch group
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)]
    per = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for row in ev:          # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = NvmlSampler(torch.cuda.current_device())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.time()
    start.record(stream)
    for i in range(steps):
        if flush_buf is not None:
            flush_buf.fill_(i & 255)
        per[i][0].record(stream)
        lm.set_trace_events(ev[i])
        step()
        per[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    lm.set_trace_events(None)
    if dist:
        dist.barrier()
    lm.workspace_status(ws)
    if flush_buf is not None:
        ms = statistics.mean(per[i][0].elapsed_time(per[i][1]) for i in range(steps))
    else:
        ms = start.elapsed_time(stop) / steps
    group_ms = [statistics.mean(ev[i][2 * g].elapsed_time(ev[i][2 * g + 1]) for i in range(steps))
                for g in range(4)]
    t_max = torch.tensor([ms], device="cuda", dtype=torch.float64)
    if dist:
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    ms_max = float(t_max.item())
    value = acc["tokens"] * world / (ms_max / 1e3)

    # ---- the same step captured once into a CUDA graph and replayed (as a serving engine replays decode steps):
    # the library's host work (validation, planning, launches) leaves the timed region
    graph = None
    if not args.no_graph:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            for _ in range(2):
                step_on(gs)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs):
            step_on(gs)
        for _ in range(3):
            cg.replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        n_g = max(3, steps)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gper = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_g)]
        with torch.cuda.stream(gs):
            g0.record(gs)
            for i in range(n_g):
                if flush_buf is not None:
                    flush_buf.fill_(i & 255)
                gper[i][0].record(gs)
                cg.replay()
                gper[i][1].record(gs)
            g1.record(gs)
        torch.cuda.synchronize()
        g_ms = (statistics.mean(gper[i][0].elapsed_time(gper[i][1]) for i in range(n_g)) if flush_buf is not None
                else g0.elapsed_time(g1) / n_g)
        gms = torch.tensor([g_ms], device="cuda", dtype=torch.float64)
        if dist:
            dist.all_reduce(gms, op=dist.ReduceOp.MAX)
        graph = {"value": acc["tokens"] * world / (float(gms.item()) / 1e3), "unit": UNIT,
                 "ms_per_step": float(gms.item()), "steps": n_g,
                 "note": "one step captured into a CUDA graph, replayed back to back (no host work per step)"}
        del cg
        lm.workspace_status(ws)

    # ---- the backward with a per-segment flag table read on the device: every other fine-tuning segment (in
    # increasing start order) takes the xA its forward saved, the rest recompute it (and a table marking all
    # saved); timed on their own beside the all-recompute backward and the saved-xA backward without a table
    flagged = None
    n_train = sum(1 for _, ln, _, t in wl.segs.tolist() if t and ln > 0)
    if extras and wl.backward and n_train > 0 and lm.xa_size(0, pool, segs) > 0:
        xs_f = torch.empty(lm.xa_size(0, pool, segs) // 2, dtype=torch.bfloat16, device="cuda")
        lm.forward(x, Wt, pool, segs, y=y, xa_save=xs_f, save_xa=True, workspace=ws, stream=stream)
        modes = {"recompute_all": None, "saved_no_table": None,
                 "saved_half": torch.tensor([1 - (i % 2) for i in range(n_train)], dtype=torch.int32, device="cuda"),
                 "saved_all": torch.ones(n_train, dtype=torch.int32, device="cuda")}

        def bwd_mode(m):
            if m == "recompute_all":
                lm.backward(x, Wt, pool, segs, dY, dX=dX, dA=dA, dB=dB, recompute=True, workspace=ws, stream=stream)
            elif m == "saved_no_table":
                lm.backward(x, Wt, pool, segs, dY, xa_saved=xs_f, dX=dX, dA=dA, dB=dB, workspace=ws, stream=stream)
            else:
                lm.backward_flagged(x, Wt, pool, segs, dY, xs_f, modes[m], dX=dX, dA=dA, dB=dB, workspace=ws,
                                    stream=stream)
        n_f = max(3, min(steps, 50))
        flagged = {"segments": n_train}
        for m in modes:
            for _ in range(3):
                bwd_mode(m)
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            f0.record(stream)
            for _ in range(n_f):
                bwd_mode(m)
            f1.record(stream)
            torch.cuda.synchronize()
            flagged[m + "_ms"] = f0.elapsed_time(f1) / n_f
        lm.workspace_status(ws)
        del xs_f

    # ---- the optimizer step that follows (AdamW on the fine-tuning adapters, fp32 masters + bf16 pool), timed
    # on its own: it is not part of the forward+backward step the metric is about
    adamw_stats = None
    if extras and wl.backward:
        tads_u = sorted(set(int(a) for _, _, a, t in wl.segs.tolist() if t))
        masterA, masterB = A.float(), B.float()
        mA, vA = torch.zeros_like(masterA), torch.zeros_like(masterA)
        mB, vB = torch.zeros_like(masterB), torch.zeros_like(masterB)
        for i in range(3):
            lm.adamw_step(pool, K, N, dA, dB, mA, vA, mB, vB, tads_u, step=1 + i, A_master=masterA, B_master=masterB,
                          stream=stream)
        n_ad = max(3, min(steps, 50))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a0.record(stream)
        for i in range(n_ad):
            lm.adamw_step(pool, K, N, dA, dB, mA, vA, mB, vB, tads_u, step=4 + i, A_master=masterA,
                          B_master=masterB, stream=stream)
        a1.record(stream)
        torch.cuda.synchronize()
        ams = a0.elapsed_time(a1) / n_ad
        elems = sum(int(wl.rank[a]) * (K + N) for a in tads_u)
        abytes = elems * (4 * 4 + 3 * 4 + 2)      # read g, m, v, master; write m, v, master, bf16 weight
        adamw_stats = {"ms": ams, "elements": elems, "algorithmic_bytes": abytes,
                       "hbm_gbs": abytes / (ams / 1e3) / 1e9, "launches_per_call": 1}
        del masterA, masterB, mA, vA, mB, vB

    # ---- end to end: every step's inputs come from pinned host memory and its results go back to pinned host
    # memory.  Two device buffer sets let the inputs of step i+1 and the results of step i-1 move on two copy
    # streams (the copy engines) while step i computes, as a serving loop would run it.
    e2e = None
    if extras and not args.no_e2e:
        x_h = torch.empty_like(x, device="cpu").pin_memory()
        x_h.copy_(x)
        trows = wl.train_rows() if wl.backward else np.zeros(0, np.int64)
        tspans = sorted((s, l) for s, l, a, t in wl.segs.tolist() if t and l > 0) if wl.backward else []
        dY_h = dY.cpu().pin_memory() if wl.backward else None
        y_h = torch.empty_like(y, device="cpu").pin_memory()
        dX_h = torch.empty_like(dX, device="cpu").pin_memory() if wl.backward else None
        tads = sorted(set(int(a) for _, _, a, t in wl.segs.tolist() if t)) if wl.backward else []
        dA_h = torch.empty_like(dA, device="cpu").pin_memory() if wl.backward else None
        dB_h = torch.empty_like(dB, device="cpu").pin_memory() if wl.backward else None
        h2d = x.numel() * 2 + int(trows.shape[0]) * N * 2
        d2h = y.numel() * 2 + int(trows.shape[0]) * K * 2 + sum(int(wl.rank[a]) * (K + N) * 4 for a in tads)

        def like(t):
            return None if t is None else torch.empty_like(t)
        sets = [dict(x=x, dY=dY, y=y, dX=dX, dA=dA, dB=dB),
                dict(x=like(x), dY=like(dY), y=like(y), dX=like(dX), dA=like(dA), dB=like(dB))]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
        for b in range(2):
            ev["comp"][b].record(stream)
            ev["out"][b].record(s_out)

        # The inputs' copy is paced: issued in chunks of ~16 MB with short spin kernels between them, spread over
        # ~80 % of a device step.  At full copy speed the copy engine's writes evict the main pass's working set
        # from L2 in a burst and slow the step by ~0.6-1.0 ms on the headline (251 MB); paced, the same bytes cost
        # ~0.04 ms.  The chunk list and the gap come from unpaced copies timed here, outside the timed region.
        def in_pieces(d):
            out = [(d["x"], x_h)] + [(d["dY"][s0:s0 + l], dY_h[s0:s0 + l]) for s0, l in tspans]
            chunks = []
            for dst, src in out:
                rows = max(1, (16 << 20) // max(1, src[0].numel() * src.element_size()))
                chunks += [(dst[r:r + rows], src[r:r + rows]) for r in range(0, src.shape[0], rows)]
            return chunks
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h2d_runs = []
        for rep in range(4):            # the first copy out of freshly pinned memory runs cold: not timed
            c0.record(s_in)
            with torch.cuda.stream(s_in):
                for dst, src in in_pieces(sets[0]):
                    dst.copy_(src, non_blocking=True)
            c1.record(s_in)
            torch.cuda.synchronize()
            if rep:
                h2d_runs.append(c0.elapsed_time(c1))
        h2d_ms = min(h2d_runs)
        pieces = [in_pieces(sets[0]), in_pieces(sets[1])]
        gap_us = max(0.0, 0.8 * ms * 1e3 - h2d_ms * 1e3) / max(1, len(pieces[0]) - 1)
        gap_cycles = int(gap_us * pk_clock_mhz())

        def e2e_step(i):
            b = i % 2
            d = sets[b]
            s_in.wait_event(ev["comp"][b])            # step i-2 has finished reading this set's inputs
            with torch.cuda.stream(s_in):
                for k, (dst, src) in enumerate(pieces[b]):
                    if k and gap_cycles:
                        torch.cuda._sleep(gap_cycles)
                    dst.copy_(src, non_blocking=True)
            ev["in"][b].record(s_in)
            stream.wait_event(ev["in"][b])
            stream.wait_event(ev["out"][b])           # step i-2's results have left this set
            if wl.forward:
                lm.forward(d["x"], Wt, pool, segs, y=d["y"], xa_save=xs, save_xa=save, workspace=ws, stream=stream)
            if wl.backward:
                lm.backward(d["x"], Wt, pool, segs, d["dY"], dX=d["dX"], dA=d["dA"], dB=d["dB"], workspace=ws,
                            stream=stream)
            ev["comp"][b].record(stream)
            s_out.wait_event(ev["comp"][b])
            with torch.cuda.stream(s_out):
                y_h.copy_(d["y"], non_blocking=True)
                for s0, l in tspans:
                    dX_h[s0:s0 + l].copy_(d["dX"][s0:s0 + l], non_blocking=True)
                for a in tads:
                    ao, bo, r = int(wl.a_off[a]), int(wl.b_off[a]), int(wl.rank[a])
                    dA_h[ao:ao + r * K].copy_(d["dA"][ao:ao + r * K], non_blocking=True)
                    dB_h[bo:bo + r * N].copy_(d["dB"][bo:bo + r * N], non_blocking=True)
            ev["out"][b].record(s_out)

        n_e2e = max(4, min(steps, 30))
        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        ems = torch.tensor([e0.elapsed_time(e1) / n_e2e], device="cuda", dtype=torch.float64)
        if dist:
            dist.all_reduce(ems, op=dist.ReduceOp.MAX)
        e2e = {"value": acc["tokens"] * world / (float(ems.item()) / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": float(ems.item()), "steps": n_e2e,
               "overlap": "inputs of step i+1 (in %d chunks, %.0f us apart) and results of step i-1 on copy streams "
                          "during step i" % (len(pieces[0]), gap_us), "h2d_unpaced_ms": h2d_ms}
        del sets

    # ---- roofline of the dominant launch (the forward main pass; the backward main pass without a forward) and of
    # the whole step
    pk = peaks()
    line = None
    if rank == 0:
        if wl.forward:
            roof = kernel_roofline("lora_main2_kernel (forward main pass: x W + fused LoRA expand, CTA pairs)",
                                   acc["fwd_main_flops"], acc["fwd_main_bytes"], group_ms[1], pk,
                                   profiled_traffic(cfg))
        else:
            roof = kernel_roofline("lora_main2_kernel (backward dX pass) + lora_tc_kernel (dA, dB)",
                                   acc["bwd_main_flops"], acc["bwd_bytes"], group_ms[3], pk)
        step_stats = step_roofline(acc["flops"], acc["bytes"], ms, pk)
        step_stats["group_ms"] = {"fwd_shrink": group_ms[0], "fwd_main": group_ms[1], "bwd_shrink": group_ms[2],
                                  "bwd_main": group_ms[3]}
        cpu = None
        if extras and not args.no_cpu_baseline and world == 1:
            t_cpu, desc, threads, _ = oracle_sample(wl, **sample_size())
            cpu = {"value": acc["tokens"] / t_cpu, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
                "warmup": warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes of the pages' workloads)",
                "config": config_dict(wl, acc, world),
                "roofline": roof, "step": step_stats, "cpu_baseline": cpu, "clocks": clocks, "e2e": e2e,
                "graph_replay": graph, "adamw": adamw_stats, "flagged_backward": flagged,
                "gpu_launches": launches_per_step(wl, fwd_info) * steps}
    if dist:
        dist.barrier()
    return line


def run_ours(args):
    rank, world, local, dist = init_ranks()
    if args.workload == "layer":
        line = measure_layer(args, rank, world, dist, args.steps, args.warmup, extras=True)
    else:
        line = measure(args, args.config, rank, world, dist, args.steps, args.warmup, extras=True)
    # the other workloads at one GPU, 20 timed steps each, so that their numbers are measured in the same run
    if world == 1 and not args.no_configs and not args.set:
        configs = {}
        for cfg in (2, 3, 4, 5):
            if args.workload == "config" and cfg == args.config:
                continue
            configs["config%d" % cfg] = compact(measure(args, cfg, 0, 1, None, 20, 5, extras=False))
        if args.workload != "layer":
            configs["layer"] = compact(measure_layer(args, 0, 1, None, 20, 5, extras=False))
        line["configs"] = configs
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def measure_layer(args, rank, world, dist, steps, warmup, extras=True):
    """One decoder layer's LoRA projections per step: forward q|k|v -> o -> gate|up -> down over every token, then
    the LoRA backward of the fine-tuning tokens in reverse order, all on one stream with one shared workspace.
    Returns rank 0's line (None elsewhere); extras: also the oracle leg."""
    import torch
    import lora_co_serving_gb300 as lm

    L = make_layer(rank, args.set if args.workload == "layer" else ())
    T = L["qkv"].T
    acc = {n: accounting(L[n]) for n in LAYER_ORDER}
    dev = {}
    need = 0
    for n in LAYER_ORDER:
        wl = L[n]
        d = {"x": to_dev(wl.x, torch), "Wt": to_dev(wl.Wt, torch), "A": to_dev(wl.A, torch),
             "B": to_dev(wl.B, torch), "dY": to_dev(wl.dY, torch)}
        d["pool"] = lm.Pool(d["A"], d["B"], wl.a_off, wl.b_off, wl.rank, wl.scale)
        d["segs"] = lm.segments(wl.segs)
        d["sl"] = lm.Slices(wl.bounds) if wl.bounds is not None else None
        d["info"] = lm.plan_describe(T, wl.K, wl.N, d["pool"], d["segs"])[1]      # the tile plan (slices alike)
        d["y"] = torch.empty((T, wl.N), dtype=torch.bfloat16, device="cuda")
        d["dX"] = torch.zeros((T, wl.K), dtype=torch.bfloat16, device="cuda")
        d["dA"] = torch.zeros(d["A"].numel(), dtype=torch.float32, device="cuda")
        d["dB"] = torch.zeros(d["B"].numel(), dtype=torch.float32, device="cuda")
        if d["sl"] is not None:
            need = max(need, lm.sliced_workspace_size(T, wl.K, wl.N, 0, d["pool"], d["sl"], d["segs"]))
        else:
            need = max(need, lm.workspace_size(T, wl.K, wl.N, 0, d["pool"], d["segs"]))
        dev[n] = d
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def fwd(n):
        d = dev[n]
        if d["sl"] is not None:
            lm.sliced_forward(d["x"], d["Wt"], d["pool"], d["sl"], d["segs"], y=d["y"], workspace=ws, stream=stream)
        else:
            lm.forward(d["x"], d["Wt"], d["pool"], d["segs"], y=d["y"], workspace=ws, stream=stream)

    def bwd(n):
        d = dev[n]
        kw = dict(dX=d["dX"], dA=d["dA"], dB=d["dB"], recompute=True, workspace=ws, stream=stream)
        if d["sl"] is not None:
            lm.sliced_backward(d["x"], d["Wt"], d["pool"], d["sl"], d["segs"], d["dY"], **kw)
        else:
            lm.backward(d["x"], d["Wt"], d["pool"], d["segs"], d["dY"], **kw)

    calls = [("fwd", n) for n in LAYER_ORDER] + [("bwd", n) for n in reversed(LAYER_ORDER)]

    def step(evs=None):
        for j, (kind, n) in enumerate(calls):
            if evs is not None:
                evs[j].record(stream)
            (fwd if kind == "fwd" else bwd)(n)
        if evs is not None:
            evs[len(calls)].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    lm.workspace_status(ws)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record(stream)
    tev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)]
    for row in tev:
        for e in row:
            e.record(stream)
    sampler = NvmlSampler(torch.cuda.current_device())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.time()
    for i in range(steps):
        # trace the launch groups of the gate|up forward (the layer's largest launch)
        for j, (kind, n) in enumerate(calls):
            evs[i][j].record(stream)
            if kind == "fwd" and n == "gate_up":
                lm.set_trace_events(tev[i])
            (fwd if kind == "fwd" else bwd)(n)
            if kind == "fwd" and n == "gate_up":
                lm.set_trace_events(None)
        evs[i][len(calls)].record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    lm.workspace_status(ws)
    ms_steps = [evs[i][0].elapsed_time(evs[i][len(calls)]) for i in range(steps)]
    ms = statistics.mean(ms_steps)
    per_call = {"%s_%s" % c: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps))
                for j, c in enumerate(calls)}
    gu_main_ms = statistics.mean(tev[i][2].elapsed_time(tev[i][3]) for i in range(steps))
    t_max = torch.tensor([ms], device="cuda", dtype=torch.float64)
    if dist:
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    ms_max = float(t_max.item())
    value = T * world / (ms_max / 1e3)
    pk = peaks()
    line = None
    if rank == 0:
        flops = sum(a["flops"] for a in acc.values())
        nbytes = sum(a["bytes"] for a in acc.values())
        roof = kernel_roofline("lora_main2_kernel (gate|up forward main pass: x W + fused LoRA expand, 2 slices)",
                               acc["gate_up"]["fwd_main_flops"], acc["gate_up"]["fwd_main_bytes"], gu_main_ms, pk)
        step_stats = step_roofline(flops, nbytes, ms, pk)
        step_stats["call_ms"] = per_call
        cpu = None
        if extras and not args.no_cpu_baseline and world == 1:
            t_cpu, desc, threads, _ = layer_oracle_sample(L, fwd_rows=16, dx_rows=8, cols=16)
            cpu = {"value": T / t_cpu, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
                "warmup": warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes of the pages' workloads)",
                "config": layer_config_dict(L, acc, world), "roofline": roof, "step": step_stats,
                "cpu_baseline": cpu, "clocks": clocks, "e2e": None,
                "gpu_launches": sum(launches_per_step(L[n], dev[n]["info"]) for n in LAYER_ORDER) * steps}
    if dist:
        dist.barrier()
    return line


def sweep_tables(L, seed=77):
    """Segment tables of the sweep: decode-only batches (Eq. II) and mixed batches of decode, prefill and
    fine-tuning tokens (Eq. I), adapters drawn like the layer workload's."""
    rng = np.random.Generator(np.random.PCG64(seed))
    wl = L["qkv"]
    n_inf = wl.n_adapters - 1
    train_ad = int(wl.meta["train_adapter"])

    def table(b_d, t_in, t_ft):
        segs, t = [], 0
        for a in workloads._zipf_ids(rng, b_d, n_inf, 1.1):
            segs.append((t, 1, int(a), 0))
            t += 1
        for ln in (workloads._draw_lengths(rng, t_in, 64, 1024) if t_in else []):
            if ln == 1:                               # a 1-token remainder would read as a decode request
                ln, segs[-1] = ln, (segs[-1][0], segs[-1][1] + 1, segs[-1][2], 0)
                t += 1
                continue
            segs.append((t, ln, int(rng.integers(0, n_inf)), 0))
            t += ln
        left = t_ft
        while left > 0:
            ln = min(1024, left)
            segs.append((t, ln, train_ad, 1))
            t += ln
            left -= ln
        return np.asarray(segs, np.int32), t

    decode = [table(b, 0, 0) for b in (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 80, 96, 128, 160, 192, 256, 320, 384,
                                       448, 512, 640, 768, 896, 1024, 1152, 1280, 1408, 1536, 1792, 2048)]
    mixed = []
    for b_d in (0, 256, 1024, 2048):
        for t_in in (0, 1024, 2048, 4096):
            for t_ft in (0, 1024, 2048):
                if t_in == 0 and t_ft == 0:
                    continue
                mixed.append(table(b_d, t_in, t_ft))
    return decode, mixed


def run_sweep(args):
    """Time the layer step over the sweep's batch compositions and fit Eq. I (mixed) and Eq. II (decode-only)."""
    import torch
    import lora_co_serving_gb300 as lm

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    lm.build()
    L = make_layer(0, args.set)
    decode, mixed = sweep_tables(L)
    dev = {}
    need = 0
    for n in LAYER_ORDER:
        wl = L[n]
        d = {"x": to_dev(wl.x, torch), "Wt": to_dev(wl.Wt, torch), "A": to_dev(wl.A, torch),
             "B": to_dev(wl.B, torch), "dY": to_dev(wl.dY, torch)}
        d["pool"] = lm.Pool(d["A"], d["B"], wl.a_off, wl.b_off, wl.rank, wl.scale)
        d["sl"] = lm.Slices(wl.bounds) if wl.bounds is not None else None
        d["y"] = torch.empty((wl.T, wl.N), dtype=torch.bfloat16, device="cuda")
        d["dX"] = torch.zeros((wl.T, wl.K), dtype=torch.bfloat16, device="cuda")
        d["dA"] = torch.zeros(d["A"].numel(), dtype=torch.float32, device="cuda")
        d["dB"] = torch.zeros(d["B"].numel(), dtype=torch.float32, device="cuda")
        for segs, T in decode + mixed:
            if d["sl"] is not None:
                need = max(need, lm.sliced_workspace_size(T, wl.K, wl.N, 0, d["pool"], d["sl"], segs))
            else:
                need = max(need, lm.workspace_size(T, wl.K, wl.N, 0, d["pool"], segs))
        dev[n] = d
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(segs, T, stream=stream):
        train = bool((segs[:, 3] != 0).any())
        for n in LAYER_ORDER:
            d = dev[n]
            if d["sl"] is not None:
                lm.sliced_forward(d["x"][:T], d["Wt"], d["pool"], d["sl"], segs, y=d["y"][:T], workspace=ws,
                                  stream=stream)
            else:
                lm.forward(d["x"][:T], d["Wt"], d["pool"], segs, y=d["y"][:T], workspace=ws, stream=stream)
        if train:
            for n in reversed(LAYER_ORDER):
                d = dev[n]
                kw = dict(dX=d["dX"][:T], dA=d["dA"], dB=d["dB"], recompute=True, workspace=ws, stream=stream)
                if d["sl"] is not None:
                    lm.sliced_backward(d["x"][:T], d["Wt"], d["pool"], d["sl"], segs, d["dY"][:T], **kw)
                else:
                    lm.backward(d["x"][:T], d["Wt"], d["pool"], segs, d["dY"][:T], **kw)

    reps = max(3, min(args.steps, 10))

    gs = torch.cuda.Stream()

    def time_point(segs, T):
        """Median device time of the step replayed from a CUDA graph (as an engine replays its steps: no host work
        in the timed region), and the median of the same step launched eagerly."""
        for _ in range(max(3, args.warmup)):
            step(segs, T)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        eager = []
        for _ in range(reps):
            torch.cuda.synchronize()
            e0.record(stream)
            step(segs, T)
            e1.record(stream)
            torch.cuda.synchronize()
            eager.append(e0.elapsed_time(e1))
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            step(segs, T, gs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            step(segs, T, gs)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ts = []
        with torch.cuda.stream(gs):
            for _ in range(reps):
                e0.record(gs)
                g.replay()
                e1.record(gs)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
        del g
        return statistics.median(ts), statistics.median(eager)

    sampler = NvmlSampler(torch.cuda.current_device())
    sampler.start()
    wall0 = time.time()
    res = {}
    for name, pts, model in (("decode", decode, lm.EQ_II), ("mixed", mixed, lm.EQ_I)):
        F = np.array([lm.latency_features(model, segs) for segs, _ in pts])
        both = [time_point(segs, T) for segs, T in pts]
        t = np.array([b[0] for b in both])
        t_eager = np.array([b[1] for b in both])
        coef = lm.latency_fit(model, F, t)
        pred = F @ coef
        rel = np.abs(pred - t) / t
        r2 = 1.0 - float(((t - pred) ** 2).sum() / max(1e-300, ((t - t.mean()) ** 2).sum()))
        # 5-fold cross-validation: relative error of each point when it is left out of the fit
        folds = np.arange(len(pts)) % 5
        cv = np.zeros(len(pts))
        for k in range(5):
            tr, te = folds != k, folds == k
            ck = lm.latency_fit(model, F[tr], t[tr])
            cv[te] = np.abs(F[te] @ ck - t[te]) / t[te]
        names = ["alpha", "beta", "gamma", "eps", "c"] if model == lm.EQ_I else ["beta'", "eps'", "c'"]
        res[name] = {"equation": "I" if model == lm.EQ_I else "II", "points": len(pts),
                     "coefficients_ms": dict(zip(names, coef.tolist())), "r2": r2,
                     "median_rel_err": float(np.median(rel)), "max_rel_err": float(rel.max()),
                     "cv_median_rel_err": float(np.median(cv)), "cv_max_rel_err": float(cv.max()),
                     "samples": [{"features": f.tolist(), "ms": float(x), "eager_ms": float(xe)}
                                 for f, x, xe in zip(F, t, t_eager)]}
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    line = {"metric": "step-latency model fit (DeltaServe Eq. I / II) over the layer step", "unit": "ms",
            "n_gpus": 1, "data": "synthetic (seeded; shapes of the pages' workloads)",
            "config": {"workload": layer_name(L) + "_sweep", "reps_per_point": reps,
                       "timing": "each point's step replayed from a CUDA graph (device time, no host work); the "
                                 "eager median is kept per sample as eager_ms",
                       "step": "forward of q|k|v, o, gate|up, down over every token + LoRA backward of the "
                               "fine-tuning tokens (xA recomputed)",
                       "features": "Eq. I {sum (n_i+B_d)^2, T_in+B_d, T_ft, K=0, 1}; Eq. II {B_d, K=0, 1}"},
            "fit": res, "clocks": clocks}
    print(json.dumps(line), flush=True)
    if args.out:
        json.dump({k: {"equation": v["equation"], "coefficients_ms": v["coefficients_ms"], "r2": v["r2"],
                       "cv_median_rel_err": v["cv_median_rel_err"], "cv_max_rel_err": v["cv_max_rel_err"],
                       "points": v["points"]} for k, v in res.items()},
                  open(args.out, "w"), indent=1)
    return 0


def run_gemm(args):
    """Calibration: the layer's main pass on a base-only batch (x W alone, no adapters) and cuBLAS's GEMM for the
    same product, each captured into a CUDA graph and replayed (median of `--steps` replays after `--warmup`); L2 is
    flushed before every replay when the operands fit in twice its size."""
    import torch
    import lora_co_serving_gb300 as lm
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    lm.build()
    kw = {"M": 4096, "K": 4096, "N": 4864, "flush": 1}
    for item in args.set:
        k, v = item.split("=", 1)
        kw[k] = int(v)
    M, K, N = kw["M"], kw["K"], kw["N"]
    g = torch.Generator(device="cuda").manual_seed(1007)
    x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    Wt = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    y = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    A = torch.zeros(16 * K, device="cuda", dtype=torch.bfloat16)
    B = torch.zeros(16 * N, device="cuda", dtype=torch.bfloat16)
    pool = lm.Pool(A, B, [0], [0], [16], [2.0])
    segs = lm.segments([(0, M, -1, 0)])
    ws = torch.empty(lm.workspace_size(M, K, N, 0, pool, segs), dtype=torch.uint8, device="cuda")
    # --set flush=0 keeps operands that fit in L2 resident between replays (the kernel's own rate, no DRAM)
    flush = torch.empty(2 * L2_NOMINAL, dtype=torch.uint8, device="cuda") \
        if kw.get("flush", 1) and 2 * (M + N) * K <= 2 * L2_NOMINAL else None

    def timed(fn):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(max(3, args.warmup)):
                fn(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            fn(s)
        ts = []
        for i in range(max(3, args.warmup) + args.steps):
            if flush is not None:
                flush.fill_(i & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            if i >= max(3, args.warmup):
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    t_ours = timed(lambda s: lm.forward(x, Wt, pool, segs, y=y, workspace=ws, stream=s))
    t_ref = timed(lambda s: torch.matmul(x, Wt.t(), out=y))
    f = 2.0 * M * N * K
    pk = peaks()
    print(json.dumps({"metric": "base-only main pass vs cuBLAS", "unit": "TFLOP/s", "M": M, "K": K, "N": N,
                      "ours_ms": t_ours, "cublas_ms": t_ref, "ours_tflops": f / t_ours / 1e9,
                      "cublas_tflops": f / t_ref / 1e9, "ratio": t_ref / t_ours,
                      "ours_frac_of_burst": f / t_ours / 1e9 / pk["bf16_tflops"],
                      "l2": "flushed before every replay" if flush is not None else "no flush",
                      "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def spawn_ranks(n):
    """Run this command again as n ranks of one node (torch.distributed.run, rendezvous on 127.0.0.1), one per GPU;
    returns the launcher's exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n), "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def selftest_ranks(args):
    """Each rank joins a gloo group and contributes its rank; rank 0 prints what met."""
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo")
    t = torch.tensor([float(dist.get_rank())])
    dist.all_reduce(t)
    if dist.get_rank() == 0:
        print(json.dumps({"ranks": dist.get_world_size(), "rank_sum": float(t.item()), "gpus": args.gpus}), flush=True)
    dist.barrier()
    dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: the command starts its own ranks when no launcher did
        return spawn_ranks(args.gpus)
    if "WORLD_SIZE" in os.environ and int(os.environ["WORLD_SIZE"]) != args.gpus:
        raise SystemExit("--gpus %d but %s ranks were launched" % (args.gpus, os.environ["WORLD_SIZE"]))
    if args.selftest_ranks:
        return selftest_ranks(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "sweep":
        return run_sweep(args)
    if args.workload == "gemm":
        return run_gemm(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
