"""Benchmark of the GB300 attention forward (one step = one forward pass).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line.  `value` is TFLOP/s with the causal FLOP count halved
(4*B*Hq*Sq*Skv*D, integer-halved when causal -- the count the Pallas page's
benchmark `main` uses), from CUDA events around each kernel launch on its
stream, inputs resident in HBM, L2 flushed (a 256 MiB write) between steps.
`e2e` is the same metric through the C ABI with pinned host buffers: the
host->device copies of Q, K, V and the device->host copies of O and LSE of
every step are inside its timed region, pipelined over two device buffer sets
(step i+1's uploads and step i-1's download overlap step i's kernel); beside it,
the machine's host link rates, the bound they put on e2e, and the step's own copies
timed alone (`step_copies_gbs`).  `roofline` relates the kernel to the measured dense
bf16 tensor peak.  `cpu_baseline` times the fp64 oracle on a bounded sample of
the same workload on the host cores.

The timed region is the K-step block repeated until it spans at least
--min-timed-seconds (default 1 s), each block bracketed by a barrier and a
device synchronisation, so the NVML sampler (every 5 ms) sees the kernel under
load; `value` is the mean over every timed step.  `roofline.clock_matched`
relates the kernel to the tensor pipe's rate at the SM clock sampled meanwhile
(8192 bf16 FLOP per clock per SM: one 128x128x16 MMA every 64 cycles, the
measured rate of this part).  `workloads` holds kernel-only timings of the
other benchmark shapes (a few steps each, same rules).

--path bwd times attn_bwd instead (one step = the gradients dq, dk, dv of one
forward, 2.5x its FLOPs); it prints no cpu_baseline.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the forward pass has no exchange step); the max over ranks of
the timed region divides the work of all ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16, causal FLOPs halved) and % of GB300 dense bf16 peak"
METRIC_BWD = "attention bwd TFLOP/s (2.5x the forward's FLOPs, causal halved)"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
# bf16 FLOP per SM clock of the tensor pipe: 2*128*128*16 per 64-cycle MMA (measured rate)
TENSOR_FLOP_PER_CLK_PER_SM = 8192
# shapes whose kernel-only throughput is reported beside the headline
OTHER_WORKLOADS = ("tiny_causal", "tiny_noncausal", "gqa_causal_2x32x8_8192", "long_sharp_1x16x16384",
                   "chunked_prefill_gqa_64x8_512x32768")


def kernel_name(w, bwd: bool) -> str:
    """The kernels one step of the timed path launches."""
    if bwd and w.D == 256:
        return ("attn_bwd step: bwd_prep_kernel + fmha_bwd_d256_kernel (dV, dK and dQ "
                "launches)")
    if bwd:
        return "attn_bwd step: bwd_prep_kernel + fmha_bwd_dkdv_kernel + fmha_bwd_dq_kernel"
    return "attn::d256::fmha_fwd_d256_kernel" if w.D == 256 else "attn::fmha_fwd_kernel"


def metric_flops(w) -> int:
    f = 4 * w.B * w.Hq * w.Sq * w.Skv * w.D
    return f // 2 if w.causal else f


def visible_pairs(w) -> int:
    """Exact number of (query row, key) pairs the mask lets through, per head and batch."""
    if not w.causal:
        return w.Sq * w.Skv
    off = w.Skv - w.Sq if w.causal == 1 else 0
    total = 0
    for i in range(w.Sq):
        total += max(0, min(w.Skv, i + off + 1))
    return total


def exact_flops(w) -> int:
    return 4 * w.D * w.B * w.Hq * visible_pairs(w)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


FWD_KERNEL_SOURCES = ("fmha_fwd_sm103.cuh", "sm103_ptx.cuh")


def kernel_source_digest() -> str:
    """Digest of the forward kernel's sources (its template and the PTX wrappers
    it is built from): a committed DRAM-traffic figure is used only while it
    matches the kernel the bench runs."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_11_gb300", "csrc")
    for name in FWD_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(workload)
        if rec and rec.get("kernel_source_digest") == kernel_source_digest():
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ clocks (NVML, read-only)
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while running."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, index: int, period_s: float = 0.005):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period = period_s
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                raise OSError("no handle")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except OSError:
            self.nvml = None

    def _run(self):
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if get_reasons(self.handle, ctypes.byref(reasons)) == 0:
                for bit, name in self.REASONS.items():
                    if reasons.value & bit and bit != 0x1:
                        self.reasons.add(name)
            time.sleep(self.period)

    def __enter__(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "NVML unavailable"}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples)}


# ------------------------------------------------------------------ CPU baseline (oracle)
def oracle_sample_rate(w, target_s: float, seed: int = 0, q=None, k=None, v=None):
    """Times the fp64 oracle on a sample of the workload's query rows sized to
    about `target_s` seconds; returns (TFLOP/s, seconds, rows, threads)."""
    import numpy as np
    import oracle
    from attention_forward_11_gb300 import inputs
    if q is None:
        q, k, v = inputs.make_workload(w, seed=seed)
    rng = np.random.default_rng(seed + 17)

    def rows_of(n):
        return np.stack([rng.integers(0, w.B, n), rng.integers(0, w.Hq, n),
                         rng.integers(0, w.Sq, n)], axis=1).astype(np.int64)

    def flops_of(rows):
        off = w.Skv - w.Sq if w.causal == 1 else 0
        vis = np.minimum(w.Skv, rows[:, 2] + off + 1) if w.causal else np.full(len(rows), w.Skv)
        return float(4 * w.D * np.maximum(vis, 0).sum())

    # calibrate: double the probe until it runs for ~1/8 of the target
    n, dt = 64, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, rows_of(n), int(w.causal), w.scale)
        dt = time.perf_counter() - t0
        if dt >= target_s / 8 or n >= 1_000_000:
            break
        n *= 2
    n = int(max(64, min(4_000_000, n * target_s / max(dt, 1e-4))))
    rows = rows_of(n)
    t0 = time.perf_counter()
    oracle.attn_rows(q, k, v, rows, int(w.causal), w.scale)
    dt = time.perf_counter() - t0
    return flops_of(rows) / dt / 1e12, dt, n, oracle.num_threads()


def oracle_one_core(workload: str, target_s: float):
    """The same oracle sample timed with one OpenMP thread, in a child process
    (the thread count is fixed when the oracle library loads)."""
    import subprocess
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "from attention_forward_11_gb300 import inputs; "
            "w = inputs.WORKLOADS[%r]; tf, dt, n, c = bench.oracle_sample_rate(w, %r); "
            "print(json.dumps([tf, dt, n, c]))") % (ROOT, workload, target_s)
    env = {**os.environ, "OMP_NUM_THREADS": "1"}
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True, timeout=600)
    tf, dt, n, cores = json.loads(out.stdout.strip().splitlines()[-1])
    return tf, dt, n, cores


def numpy_fp64_rate(w, seed: int = 0):
    """numpy fp64 (BLAS matmuls) on one (batch, head) slice of the workload: the
    plain masked softmax(scale Q K^T) V, timed; returns (TFLOP/s, seconds)."""
    import numpy as np
    from attention_forward_11_gb300 import inputs
    q = inputs.normal_bf16((w.Sq, w.D), w.q_sigma, seed, 0).astype(np.uint32) << 16
    k = inputs.normal_bf16((w.Skv, w.D), w.kv_sigma, seed, 1).astype(np.uint32) << 16
    v = inputs.normal_bf16((w.Skv, w.D), w.kv_sigma, seed, 2).astype(np.uint32) << 16
    q, k, v = (t.view(np.float32).astype(np.float64) for t in (q, k, v))
    t0 = time.perf_counter()
    s = w.scale * (q @ k.T)
    if w.causal:
        off = w.Skv - w.Sq if w.causal == 1 else 0
        s[np.arange(w.Skv)[None, :] > np.arange(w.Sq)[:, None] + off] = -np.inf
    m = s.max(axis=1, keepdims=True)
    m[~np.isfinite(m)] = 0.0
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ v) / np.where(l > 0, l, 1.0)
    dt = time.perf_counter() - t0
    del o
    flops = 4 * w.D * visible_pairs(w)
    return flops / dt / 1e12, dt


# ------------------------------------------------------------------ multi-rank helpers
def max_over_ranks(values, device):
    """Element-wise max of `values` over all ranks of the default process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(world: int, flops_per_step: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step`;
    `seconds` is the slowest rank's timed region."""
    return world * flops_per_step * steps / seconds / 1e12


# ------------------------------------------------------------------ main arms
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from attention_forward_11_gb300 import inputs
    oracle.build()
    q, k, v = inputs.make_workload(w, seed=0)
    per_step = args.ref_step_seconds
    vals, secs, rows = [], [], 0
    for i in range(args.warmup + args.steps):
        tf, dt, n, cores = oracle_sample_rate(w, per_step, seed=i, q=q, k=k, v=v)
        if i >= args.warmup:
            vals.append(tf)
            secs.append(dt)
            rows = n
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * metric_flops(w) / (value * 1e12),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {**w.as_dict(), "parallelism": "replicas" if args.gpus > 1 else "single"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} random query rows of the workload per step, "
                                   f"~{per_step:.0f} s each; ms_per_step extrapolated to the "
                                   f"whole workload"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    del np
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import numpy as np
    import torch

    import attention_forward_11_gb300 as fa
    from attention_forward_11_gb300 import build as libbuild
    from attention_forward_11_gb300 import inputs

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        libbuild.build()
    if world > 1:
        dist.barrier()
    fa.load_library()

    q_h, k_h, v_h = inputs.make_qkv(w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, seed=rank,
                                    q_sigma=w.q_sigma, kv_sigma=w.kv_sigma, dtype=args.dtype)
    tdtype = torch.float16 if args.dtype == "f16" else torch.bfloat16

    def pinned(bits):
        t = torch.from_numpy(bits.view(np.int16)).view(tdtype)
        return t.pin_memory()

    qp, kp, vp = pinned(q_h), pinned(k_h), pinned(v_h)
    q = qp.to(dev)
    k = kp.to(dev)
    v = vp.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    o_h = torch.empty(o.shape, dtype=tdtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    ws_bytes = 0
    if args.path == "splitkv":  # the caller's scratch, allocated once outside the timed region
        ws_bytes = fa.attn_fwd_splitkv_workspace_size(w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, w.causal)
    elif args.path == "bwd":
        ws_bytes = fa.attn_bwd_workspace_size(w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    dtype_code = fa.ATTN_DTYPE_F16 if args.dtype == "f16" else fa.ATTN_DTYPE_BF16
    if args.path == "bwd":
        # the backward step's other inputs: the forward's O and LSE, and a seeded dO
        st = fa.attn_fwd_ex_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, w.causal, w.scale, dtype_code, sh)
        if st != fa.ATTN_OK:
            raise fa.AttnError(st, "attn_fwd_ex")
        dop = pinned(inputs.normal_bf16(q_h.shape, 1.0, rank, 3, args.dtype))
        do = dop.to(dev)
        op = torch.empty(o.shape, dtype=tdtype).pin_memory()
        op.copy_(o)
        lsep = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        lsep.copy_(lse)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dq_h = torch.empty(dq.shape, dtype=tdtype).pin_memory()
        dk_h = torch.empty(dk.shape, dtype=tdtype).pin_memory()
        dv_h = torch.empty(dv.shape, dtype=tdtype).pin_memory()

    bufs0 = {"q": q, "k": k, "v": v, "o": o, "lse": lse}
    if args.path == "bwd":
        bufs0.update(do=do, dq=dq, dk=dk, dv=dv)

    def step(b=None):
        b = bufs0 if b is None else b
        q, k, v, o, lse = b["q"], b["k"], b["v"], b["o"], b["lse"]
        if args.path == "bwd":
            do, dq, dk, dv = b["do"], b["dq"], b["dk"], b["dv"]
            st = fa.attn_bwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.Sq,
                                 w.Skv, w.Hq, w.Hkv, w.D, w.causal, w.scale, dtype_code, ws.data_ptr(),
                                 ws_bytes, sh)
        elif args.path == "splitkv":
            st = fa.attn_fwd_splitkv_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D,
                                         w.causal, w.scale, ws.data_ptr(), ws_bytes, sh)
        elif args.dtype == "f16":
            st = fa.attn_fwd_ex_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, w.causal,
                                    w.scale, fa.ATTN_DTYPE_F16, sh)
        else:
            st = fa.attn_fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, w.causal,
                                 w.scale, sh)
        if st != fa.ATTN_OK:
            raise fa.AttnError(st, "attn_fwd")

    # ---- warm-up (timed too, only to size the timed region)
    w_start = torch.cuda.Event(enable_timing=True)
    w_end = torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        flush.zero_()
        if i == args.warmup - 1:
            w_start.record(stream)
        step()
        if i == args.warmup - 1:
            w_end.record(stream)
    if fa.attn_check_device_status(stream) != fa.ATTN_OK:
        raise RuntimeError("device status not OK after warm-up")
    est_step_s = max(w_start.elapsed_time(w_end) / 1e3, 1e-6)
    # the K-step block is repeated until the timed region spans min_timed_seconds
    repeats = max(1, math.ceil(args.min_timed_seconds / (args.steps * (est_step_s + 50e-6))))
    if world > 1:
        repeats = int(max_over_ranks([repeats], dev)[0])

    # ---- timed: repeats x K steps, L2 flushed between steps, events around each launch
    n_timed = repeats * args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    launches0 = fa.attn_kernel_launches()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for r in range(repeats):
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize(dev)
            for i in range(r * args.steps, (r + 1) * args.steps):
                flush.zero_()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    launches = fa.attn_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    if fa.attn_check_device_status(stream) != fa.ATTN_OK:
        raise RuntimeError("device status not OK after the timed region")
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_s = sum(times_ms) / 1e3 / repeats  # per block of K steps

    # ---- the host link the e2e figure runs over (outside every timed region)
    link = host_link_rates(dev)

    # ---- e2e: pinned host buffers; every step's host->device copies of its inputs
    # and the read of its result are inside the timed region, pipelined over two
    # device buffer sets: the uploads of step i+1 and the download of step i-1
    # run on their own streams while step i computes
    e2e_steps = max(3, min(args.steps, 20))
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    host_in = {"q": qp, "k": kp, "v": vp}
    host_out = {"o": o_h, "lse": lse_h}
    if args.path == "bwd":
        host_in.update(o=op, lse=lsep, do=dop)
        host_out = {"dq": dq_h, "dk": dk_h, "dv": dv_h}
    sets = [bufs0, {name: torch.empty_like(t) for name, t in bufs0.items()}]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # the step's own copies, timed alone (outside the timed region): a box whose
    # e2e falls far below link_bound shows here whether these buffers copy slower
    step_copy = {}
    for direction, pairs in (("h2d", [(sets[1][n], h) for n, h in host_in.items()]),
                             ("d2h", [(h, sets[1][n]) for n, h in host_out.items()])):
        best = 0.0
        nbytes = sum(src.numel() * src.element_size() for _, src in pairs)
        for _ in range(2):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            with torch.cuda.stream(up):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize(dev)
            best = max(best, nbytes / (time.perf_counter() - t0) / 1e9)
        step_copy[direction] = best
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    up.wait_event(e_start)
    for i in range(e2e_steps):
        si = i % 2
        b = sets[si]
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(ev_comp[si])  # step i-2 has finished reading this set's inputs
            for name, h in host_in.items():
                b[name].copy_(h, non_blocking=True)
            ev_up[si].record(up)
        stream.wait_event(ev_up[si])
        if i >= 2:
            stream.wait_event(ev_down[si])  # step i-2's result has been read out of this set
        step(b)
        ev_comp[si].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_comp[si])
            for name, h in host_out.items():
                h.copy_(b[name], non_blocking=True)
            ev_down[si].record(down)
    stream.wait_event(ev_down[(e2e_steps - 1) % 2])
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = e_start.elapsed_time(e_end) / 1e3

    if world > 1:
        kernel_s, e2e_s = max_over_ranks([kernel_s, e2e_s], dev)
        dist.destroy_process_group()
    if rank != 0:
        return

    bwd = args.path == "bwd"
    # backward: 2.5 x the forward's FLOPs (five products of 2 D FLOPs per pair, not two)
    fl_mult = 2.5 if bwd else 1.0
    flops = int(fl_mult * metric_flops(w))
    value = job_tflops(world, flops, args.steps, kernel_s)
    e2e_value = job_tflops(world, flops, e2e_steps, e2e_s)
    peak, peak_kind = load_peaks()
    exact = int(fl_mult * exact_flops(w))
    mean_launch_s = kernel_s / args.steps
    achieved = exact / mean_launch_s / 1e12
    clk = clocks.summary()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clock_peak = (TENSOR_FLOP_PER_CLK_PER_SM * sms * clk["sm_mhz"] * 1e6 / 1e12) if clk.get("sm_mhz") else None
    bytes_in = q.numel() * 2 + k.numel() * 2 + v.numel() * 2
    bytes_out = o.numel() * 2 + lse.numel() * 4
    if bwd:
        bytes_in += o.numel() * 2 + lse.numel() * 4 + do.numel() * 2
        bytes_out = dq.numel() * 2 + dk.numel() * 2 + dv.numel() * 2
    entry = {"fwd": "attn_fwd_ex" if args.dtype == "f16" else "attn_fwd",
             "splitkv": "attn_fwd_splitkv", "bwd": "attn_bwd"}[args.path]

    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * mean_launch_s, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {**w.as_dict(), "parallelism": "replicas" if world > 1 else "single",
                   "entry_point": entry,
                   "workspace_bytes": ws_bytes,
                   "l2": "flushed between steps (256 MiB write); inputs also exceed L2",
                   "metric_flops_per_step": flops, "exact_visible_pair_flops_per_step": exact,
                   "pct_of_peak": 100.0 * value / peak},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": None if bwd else load_traffic(w.name),
                     "peak_source": f"bf16_tflops (burst) of {peak_kind}",
                     "kernel": kernel_name(w, bwd),
                     "algorithmic_unit": ("10*D FLOPs per visible (q-row, key, q-head)" if bwd else
                                          "4*D FLOPs per visible (q-row, key, q-head)"),
                     "clock_matched": {
                         "peak": clock_peak, "frac": (achieved / clock_peak) if clock_peak else None,
                         "unit": "TFLOP/s", "flop_per_clk_per_sm": TENSOR_FLOP_PER_CLK_PER_SM,
                         "sms": sms, "sm_mhz_median": clk.get("sm_mhz"),
                         "note": "tensor pipe at the SM clock sampled during the timed region "
                                 "(one 128x128x16 bf16 MMA per 64 cycles per SM, measured)"}},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": bytes_in,
                "d2h_bytes_per_step": bytes_out, "steps": e2e_steps,
                "pipelining": "two device buffer sets; uploads and downloads on their own streams "
                              "overlap the neighbouring steps' kernels",
                "host_link_gbs": link,
                "step_copies_gbs": step_copy,
                "link_bound": link_bound(link, bytes_in, bytes_out, flops)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "timed_repeats": repeats,
        "timed_steps_total": n_timed,
        "wall_s_timed_region": t_wall,
        "kernel_ms": {"min": min(times_ms), "median": statistics.median(times_ms),
                      "max": max(times_ms)},
    }
    if not bwd and args.dtype == "bf16" and args.path == "fwd" and not args.no_other_workloads:
        line["workloads"] = other_workload_timings(fa, inputs, torch, dev, stream, flush, w.name,
                                                   rank)
    if world == 1 and not args.no_cpu_baseline and not bwd:
        tf, dt, n, cores = oracle_sample_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{n} random query rows of {w.name} "
                                          f"({dt:.1f} s of fp64 oracle work)"}
        line["cpu_baseline"]["other_points"] = cpu_reference_points(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def host_link_rates(dev):
    """Pinned host<->device copy rates (GB/s) of this box: one direction at a
    time and both at once, 64 MiB per copy, best of three."""
    import torch
    n = 64 << 20
    h_in = torch.empty(n, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(n, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(n, dtype=torch.uint8, device=dev)
    d_out = torch.empty(n, dtype=torch.uint8, device=dev)
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    res = {}
    for name in ("h2d", "d2h", "both"):
        best = 0.0
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if name in ("h2d", "both"):
                with torch.cuda.stream(s_up):
                    d_in.copy_(h_in, non_blocking=True)
            if name in ("d2h", "both"):
                with torch.cuda.stream(s_down):
                    h_out.copy_(d_out, non_blocking=True)
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
            best = max(best, (2 if name == "both" else 1) * n / dt / 1e9)
        res[name] = best
    return res


def link_bound(link, bytes_in, bytes_out, flops):
    """Throughput bound of the e2e step by the host link alone: every step's
    uploads and downloads at the measured rates (directions overlapped)."""
    t = max(bytes_in / (link["h2d"] * 1e9), bytes_out / (link["d2h"] * 1e9),
            (bytes_in + bytes_out) / (link["both"] * 1e9))
    return {"min_ms_per_step": 1e3 * t, "max_tflops": flops / t / 1e12}


def other_workload_timings(fa, inputs, torch, dev, stream, flush, headline: str, rank: int,
                           warmup: int = 3, steps: int = 10):
    """Kernel-only attn_fwd throughput of the other benchmark shapes (same
    timing rules as the headline: events on the launching stream, L2 flushed
    between steps, inputs resident in HBM)."""
    import numpy as np
    out = {}
    for name in OTHER_WORKLOADS:
        if name == headline:
            continue
        w = inputs.WORKLOADS[name]
        q_h, k_h, v_h = inputs.make_workload(w, seed=rank)

        def dev_t(bits):
            return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

        q, k, v = dev_t(q_h), dev_t(k_h), dev_t(v_h)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        sh = stream.cuda_stream
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(warmup + steps):
            flush.zero_()
            if i >= warmup:
                ev[i - warmup][0].record(stream)
            st = fa.attn_fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, w.causal,
                                 w.scale, sh)
            if st != fa.ATTN_OK:
                raise fa.AttnError(st, "attn_fwd")
            if i >= warmup:
                ev[i - warmup][1].record(stream)
        torch.cuda.synchronize(dev)
        if fa.attn_check_device_status(stream) != fa.ATTN_OK:
            raise RuntimeError(f"device status not OK after {name}")
        ms = [a.elapsed_time(b) for a, b in ev]
        mean_s = sum(ms) / len(ms) / 1e3
        out[name] = {"value": metric_flops(w) / mean_s / 1e12,
                     "exact_tflops": exact_flops(w) / mean_s / 1e12,
                     "ms_per_step": 1e3 * mean_s, "steps": steps, "warmup": warmup,
                     "entry_point": "attn_fwd"}
        del q, k, v, o, lse
    return out


def cpu_reference_points(w, target_s: float):
    """Second CPU reference points: the oracle on one core for the tiny and the
    headline shapes (larger shapes' one-core figures would be extrapolations),
    and numpy fp64 (BLAS) on one (batch, head) slice of the workload."""
    from attention_forward_11_gb300 import inputs
    pts = {}
    for name in ("tiny_causal", "mha_causal_4x16x4096"):
        tf, dt, n, cores = oracle_one_core(name, min(target_s, 6.0))
        pts[f"oracle_1core_{name}"] = {"value": tf, "unit": UNIT, "cores": cores,
                                       "sample": f"{n} random query rows ({dt:.1f} s)"}
    tf, dt = numpy_fp64_rate(w)
    pts["numpy_fp64_blas"] = {"value": tf, "unit": UNIT, "cores": os.cpu_count(),
                              "sample": f"one (batch, head) slice of {w.name}: {w.Sq} x {w.Skv} "
                                        f"dense masked logits ({dt:.2f} s)"}
    del inputs
    return pts


SWEEP_SHAPES = [(1, hq, hkv, sq, skv) for (hq, hkv) in ((8, 1), (64, 8), (32, 8), (16, 16))
                for sq in (1, 128, 512, 1024, 2048) for skv in (8192, 32768, 131072)] + [
    (4, 32, 8, 128, 32768), (4, 64, 8, 512, 32768), (2, 16, 16, 1024, 65536), (8, 8, 1, 1, 32768),
    (2, 8, 8, 256, 16384)]


def splitkv_sweep(args):
    """attn_fwd against attn_fwd_splitkv (the planner's own choice, with the
    workspace it asks for) on few-tile shapes: bottom-right causal, D = 128,
    seeded normal inputs made on the device (timing only; parity is the tests'
    job).  One JSON line per shape: median of `--steps` launches each, L2 flushed
    between launches."""
    import torch
    import attention_forward_11_gb300 as fa
    from attention_forward_11_gb300 import build as libbuild
    libbuild.build()
    fa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    gen = torch.Generator(device=dev)
    D = 128

    def median_ms(fn):
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    for (B, Hq, Hkv, Sq, Skv) in SWEEP_SHAPES:
        gen.manual_seed(B * 7 + Hq + Sq + Skv)
        q = torch.randn(B, Sq, Hq, D, device=dev, generator=gen).to(torch.bfloat16)
        k = torch.randn(B, Skv, Hkv, D, device=dev, generator=gen).to(torch.bfloat16)
        v = torch.randn(B, Skv, Hkv, D, device=dev, generator=gen).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=dev)
        ws_n = fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, 1)
        ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)
        sc = 1.0 / math.sqrt(D)

        def plain():
            st = fa.attn_fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 B, Sq, Skv, Hq, Hkv, D, 1, sc, sh)
            if st != fa.ATTN_OK:
                raise fa.AttnError(st, "attn_fwd")

        def split():
            st = fa.attn_fwd_splitkv_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, Sq, Skv, Hq, Hkv, D, 1, sc, ws.data_ptr(),
                                         ws_n, sh)
            if st != fa.ATTN_OK:
                raise fa.AttnError(st, "attn_fwd_splitkv")

        tp, ts = median_ms(plain), median_ms(split)
        if fa.attn_check_device_status(stream) != fa.ATTN_OK:
            raise RuntimeError("device status not OK in the split-KV sweep")
        w = type("W", (), dict(B=B, Hq=Hq, Sq=Sq, Skv=Skv, D=D, causal=1))
        fl = exact_flops(w)
        print(json.dumps({"B": B, "Hq": Hq, "Hkv": Hkv, "Sq": Sq, "Skv": Skv, "D": D, "causal": 1,
                          "split": ws_n > 0, "workspace_bytes": ws_n, "attn_fwd_ms": tp,
                          "attn_fwd_splitkv_ms": ts, "attn_fwd_tflops": fl / tp / 1e9,
                          "attn_fwd_splitkv_tflops": fl / ts / 1e9, "gain": tp / ts}), flush=True)
        del q, k, v, o, lse, ws


def main():
    from attention_forward_11_gb300 import inputs
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the kernel-only timings of the other benchmark shapes")
    ap.add_argument("--min-timed-seconds", type=float, default=1.0,
                    help="repeat the K-step block until the timed region spans this long")
    ap.add_argument("--splitkv-sweep", action="store_true",
                    help="time attn_fwd against attn_fwd_splitkv on few-tile shapes (one JSON "
                         "line per shape) instead of the benchmark")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16",
                    help="element type of Q, K, V, O (f16 goes through attn_fwd_ex)")
    ap.add_argument("--path", choices=["fwd", "splitkv", "bwd"], default="fwd",
                    help="entry point timed: attn_fwd, attn_fwd_splitkv with its workspace, or "
                         "attn_bwd (one step = the backward of one forward)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.dtype == "f16" and args.path == "splitkv":
        ap.error("the split-KV entry points take bf16")
    w = inputs.WORKLOADS[args.workload]
    if args.splitkv_sweep:
        args.steps = min(args.steps, 10)
        splitkv_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
