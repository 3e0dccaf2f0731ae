"""Benchmark of the selective-scan forward on GB300: state-updates/s and roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload KEY] [--op fwd|decode]

A step is one selective-scan forward (one ss_selective_scan_fwd call) over the
workload's synthetic inputs, already resident in HBM.  The default workload is
the largest one-GPU configuration: the sequence sweep shaped like the Blelloch
article's benchmark at its longest length (batch 16, dim 1536, dstate 16,
seqlen 16384, fp32 I/O, silu gate; 6.5 GB of inputs and outputs, far above
the 129 MB L2).  Workloads that fit in L2 rotate over enough input sets to
exceed twice the L2 size, and also report the time with one L2-resident set
("unflushed").

--series seqlen prints one line per length of the sequence sweep
(L = 256, 1024, 4096, 16384): the time-against-seqlen record.

Under torchrun each rank runs the same workload on its own GPU (weak scaling,
no collective on the data path); rank 0 prints one JSON line with the
whole-job throughput measured over the slowest rank.

--impl reference times the CPU oracle (the plain fp64 C implementation the
tests check against) on the host cores, on a bounded sample of the same
workload, and prints the same metric.

--op decode measures the one-token step instead (ss_selective_state_update,
default workload: 64 sequences of a dim-5120, 16-state bf16 layer), with the
state of every call taken from a rotating set larger than twice the L2.

--op bwd measures the backward pass (ss_selective_scan_bwd) on a forward
workload (default: the Mamba-2.8B-shaped layer).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

REPO = Path(__file__).resolve().parent
sys.path.insert(0, str(REPO))

METRIC = "selective-scan fwd state-updates/s (B*D*L*N/s) at 1 GB300; % of roofline"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=40)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="workload key (inputs.WORKLOADS; with --op decode, inputs.DECODE_WORKLOADS)")
    ap.add_argument("--op", choices=["fwd", "decode", "bwd", "mamba2"], default="fwd",
                    help="fwd: the forward scan (default); decode: one token per call; "
                         "bwd: the backward pass; mamba2: the Mamba-2 forward (tensor cores)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--series", choices=["seqlen"], default=None,
                    help="seqlen: one line per length of the sequence sweep (forward only)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-seconds", type=float, default=150.0,
                    help="total CPU time budget of the reference arm's timed steps")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.gpu_id = gpu_id
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[str] = []

    def _query(self, extra=()):
        return ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                "--format=csv,noheader,nounits", *extra]

    def start(self):
        try:
            self.proc = subprocess.Popen(self._query([f"-lms", str(self.period_ms)]),
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        self._reader = threading.Thread(target=self._read, daemon=True)
        if self.proc:
            self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._reader.join(timeout=2)
        samples = list(self.lines)
        if not samples:  # region shorter than one period: one sample right after
            try:
                out = subprocess.run(self._query(), capture_output=True, text=True, timeout=20)
                samples = [l.strip() for l in out.stdout.splitlines() if l.strip()]
            except (FileNotFoundError, OSError, subprocess.TimeoutExpired):
                samples = []
        sm, smax, power, reasons = [], [], [], set()
        for line in samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def gpu_id_for(device_index: int) -> str:
    import torch
    props = torch.cuda.get_device_properties(device_index)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        return s if s.startswith("GPU-") else f"GPU-{s}"
    return str(device_index)


# ---------------------------------------------------------------- peaks
def measured_peaks() -> dict:
    p = REPO / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                    "source": "measured"}
        except (ValueError, KeyError):
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}


def unit_rates() -> dict:
    """Per-clock per-SM rates of MUFU ex2 and FP32 FMA lane-ops (microbenchmarks)."""
    from mamba_selective_scan_ss_gb300 import peaks
    ex2 = peaks.measure("ex2")
    ffma = peaks.measure("ffma2")
    return {"ex2_per_clk_sm": ex2["per_clk_per_sm"], "fp32_per_clk_sm": ffma["per_clk_per_sm"],
            "sms": ex2["sms"], "probe_mhz": ex2["sm_mhz"]}


def traffic_record(kernel_sources: list[Path], workload_name: str):
    """dram bytes per launch from the committed ncu summary, if it matches the source."""
    import hashlib
    h = hashlib.sha256()
    for src in kernel_sources:
        h.update(src.read_bytes())
    digest = h.hexdigest()[:16]
    for f in sorted((REPO / "profiles").glob("*.txt")):
        kv = {}
        for line in f.read_text().splitlines():
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("workload") == workload_name and kv.get("kernel_source_sha256_16") == digest:
            try:
                return float(kv["dram_bytes_per_step"]), f.name
            except (KeyError, ValueError):
                pass
    return None, None


# ---------------------------------------------------------------- oracle leg
def oracle_rate(w, budget_s: float, inp_cpu=None, threads: int | None = None) -> dict:
    """Time the CPU oracle on a bounded sample of the workload (rows subset),
    on every host core (or on `threads` of them)."""
    import oracle
    from mamba_selective_scan_ss_gb300.inputs import make_inputs
    orc = oracle.default()
    inp = inp_cpu if inp_cpu is not None else make_inputs(w)
    cores = threads or os.cpu_count() or 1

    def run(ch):
        sub = {k: v for k, v in inp.items()}
        sub["u"] = inp["u"][:, :ch].contiguous()
        sub["delta"] = inp["delta"][:, :ch].contiguous()
        sub["z"] = inp["z"][:, :ch].contiguous() if inp["z"] is not None else None
        sub["A"] = inp["A"][:ch].contiguous()
        sub["D"] = inp["D"][:ch].contiguous() if inp["D"] is not None else None
        sub["delta_bias"] = inp["delta_bias"][:ch].contiguous() if inp["delta_bias"] is not None else None
        if w.bc_per_channel:
            sub["B"] = inp["B"][:, :ch].contiguous()
            sub["C"] = inp["C"][:, :ch].contiguous()
        t0 = time.perf_counter()
        orc.fwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"], sub["z"],
                sub["delta_bias"], sub["delta_softplus"], dtype=w.dtype, nthreads=cores,
                bc_per_channel=w.bc_per_channel)
        return time.perf_counter() - t0

    probe_ch = min(w.dim, max(1, cores))
    t_probe = run(probe_ch)
    per_ch = t_probe / probe_ch
    ch = int(max(1, min(w.dim, budget_s / max(per_ch, 1e-9))))
    # whole passes over the chosen channels until the budget is spent
    reps, dt = 0, 0.0
    while True:
        dt += run(ch)
        reps += 1
        if dt >= budget_s or (reps >= 1 and dt * (reps + 1) / reps > 2.5 * budget_s):
            break
    upd = w.batch * ch * w.seqlen * w.dstate * reps
    return {"value": upd / dt, "seconds": dt, "channels": ch, "reps": reps, "updates": upd,
            "cores": cores}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle as it stands, on the host cores.

    Every one of the --warmup + --steps steps runs the oracle once on the same
    bounded sample of the workload (the first channels, and if one channel is
    too much the first batch rows, each over the full sequence), sized from one
    probe so that all the steps together take about --reference-seconds."""
    from mamba_selective_scan_ss_gb300.inputs import WORKLOADS, make_inputs
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    import oracle
    oracle.build()
    orc = oracle.default()
    cores = os.cpu_count() or 1

    def run(nb, ch):  # the first nb batch rows and ch channels, the whole sequence
        sub = dict(inp)
        for k in ("u", "delta", "z"):
            if inp[k] is not None:
                sub[k] = inp[k][:nb, :ch].contiguous()
        for k in ("A", "D", "delta_bias"):
            if inp[k] is not None:
                sub[k] = inp[k][:ch].contiguous()
        for k in ("B", "C"):
            sub[k] = (inp[k][:nb, :ch] if w.bc_per_channel else inp[k][:nb]).contiguous()
        t0 = time.perf_counter()
        orc.fwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"], sub["z"],
                sub["delta_bias"], sub["delta_softplus"], dtype=w.dtype, nthreads=cores,
                bc_per_channel=w.bc_per_channel)
        return time.perf_counter() - t0

    row_updates = w.seqlen * w.dstate  # updates of one (batch row, channel)
    probe_ch = min(w.dim, cores)
    per_row = run(w.batch, probe_ch) / (w.batch * probe_ch)  # seconds per (batch row, channel)
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    rows = max(1, int(per_step / max(per_row, 1e-12)))
    ch = max(1, min(w.dim, rows // w.batch))
    nb = w.batch if rows >= w.batch else max(1, rows)
    for _ in range(args.warmup):
        run(nb, ch)
    tot_s = 0.0
    for _ in range(args.steps):
        tot_s += run(nb, ch)
    steps = max(1, args.steps)
    tot_upd = nb * ch * row_updates * steps
    value = tot_upd / max(tot_s, 1e-12)
    sample = (f"the first {nb} of {w.batch} batch rows x the first {ch} of {w.dim} channels, "
              f"full seqlen {w.seqlen}, dstate {w.dstate} ({nb * ch * row_updates} updates) "
              f"per step, {args.warmup} + {args.steps} steps")
    line = {
        "metric": METRIC, "value": value, "unit": "state-updates/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "seqlen": w.seqlen, "io_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": "state-updates/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "state-updates/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch
    import mamba_selective_scan_ss_gb300 as ss
    from mamba_selective_scan_ss_gb300 import _build
    from mamba_selective_scan_ss_gb300.inputs import WORKLOADS, make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the selective scan runs only on the GPU)")
    if rank == 0:
        _build.build_all()
    barrier(world)
    ss.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    nbytes = w.algorithmic_bytes()
    nsets = 1 if nbytes >= 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / nbytes)) + 1
    sets = []
    for _ in range(nsets):
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        y = torch.empty_like(d["u"])
        st = torch.empty((w.batch, w.dim, w.dstate), device=dev, dtype=torch.float32)
        sets.append((d, y, st))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if w.bc_per_channel:  # ss_selective_scan_fwd_pc: one kernel, no chunks
        plan = {"nchunks": 1, "kernel_launches": 1}
    else:
        plan = ss.ss_selective_scan_plan(w.batch, w.dim, w.dstate, w.seqlen,
                                         ss.SS_F32 if w.dtype == "f32" else ss.SS_BF16, True, sms)

    def step(i):
        d, y, st = sets[i % nsets]
        ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                              d["delta_bias"], d["delta_softplus"], y=y, last_state=st,
                              stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize(dev)
    status = ss.ss_selective_scan_check(stream.cuda_stream)
    if status != ss.SS_OK:
        raise SystemExit(f"device status after warm-up: {ss.ss_status_string(status)}")

    rates = unit_rates() if rank == 0 else None
    sampler = ClockSampler(gpu_id_for(dev.index))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    ms_total = ev0.elapsed_time(ev1)
    status = ss.ss_selective_scan_check(stream.cuda_stream)
    if status != ss.SS_OK:
        raise SystemExit(f"device status after timing: {ss.ss_status_string(status)}")
    ms_max = max_over_ranks(ms_total, world)
    ms_step = ms_max / args.steps
    total_updates = w.updates * args.steps * world
    value = total_updates / (ms_max * 1e-3)

    # the same steps on one L2-resident input set (workloads smaller than L2)
    unflushed = None
    if nsets > 1:
        n_u = min(args.steps, 2000)
        with torch.cuda.stream(stream):
            for _ in range(3):
                step(0)
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for _ in range(n_u):
                step(0)
            u1.record(stream)
        torch.cuda.synchronize(dev)
        u_ms = max_over_ranks(u0.elapsed_time(u1), world) / n_u
        unflushed = {"value": w.updates * world / (u_ms * 1e-3), "unit": "state-updates/s",
                     "ms_per_step": u_ms, "steps": n_u,
                     "note": "one input set reused every step: inputs L2-resident"}

    # e2e: pinned host inputs -> device, the call, outputs -> pinned host, every step
    e2e = None
    if args.e2e_steps > 0:
        host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        d, y, st = sets[0]
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        st_host = torch.empty(st.shape, dtype=st.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values()
                  if isinstance(v, torch.Tensor))
        d2h = y_host.numel() * y_host.element_size() + st_host.numel() * st_host.element_size()

        # the C-ABI call on host buffers: it copies the rows in, scans and
        # copies y and last_state out, overlapping copies and scan over
        # segments of the sequence (ss_selective_scan_fwd_host)
        def e2e_step():
            ss.selective_scan_fwd_host(host["u"], host["delta"], host["A"], host["B"],
                                       host["C"], host["D"], host["z"], host["delta_bias"],
                                       host["delta_softplus"], y=y_host, last_state=st_host,
                                       stream=stream)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        e2e = {"value": w.updates * args.e2e_steps * world / (e_ms * 1e-3),
               "unit": "state-updates/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms / args.e2e_steps}

    if rank != 0:
        return
    # roofline of one step (all kernels of one call): slowest of HBM bytes, MUFU
    # exps and FP32 lane-ops, at the SM clock sampled during the timed region
    pk = measured_peaks()
    mhz = clocks["sm_mhz"] or rates["probe_mhz"]
    r_sfu = rates["ex2_per_clk_sm"] * rates["sms"] * mhz * 1e6         # ex2 / s
    r_fp32 = rates["fp32_per_clk_sm"] * rates["sms"] * mhz * 1e6       # lane-ops / s
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_sfu = w.updates / r_sfu
    t_fp32 = 4 * w.updates / r_fp32
    t_step = ms_step * 1e-3 / world * world  # per-rank step time
    srcs = (("ss_pc.cuh", "ss_device.cuh", "ss_api.cu") if w.bc_per_channel else
            ("ss_fwd.cuh", "ss_sched.cuh", "ss_device.cuh", "ss_api.cu"))
    kernel_src = [REPO / "mamba_selective_scan_ss_gb300" / "csrc" / f for f in srcs]
    traffic, traffic_src = traffic_record(kernel_src, w.name)
    if t_hbm >= max(t_sfu, t_fp32):
        achieved = nbytes / t_step / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"]}
    else:
        alu_peak = min(r_sfu, r_fp32 / 4)
        achieved = w.updates / t_step
        roof = {"bound": "alu", "achieved": achieved / 1e9, "peak": alu_peak / 1e9,
                "unit": "Gupdate/s", "frac": achieved / alu_peak,
                "peak_source": (f"microbenchmarks: {rates['ex2_per_clk_sm']:.1f} ex2 and "
                                f"{rates['fp32_per_clk_sm']:.1f} fp32 lane-ops /clk/SM x "
                                f"{rates['sms']} SMs x {mhz:.0f} MHz sampled")}
    roof.update({"traffic": traffic, "traffic_source": traffic_src,
                 "algorithmic_bytes_per_step": nbytes, "updates_per_step": w.updates,
                 "t_hbm_us": t_hbm * 1e6, "t_sfu_us": t_sfu * 1e6, "t_fp32_us": t_fp32 * 1e6,
                 "measured_step_us": t_step * 1e6,
                 "scope": (f"one ss_selective_scan_fwd{'_pc' if w.bc_per_channel else ''} call"
                           f" = {plan['kernel_launches']} kernel(s)")})

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r = oracle_rate(w, args.cpu_baseline_seconds, inp)
        cpu = {"value": r["value"], "unit": "state-updates/s", "cores": r["cores"],
               "kind": "oracle",
               "sample": (f"{r['reps']} pass(es) over the first {r['channels']} of {w.dim} "
                          f"channels of every batch row, full seqlen {w.seqlen}, dstate "
                          f"{w.dstate}: {r['updates']} updates in {r['seconds']:.1f} s")}
        r1 = oracle_rate(w, min(5.0, args.cpu_baseline_seconds), inp, threads=1)
        cpu["single_core"] = {"value": r1["value"], "cores": 1,
                              "sample": f"{r1['updates']} updates in {r1['seconds']:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": "state-updates/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "compute_dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "seqlen": w.seqlen, "io_dtype": w.dtype, "z_gate": w.has_z,
                   "l2": (f"{nsets} rotating input sets ({nsets * nbytes / 2**20:.0f} MiB > 2x L2)"
                          if nsets > 1 else "inputs larger than 2x L2"),
                   "nchunks": plan["nchunks"], "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "unflushed": unflushed,
        "gpu_launches": int(plan["kernel_launches"] * args.steps),
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- decode step
DECODE_METRIC = "selective-scan decode state-updates/s (B*D*N per token) at 1 GB300; % of roofline"


def run_decode(args, world, rank, local):
    """One token per call (ss_selective_state_update): the state of each call is
    a different buffer of a rotating set larger than 2x L2, as in a stack of
    layers, so every call reads and writes its state in HBM."""
    import torch
    import mamba_selective_scan_ss_gb300 as ss
    from mamba_selective_scan_ss_gb300 import _build
    from mamba_selective_scan_ss_gb300.inputs import DECODE_WORKLOADS, make_decode_inputs

    w = DECODE_WORKLOADS[args.workload]
    inp = make_decode_inputs(w)
    if args.impl == "reference":
        if rank == 0:
            r = decode_oracle_rate(w, inp, max(0.5, args.reference_seconds / 10))
            print(json.dumps({
                "metric": DECODE_METRIC, "value": r["value"], "unit": "state-updates/s",
                "n_gpus": args.gpus, "steps": r["reps"], "warmup": 0,
                "ms_per_step": 1e3 * r["seconds"] / r["reps"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "impl": "reference", "op": "decode",
                "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                           "io_dtype": w.dtype},
                "cpu_baseline": {"value": r["value"], "unit": "state-updates/s",
                                 "cores": r["cores"], "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "state-updates/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the selective scan runs only on the GPU)")
    if rank == 0:
        _build.build_all()
    barrier(world)
    ss.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    nbytes = w.algorithmic_bytes()
    nsets = int(math.ceil(2 * L2_BYTES / nbytes)) + 1
    shared = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v)
              for k, v in inp.items() if k in ("A", "D", "dt_bias")}
    sets = []
    for _ in range(nsets):
        d = {k: v.to(dev) for k, v in inp.items()
             if isinstance(v, torch.Tensor) and k not in shared}
        d.update(shared)
        d["y"] = torch.empty_like(d["x"])
        sets.append(d)

    def step(i):
        d = sets[i % nsets]
        ss.selective_state_update(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                  d.get("z"), d["dt_bias"], True, y=d["y"], stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_id_for(dev.index))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    ms_max = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_max / args.steps
    value = w.updates * args.steps * world / (ms_max * 1e-3)

    # e2e: the token's inputs from pinned host memory, y back to it; the state
    # stays resident on the device between tokens, as in serving
    e2e = None
    if args.e2e_steps > 0:
        d = sets[0]
        keys = [k for k in ("x", "dt", "B", "C", "z") if d.get(k) is not None]
        host = {k: inp[k].pin_memory() for k in keys}
        y_host = torch.empty(d["y"].shape, dtype=d["y"].dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = y_host.numel() * y_host.element_size()

        def e2e_step():
            with torch.cuda.stream(stream):
                for k, v in host.items():
                    d[k].copy_(v, non_blocking=True)
                ss.selective_state_update(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"],
                                          d["D"], d.get("z"), d["dt_bias"], True, y=d["y"],
                                          stream=stream)
                y_host.copy_(d["y"], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        e2e = {"value": w.updates * args.e2e_steps * world / (e_ms * 1e-3),
               "unit": "state-updates/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms / args.e2e_steps}
    if rank != 0:
        return
    pk = measured_peaks()
    rates = unit_rates()
    mhz = clocks["sm_mhz"] or rates["probe_mhz"]
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_sfu = w.updates / (rates["ex2_per_clk_sm"] * rates["sms"] * mhz * 1e6)
    t_step = ms_step * 1e-3
    kernel_src = [REPO / "mamba_selective_scan_ss_gb300" / "csrc" / f
                  for f in ("ss_decode.cuh", "ss_device.cuh", "ss_api.cu")]
    traffic, traffic_src = traffic_record(kernel_src, w.name)
    achieved = nbytes / t_step / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"],
            "traffic": traffic, "traffic_source": traffic_src,
            "algorithmic_bytes_per_step": nbytes, "updates_per_step": w.updates,
            "t_hbm_us": t_hbm * 1e6, "t_sfu_us": t_sfu * 1e6, "measured_step_us": t_step * 1e6,
            "scope": "one ss_selective_state_update call = 1 kernel"}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r = decode_oracle_rate(w, inp, min(args.cpu_baseline_seconds, 4.0))
        cpu = {"value": r["value"], "unit": "state-updates/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"]}
    print(json.dumps({
        "metric": DECODE_METRIC, "value": value, "unit": "state-updates/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "compute_dtype": "f32", "data": "synthetic", "op": "decode",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "io_dtype": w.dtype, "z_gate": w.has_z,
                   "l2": f"{nsets} rotating state sets ({nsets * nbytes / 2**20:.0f} MiB > 2x L2)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(args.steps), "clocks": clocks, "wall_s_timed_region": t_wall,
    }), flush=True)


BWD_METRIC = "selective-scan bwd state-updates/s (B*D*L*N/s) at 1 GB300; % of roofline"
# algorithmic work of the backward per state update: one forward recompute
# (1 ex2, 2 FP32 lane-ops) and the reverse step (1 ex2, 10 FP32 lane-ops: the
# g update and the dC, dB, dA, d(dt) and du terms)
BWD_EX2_PER_UPDATE, BWD_FP32_PER_UPDATE = 2, 12


def run_bwd(args, world, rank, local):
    """The backward on a forward workload: inputs and dy resident in HBM."""
    import torch
    import mamba_selective_scan_ss_gb300 as ss
    from mamba_selective_scan_ss_gb300 import _build
    from mamba_selective_scan_ss_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[args.workload]
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the selective scan runs only on the GPU)")
    if rank == 0:
        _build.build_all()
    barrier(world)
    ss.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    inp = make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = torch.Generator().manual_seed(w.seed + 1000)
    dy = torch.randn(d["u"].shape, generator=g).to(d["u"].dtype).to(dev)
    elt = w.elt
    x_bytes = w.batch * w.dim * w.seqlen * elt
    # u, delta, dy (+ z) read once; du, ddelta (+ dz) written once
    nbytes = (3 + int(w.has_z)) * x_bytes + (2 + int(w.has_z)) * x_bytes
    nbytes += 2 * w.batch * w.dstate * w.seqlen * (elt + 4)          # B, C in; dB, dC out (fp32)
    nbytes += 2 * 4 * w.dim * w.dstate + 4 * 4 * w.dim               # A, dA; D, bias, dD, dbias

    def step():
        return ss.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                     d["delta_bias"], d["delta_softplus"], dy=dy, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_id_for(dev.index))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    ms_max = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_max / args.steps
    value = w.updates * args.steps * world / (ms_max * 1e-3)

    # e2e: the forward's inputs and dy from pinned host memory, every gradient
    # back to pinned host memory, every step
    e2e = None
    if args.e2e_steps > 0:
        host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        dy_host = dy.cpu().pin_memory()
        dy_dev = torch.empty_like(dy)
        with torch.cuda.stream(stream):
            probe = step()
        torch.cuda.synchronize(dev)
        g_host = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                  for k, v in probe.items() if v is not None}
        del probe
        h2d = sum(v.numel() * v.element_size() for v in host.values()
                  if isinstance(v, torch.Tensor)) + dy_host.numel() * dy_host.element_size()
        d2h = sum(v.numel() * v.element_size() for v in g_host.values())

        def e2e_step():
            with torch.cuda.stream(stream):
                for k, v in host.items():
                    if isinstance(v, torch.Tensor):
                        d[k].copy_(v, non_blocking=True)
                dy_dev.copy_(dy_host, non_blocking=True)
                got = ss.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                            d["z"], d["delta_bias"], d["delta_softplus"],
                                            dy=dy_dev, stream=stream)
                for k, v in g_host.items():
                    v.copy_(got[k], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        e2e = {"value": w.updates * args.e2e_steps * world / (e_ms * 1e-3),
               "unit": "state-updates/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms / args.e2e_steps}

    if rank != 0:
        return
    pk = measured_peaks()
    rates = unit_rates()
    mhz = clocks["sm_mhz"] or rates["probe_mhz"]
    r_sfu = rates["ex2_per_clk_sm"] * rates["sms"] * mhz * 1e6
    r_fp32 = rates["fp32_per_clk_sm"] * rates["sms"] * mhz * 1e6
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_sfu = BWD_EX2_PER_UPDATE * w.updates / r_sfu
    t_fp32 = BWD_FP32_PER_UPDATE * w.updates / r_fp32
    t_step = ms_step * 1e-3
    if t_hbm >= max(t_sfu, t_fp32):
        achieved = nbytes / t_step / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"]}
    else:
        alu_peak = w.updates / max(t_sfu, t_fp32)
        roof = {"bound": "alu", "achieved": w.updates / t_step / 1e9, "peak": alu_peak / 1e9,
                "unit": "Gupdate/s", "frac": max(t_sfu, t_fp32) / t_step,
                "peak_source": (f"{BWD_EX2_PER_UPDATE} ex2 and {BWD_FP32_PER_UPDATE} fp32 "
                                f"lane-ops per update at the probes' {rates['ex2_per_clk_sm']:.1f} "
                                f"and {rates['fp32_per_clk_sm']:.1f} /clk/SM x {rates['sms']} SMs "
                                f"x {mhz:.0f} MHz sampled")}
    kernel_src = [REPO / "mamba_selective_scan_ss_gb300" / "csrc" / f
                  for f in ("ss_bwd.cuh", "ss_device.cuh", "ss_api.cu")]
    traffic, traffic_src = traffic_record(kernel_src, w.name)
    roof.update({"traffic": traffic, "traffic_source": traffic_src,
                 "traffic_scope": "ss_bwd_main, the call's dominant kernel",
                 "algorithmic_bytes_per_step": nbytes,
                 "updates_per_step": w.updates, "t_hbm_us": t_hbm * 1e6,
                 "t_sfu_us": t_sfu * 1e6, "t_fp32_us": t_fp32 * 1e6,
                 "measured_step_us": t_step * 1e6,
                 "scope": "one ss_selective_scan_bwd call = 3 kernels"})
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = bwd_oracle_rate(w, inp, dy.cpu(), min(args.cpu_baseline_seconds, 8.0))
    print(json.dumps({
        "metric": BWD_METRIC, "value": value, "unit": "state-updates/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "compute_dtype": "f32", "data": "synthetic", "op": "bwd",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "seqlen": w.seqlen, "io_dtype": w.dtype, "z_gate": w.has_z,
                   "l2": "inputs larger than L2" if 4 * x_bytes > 2 * L2_BYTES else
                         "inputs partly L2-resident between calls",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 3 * args.steps, "clocks": clocks, "wall_s_timed_region": t_wall,
    }), flush=True)


def bwd_oracle_rate(w, inp, dy, budget_s: float) -> dict:
    """The oracle's backward on the first channels of every batch row, repeated."""
    import oracle

    orc = oracle.default()
    ch = max(1, min(w.dim, int(4e6 // max(1, w.batch * w.seqlen * w.dstate))))
    sub = {k: (v[:, :ch].contiguous() if k in ("u", "delta", "z") and v is not None else v)
           for k, v in inp.items()}
    sub["A"] = inp["A"][:ch].contiguous()
    sub["D"] = None if inp["D"] is None else inp["D"][:ch].contiguous()
    sub["delta_bias"] = None if inp["delta_bias"] is None else inp["delta_bias"][:ch].contiguous()
    dys = dy[:, :ch].contiguous()
    cores = os.cpu_count() or 1
    reps, t0 = 0, time.perf_counter()
    while True:
        orc.bwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"], sub["z"],
                sub["delta_bias"], sub["delta_softplus"], dy=dys, dtype=w.dtype, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    upd = w.batch * ch * w.seqlen * w.dstate
    return {"value": upd * reps / el, "unit": "state-updates/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} backward pass(es) over the first {ch} of {w.dim} channels of every "
                      f"batch row, full seqlen {w.seqlen}: {upd} updates each, {el:.1f} s"}


def decode_oracle_rate(w, inp, budget_s: float) -> dict:
    """The oracle's one-step forward from the state, repeated for about budget_s."""
    import oracle

    orc = oracle.default()

    def col(v):
        return None if v is None else v.unsqueeze(-1).contiguous()

    args = (col(inp["x"]), col(inp["dt"]), inp["A"], col(inp["B"]), col(inp["C"]), inp["D"],
            col(inp["z"]), inp["dt_bias"], True)
    h0 = inp["state"].double().numpy()
    cores = os.cpu_count() or 1
    reps, t0 = 0, time.perf_counter()
    while True:
        orc.fwd(*args, h0=h0, dtype=w.dtype, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": w.updates * reps / el, "reps": reps, "seconds": el, "cores": cores,
            "sample": f"{reps} full decode step(s) of the workload ({w.updates} updates each) "
                      f"in {el:.1f} s"}


M2_METRIC = "Mamba-2 fwd state-updates/s (B*L*H*P*N/s) at 1 GB300; % of roofline"
M2_CHUNK = 128  # steps per chunk of the kernel (the tensor-core MMA's M)


def m2_oracle_rate(w, inp, budget_s: float) -> dict:
    """The oracle's Mamba-2 forward on the first heads of every batch row, repeated."""
    import oracle

    orc = oracle.default()
    per_head = w.batch * w.seqlen * w.headdim * w.dstate
    hpg = w.nheads // w.ngroups
    heads = min(w.nheads, max(1, int(4e8 // per_head)))
    if heads >= hpg:
        heads -= heads % hpg  # whole groups, so the sub-problem maps heads to the same groups
    groups = max(1, heads // hpg)
    sub = {"x": inp["x"][:, :, :heads].contiguous(), "dt": inp["dt"][:, :, :heads].contiguous(),
           "A": inp["A"][:heads].contiguous(),
           "B": inp["B"][:, :, :groups].contiguous(), "C": inp["C"][:, :, :groups].contiguous(),
           "D": None if inp["D"] is None else inp["D"][:heads].contiguous(),
           "dt_bias": None if inp["dt_bias"] is None else inp["dt_bias"][:heads].contiguous()}
    cores = os.cpu_count() or 1
    reps, t0 = 0, time.perf_counter()
    while True:
        orc.ssd(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"], sub["dt_bias"], True,
                dtype=w.dtype, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    upd = per_head * heads
    return {"value": upd * reps / el, "reps": reps, "seconds": el,
            "cores": min(cores, w.batch * heads),
            "sample": f"{reps} pass(es) over the first {heads} of {w.nheads} heads of every batch "
                      f"row, full seqlen {w.seqlen}: {upd} updates each, {el:.1f} s"}


def run_mamba2(args, world, rank, local):
    """The Mamba-2 forward (ss_mamba2_fwd, one kernel per call on the tensor
    cores); inputs resident in HBM and larger than 2x L2."""
    import torch
    import mamba_selective_scan_ss_gb300 as ss
    from mamba_selective_scan_ss_gb300 import _build
    from mamba_selective_scan_ss_gb300.inputs import MAMBA2_WORKLOADS, make_mamba2_inputs

    w = MAMBA2_WORKLOADS[args.workload]
    inp = make_mamba2_inputs(w)
    config = {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
              "headdim": w.headdim, "ngroups": w.ngroups, "dstate": w.dstate,
              "io_dtype": w.dtype, "chunk": M2_CHUNK}
    if args.impl == "reference":
        if rank == 0:
            r = m2_oracle_rate(w, inp, max(1.0, args.reference_seconds / 10))
            print(json.dumps({
                "metric": M2_METRIC, "value": r["value"], "unit": "state-updates/s",
                "n_gpus": args.gpus, "steps": r["reps"], "warmup": 0,
                "ms_per_step": 1e3 * r["seconds"] / r["reps"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "impl": "reference", "op": "mamba2", "config": config,
                "cpu_baseline": {"value": r["value"], "unit": "state-updates/s",
                                 "cores": r["cores"], "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "state-updates/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the Mamba-2 forward runs only on the GPU)")
    if rank == 0:
        _build.build_all()
    barrier(world)
    ss.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    fs = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), device=dev, dtype=torch.float32)
    nbytes = w.algorithmic_bytes()
    flops = w.chunk_flops(M2_CHUNK)

    def step():
        ss.mamba2_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], True,
                      y=y, final_state=fs, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_id_for(dev.index))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    if ss.ss_selective_scan_check(stream.cuda_stream) != ss.SS_OK:
        raise SystemExit("bench.py: the Mamba-2 kernel reported a device-side error")
    ms_max = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_max / args.steps
    value = w.updates * args.steps * world / (ms_max * 1e-3)

    e2e = None
    if args.e2e_steps > 0:
        keys = ["x", "dt", "B", "C"]
        host = {k: inp[k].pin_memory() for k in keys}
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = y_host.numel() * y_host.element_size()

        def e2e_step():
            with torch.cuda.stream(stream):
                for k, v in host.items():
                    d[k].copy_(v, non_blocking=True)
                ss.mamba2_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], True,
                              y=y, final_state=fs, stream=stream)
                y_host.copy_(y, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        e2e = {"value": w.updates * args.e2e_steps * world / (e_ms * 1e-3),
               "unit": "state-updates/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms / args.e2e_steps}
    if rank != 0:
        return
    pk = measured_peaks()
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    t_step = ms_step * 1e-3
    kernel_src = [REPO / "mamba_selective_scan_ss_gb300" / "csrc" / f
                  for f in ("ss_ssd.cuh", "ss_device.cuh", "ss_api.cu")]
    traffic, traffic_src = traffic_record(kernel_src, w.name)
    if t_hbm >= t_tc:
        achieved = nbytes / t_step / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"]}
    else:
        achieved = flops / t_step / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                "peak_source": pk["source"] + " bf16 burst"}
    roof.update({"traffic": traffic, "traffic_source": traffic_src,
                 "algorithmic_bytes_per_step": nbytes, "chunk_flops_per_step": flops,
                 "tensor_tflops_achieved": flops / t_step / 1e12,
                 "updates_per_step": w.updates, "t_hbm_us": t_hbm * 1e6,
                 "t_tensor_us": t_tc * 1e6, "measured_step_us": t_step * 1e6,
                 "scope": "one ss_mamba2_fwd call = 1 kernel"})
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r = m2_oracle_rate(w, inp, min(args.cpu_baseline_seconds, 10.0))
        cpu = {"value": r["value"], "unit": "state-updates/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"]}
    in_bytes = nbytes // 2  # x, dt, B, C: about half of the call's traffic
    config["l2"] = ("inputs larger than L2" if in_bytes > L2_BYTES else
                    "inputs partly L2-resident between calls")
    config["parallelism"] = f"replicas x{world}"
    print(json.dumps({
        "metric": M2_METRIC, "value": value, "unit": "state-updates/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "op": "mamba2", "config": config,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(args.steps), "clocks": clocks, "wall_s_timed_region": t_wall,
    }), flush=True)


def main():
    args = parse_args()
    if args.workload is None:
        args.workload = {"decode": "decode_64", "bwd": "2",
                         "mamba2": "m2_2.7b"}.get(args.op, "4_16384")
    world, rank, local = dist_setup(args)
    try:
        if args.op == "decode":
            run_decode(args, world, rank, local)
        elif args.op == "mamba2":
            run_mamba2(args, world, rank, local)
        elif args.op == "bwd":
            if args.impl == "reference":
                raise SystemExit("bench.py: --op bwd has no reference arm; its cpu_baseline "
                                 "times the oracle's backward")
            run_bwd(args, world, rank, local)
        elif args.impl == "reference":
            run_reference(args, world, rank)
        elif args.series == "seqlen":
            for key in ("4_256", "4_1024", "4_4096", "4_16384"):
                args.workload = key
                run_ours(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
