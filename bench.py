"""Benchmark of the fused GEMM + reduce-scatter on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the whole hot path: one fused-kernel call that computes
Y = sum_r (alpha*A_r*B_r + beta*C) over one batch of synthetic inputs.  By default
the workload is ffn_w8_m8192_bias, the largest of the five: W = 8 logical ranks,
M = N = 8192, K = 28672 (3584 per rank), alpha = 0.5, beta = 1 with a bf16 C,
bf16 inputs, bf16 Y.  --workload picks another (ffn_w8_m4096, ffn_w4_m16384_x20,
decode_w8_m64, tiny_w2).  Inputs are seeded and synthetic (see
tensor_gemm_reduce_tcgen05_gb300/inputs.py) and stay resident in HBM during the
timed region.  A + B (940 MB) plus the partial workspace (2.1 GB) are larger
than the 129 MB L2, so no L2 flush is needed between steps.

The timed region is exactly --steps calls.  Right after it, the same calls run
back to back for at least --sustain-seconds (the "sustained" figures): long
enough for the 200 ms clock sampler to see the SM clock the kernel runs at once
the board sits at its power cap.

Rank 0 prints one JSON line.  It has the metric (fused TFLOP/s, whole job), the
kernel's roofline fraction, the end-to-end figure through the public API with
host<->device copies in the timed region, the unfused same-GPU baseline
(batched cuBLAS per-rank GEMMs, then the library's separate reduce kernel), a
full-K GEMM for context, the clear-kernel-sync ablation, the oracle timed on
the host cores (cpu_baseline), and the SM clocks sampled during the run.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU.
The path has no cross-GPU exchange here, so there are no collectives on the
data path.  Timing is the max over ranks.

--impl reference times the CPU oracle (the only reference this path has) on a
bounded row sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+RS TFLOP/s and % of GB300 bf16 tensor peak vs unfused, 1 GPU"
# gemm_rs_set_reduce_mode codes (include/gemm_rs.h)
REDUCE_MODES = {"chain": 0, "last_arriver": 1, "two_level": 2}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 256 * 1024 * 1024  # written between calls to push earlier data out of L2


# --------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Max of a float over all ranks (identity at world size 1)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed / the slowest rank's time."""
    return units_per_rank * world / max_seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


# The device code of the fused kernels: a recorded ncu traffic figure is valid
# only for the source it was taken on (host-side heuristics enter through the
# plan, which is recorded beside it).
KERNEL_SOURCES = ("gemm_rs_kernel.cuh", "ptx.cuh", "schedule.cuh")


AG_KERNEL_SOURCES = ("ag_gemm_kernel.cuh", "gemm_rs_kernel.cuh", "ptx.cuh")


def code_only(text: str) -> str:
    """C/C++ source with its comments removed and each line's whitespace
    trimmed (blank lines dropped): what the compiler sees of the code, so that
    editing a comment does not change a kernel's identity.  String and
    character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = (line.strip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    """Identity of the kernels' code (comments and layout whitespace ignored)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_gemm_reduce_tcgen05_gb300", "csrc")
    for name in sources:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def plan_key(plan) -> str:
    if "slices" in plan:  # the AG+GEMM plan
        return "grid={grid} stages={stages} slice_rows={slice_rows} slices={slices}".format(**plan)
    return ("bm={bm} bn={bn} colgroup={colgroup} rowgroup={rowgroup} rank_order={rank_order} "
            "reduce_mode={reduce_mode}").format(**plan)


def kernel_name(plan) -> str:
    """The kernel a plan launches: the CTA-pair kernel for 256-row tiles."""
    return "gemm_rs_pair_kernel" if plan["bm"] == 256 else "gemm_rs_fused_kernel"


def recorded_traffic(kernel: str, workload: str, plan, sources=KERNEL_SOURCES):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    if that summary was taken on the current kernel source and the same plan."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_sha256:\s*([0-9a-f]+)\s+plan:\s*([^\n]+)",
                  text)
    if not m or m.group(2) != kernel_source_hash(sources) or m.group(3).strip() != plan_key(plan):
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while active."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in loaded if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        power = [num(r[3]) for r in loaded if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(power) if power else None}


def algorithmic_bytes(w) -> int:
    """Compulsory bytes of one call: A + B (+ C once per rank when beta != 0) + Y,
    plus the reduce-scatter exchange through the workspace: (W-1)*M*N fp32
    partials written and read back."""
    a = w.W * w.M * w.Kpr * 2
    b = w.W * w.Kpr * w.N * 2
    c = w.W * w.M * w.N * 2 if w.beta != 0 else 0
    y = w.M * w.N * (2 if w.y_dtype == "bf16" else 4)
    ex = 2 * (w.W - 1) * w.M * w.N * 4
    return a + b + c + y + ex


def oracle_sample(w, A, B, C, rows_wanted: int, threads: int):
    """Time the oracle on `rows_wanted` evenly spread rows.  Returns (seconds, rows)."""
    import oracle
    from tensor_gemm_reduce_tcgen05_gb300.inputs import bf16_bits
    step = max(1, w.M // max(1, rows_wanted))
    rows = list(range(0, w.M, step))[:rows_wanted]
    Ab, Bb = bf16_bits(A), bf16_bits(B)
    Cb = None if C is None else bf16_bits(C)
    t0 = time.perf_counter()
    oracle.gemm_rs(Ab, Bb, Cb, w.alpha, w.beta, w.y_dtype, rows=rows, threads=threads)
    return time.perf_counter() - t0, len(rows)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: implementer
    and part numbers), else the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = (x.strip() for x in line.split(":", 1))
                    fields.setdefault(k, v)
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("CPU implementer"):
        return (f"{platform.machine()} implementer {fields['CPU implementer']} "
                f"part {fields.get('CPU part', '?')}")
    return platform.machine() or "unknown"


def calibrate_rows(w, A, B, C, threads: int, target_s: float):
    """Rows per oracle sample such that one sample takes about target_s seconds."""
    t, n = oracle_sample(w, A, B, C, threads, threads)
    per_row = t / n
    rows = max(threads, int(target_s / per_row) // threads * threads)
    return min(rows, w.M), per_row


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from tensor_gemm_reduce_tcgen05_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[args.workload]
    A, B, C = workload_inputs(w)
    cores = host_cores()
    # Each step is a bounded row sample (about 2 s), so that warm-up + steps end
    # within a few minutes.
    rows, _ = calibrate_rows(w, A, B, C, cores, target_s=2.0)
    for _ in range(args.warmup):
        oracle_sample(w, A, B, C, rows, cores)
    times = []
    for _ in range(args.steps):
        t, n = oracle_sample(w, A, B, C, rows, cores)
        times.append(t)
    sec = sum(times) / len(times)
    flops = 2.0 * rows * w.N * w.K
    value = flops / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                         "cpu": host_cpu_model(), "kind": "oracle",
                         "sample": f"{rows} of {w.M} output rows per step (all N columns, all W ranks)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(w) -> dict:
    return {"workload": w.name, "W": w.W, "M": w.M, "N": w.N, "K": w.K, "K_per_rank": w.Kpr,
            "alpha": w.alpha, "beta": w.beta, "y_dtype": w.y_dtype,
            "inputs": f"A {w.a_dist}, B {w.b_dist}" + (f", C {w.c_dist}" if w.c_dist else ""),
            "l2": l2_note(w)}


def working_set_bytes(w) -> int:
    ab = w.W * w.M * w.Kpr * 2 + w.W * w.Kpr * w.N * 2
    c = w.M * w.N * 2 if w.beta != 0 else 0
    return ab + c + w.W * w.M * w.N * 4


def fits_l2(w) -> bool:
    return working_set_bytes(w) <= L2_BYTES


def l2_note(w) -> str:
    ab = w.W * w.M * w.Kpr * 2 + w.W * w.Kpr * w.N * 2
    ws = w.W * w.M * w.N * 4
    if not fits_l2(w):
        return (f"inputs larger than L2: A+B {ab / 1e6:.0f} MB + partial workspace {ws / 1e6:.0f} MB"
                " > 129 MB L2, no flush between steps")
    return (f"working set {working_set_bytes(w) / 1e6:.1f} MB fits in L2: a "
            f"{FLUSH_BYTES >> 20} MB buffer is written between timed calls (L2 flush) and "
            "ms_per_step is the mean of the per-call CUDA-event times")


def chunked_baseline(W, M, N, alpha, beta, y_code, Ad, Bd, Cd, Y, stream, dev):
    """The chunked two-stream baseline (async-TP style, an unfused comparator):
    for each output chunk c, the W per-rank GEMMs of the chunk's rows run on
    `stream` into fp32 partials while the reduce of chunk c-1 runs on a second
    stream; two chunk buffers alternate.  Returns a callable that runs one
    call; `stream` has waited for all of its work when it returns."""
    import torch
    from tensor_gemm_reduce_tcgen05_gb300 import binding
    R = M // W
    s_red = torch.cuda.Stream(device=dev)
    Pc = [torch.empty((W, R, N), dtype=torch.float32, device=dev) for _ in range(2)]
    ev_p = [torch.cuda.Event() for _ in range(2)]
    ev_r = [torch.cuda.Event() for _ in range(2)]
    y_elt = Y.element_size()

    def run():
        for c in range(W):
            buf = c % 2
            if c >= 2:
                stream.wait_event(ev_r[buf])  # chunk c-2's reduce is done with the buffer
            with torch.cuda.stream(stream):
                torch.bmm(Ad[:, c * R:(c + 1) * R, :], Bd, out_dtype=torch.float32, out=Pc[buf])
            ev_p[buf].record(stream)
            s_red.wait_event(ev_p[buf])
            binding.gemm_rs_reduce_partials(
                Pc[buf].data_ptr(), binding.GEMM_RS_FP32,
                0 if Cd is None else Cd.data_ptr() + c * R * N * 2,
                Y.data_ptr() + c * R * N * y_elt, R, N, W, alpha, beta, y_code,
                s_red.cuda_stream)
            ev_r[buf].record(s_red)
        stream.wait_stream(s_red)

    return run


# --------------------------------------------------------------------------- our arm
def time_loop(fn, steps, stream):
    """Mean ms per call over `steps` calls of fn on `stream`.  Each call is
    bracketed by its own event pair, the pattern of the fused arm's timed
    region when an L2 flush separates its calls, so every arm pays the same
    event overhead between calls."""
    import torch
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    per_call = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(steps)]
    torch.cuda.synchronize()
    s.record(stream)
    for a, b in per_call:
        a.record(stream)
        fn()
        b.record(stream)
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def interleaved(arms, rounds, n, stream, timer=None):
    """Mean ms per call of each arm ({name: fn}), timed in `rounds` rounds of
    n calls per arm, the arms' order reversed every other round.  Under the
    board's power cap the clock drifts down as a run goes on, so arms timed one
    after the other are not comparable; interleaved rounds see the same clocks."""
    timer = timer or time_loop
    names = list(arms)
    per = {k: [] for k in names}
    for r in range(rounds):
        for k in (names if r % 2 == 0 else names[::-1]):
            per[k].append(timer(arms[k], n, stream))
    return {k: sum(v) / len(v) for k, v in per.items()}


def sustained_run(step, w, stream, seconds: float, cold: bool, flush) -> dict:
    """The fused calls back to back for at least `seconds`: blocks of calls
    sized from a first probe block, each block timed with one event pair
    (with an L2 flush before each call when the working set fits in L2, whose
    time the calls' own events then exclude)."""
    import torch
    probe = max(1, min(200, int(0.05 / max(w.flops / 2.0e15, 1e-6))))
    ms_probe = time_loop_b2b(step, probe, stream) if not cold else time_loop(step, probe, stream)
    block = max(1, int(200.0 / max(ms_probe, 1e-3)))  # about 0.2 s per block
    calls, total_ms, per_block = 0, 0.0, []
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        if cold:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(block)]
            for a, b in evs:
                flush()
                a.record(stream)
                step()
                b.record(stream)
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in evs)
        else:
            ms = time_loop_b2b(step, block, stream) * block
        per_block.append(ms / block)
        total_ms += ms
        calls += block
    ms_call = total_ms / calls
    return {"calls": calls, "seconds": total_ms / 1e3, "ms_per_call": ms_call,
            "ms_per_call_first_block": per_block[0], "ms_per_call_last_block": per_block[-1],
            "tflops": w.flops / (ms_call / 1e3) / 1e12}


def time_loop_b2b(fn, steps, stream):
    """Mean ms per call with the calls back to back (no events between them):
    what a caller that issues them in a row sees."""
    import torch
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record(stream)
    for _ in range(steps):
        fn()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def profile_unfused(args, w, Ad, Bd, Cd, Y, stream):
    """Profiling run of the unfused arm alone: batched per-rank cuBLAS GEMMs into
    fp32 partials, then the separate reduce kernel, warm-up + steps calls."""
    import torch
    from tensor_gemm_reduce_tcgen05_gb300 import binding
    P = torch.empty((w.W, w.M, w.N), dtype=torch.float32, device=Ad.device)
    y_code = binding.GEMM_RS_BF16 if w.y_dtype == "bf16" else binding.GEMM_RS_FP32

    def unfused():
        torch.bmm(Ad, Bd, out_dtype=torch.float32, out=P)
        binding.gemm_rs_reduce_partials(P.data_ptr(), binding.GEMM_RS_FP32,
                                        0 if Cd is None else Cd.data_ptr(), Y.data_ptr(), w.M, w.N,
                                        w.W, w.alpha, w.beta, y_code, stream.cuda_stream)
    for _ in range(args.warmup):
        unfused()
    ms = time_loop(unfused, args.steps, stream)
    print(json.dumps({"metric": METRIC, "arm": "unfused", "ms_per_step": ms,
                      "config": workload_config(w),
                      "note": "profiling run: unfused arm only (torch.bmm fp32 out + reduce kernel)"}))
    return 0


def run_ours(args):
    import torch
    from tensor_gemm_reduce_tcgen05_gb300 import binding
    from tensor_gemm_reduce_tcgen05_gb300.inputs import WORKLOADS, workload_inputs

    rank, world, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    w = WORKLOADS[args.workload]
    peaks = load_peaks()
    binding.lib()

    A, B, C = workload_inputs(w)
    A_pin, B_pin = A.pin_memory(), B.pin_memory()
    C_pin = None if C is None else C.pin_memory()
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = None if C is None else C.to(dev)
    op = binding.GemmRS(w.M, w.N, w.K, w.W, w.alpha, w.beta, w.y_dtype, device=dev)
    if args.tile_n:
        binding.gemm_rs_set_tile_n(op.handle, args.tile_n)
    if args.reduce_mode:
        binding.gemm_rs_set_reduce_mode(op.handle, REDUCE_MODES[args.reduce_mode])
    Y = op.new_output()
    Y_pin = torch.empty(Y.shape, dtype=Y.dtype, pin_memory=True)
    if args.unfused_only:
        return profile_unfused(args, w, Ad, Bd, Cd, Y, stream)

    def step():
        op.run(Ad, Bd, Cd, Y, stream)

    # A buffer larger than L2, written between timed calls when the working set
    # would otherwise stay in L2 from one call to the next.
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush_buf.fill_(1.0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if op.status(stream) != 0:
        raise RuntimeError("device timeout during warm-up: " + binding.gemm_rs_last_error())
    # clocks of the fused region: the timed steps and the sustained run after them
    sampler = ClockSampler(local)
    sampler.start()

    # ---- timed region: K fused calls.  With an L2 flush between calls, events
    # around each launch give the calls' own device time.  Without one, the K
    # calls run back to back between two events: an event recorded between two
    # launches would keep a call's prologue (barrier and TMEM set-up, before its
    # griddepcontrol.wait) from overlapping the previous call, which a caller
    # issuing calls back to back gets.  The average launch duration is then the
    # region over K (the region holds nothing but the K launches).
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize()
    cold = fits_l2(w)
    t0.record(stream)
    for i in range(args.steps):
        if cold:
            flush_l2()
            starts[i].record(stream)
        step()
        if cold:
            ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    if op.status(stream) != 0:
        raise RuntimeError("device timeout in the timed region: " + binding.gemm_rs_last_error())
    if cold:
        kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        kernel_avg_ms = sum(kernel_ms) / len(kernel_ms)
        ms_step = kernel_avg_ms
    else:
        ms_step = t0.elapsed_time(t1) / args.steps
        kernel_avg_ms = ms_step
        # the spread of single calls, each between its own events (diagnostic)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_sorted = sorted(kernel_ms)
    kernel_median_ms = kernel_sorted[len(kernel_sorted) // 2]
    kernel_min_ms = kernel_sorted[0]
    kernel_note = ("each timed call between its own events, an L2 flush before each" if cold else
                   "kernel_ms: the back-to-back timed region over its launches; median and min: "
                   "calls timed one at a time between their own events after the region")

    ms_step_max = max_over_ranks(dist, ms_step, dev)
    value = aggregate_throughput(w.flops, world, ms_step_max / 1e3) / 1e12

    # ---- sustained: the same calls back to back for at least --sustain-seconds
    sustained = None
    if args.sustain_seconds > 0:
        sustained = sustained_run(step, w, stream, args.sustain_seconds, cold, flush_l2)
    clocks = sampler.stop()
    if sustained is not None:
        sustained["sm_mhz_median"] = clocks.get("sm_mhz")
        sustained["samples_under_load"] = clocks.get("samples_under_load")
        if clocks.get("sm_mhz"):
            sustained["ms_x_ghz"] = sustained["ms_per_call"] * clocks["sm_mhz"] / 1e3
        sustained["frac_of_sustained_peak"] = sustained["tflops"] / peaks["bf16_tflops_sustained"]
        sustained["frac_of_burst_peak"] = sustained["tflops"] / peaks["bf16_tflops"]
    if op.status(stream) != 0:
        raise RuntimeError("device timeout in the sustained run: " + binding.gemm_rs_last_error())
    sampler = ClockSampler(local)  # the rest of the run (baselines, ablations)
    sampler.start()

    if args.skip_extras:
        rest = sampler.stop()
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step_max,
                "kernel_ms": kernel_avg_ms, "kernel_ms_median": kernel_median_ms,
                "kernel_ms_min": kernel_min_ms, "kernel_ms_note": kernel_note,
                "config": workload_config(w), "plan": op.plan,
                "clocks": clocks, "sustained": sustained, "clocks_rest": rest,
                "note": "profiling run: fused kernel only"}
        if rank == 0:
            print(json.dumps(line))
        op.close()
        if dist is not None:
            dist.destroy_process_group()
        return 0

    # ---- end to end through the public API: H2D inputs, run, D2H result.
    # gemm_rs_run_streamed copies each rank's operands on a copy stream while
    # the kernel consumes the ranks that have landed; the serial variant
    # (copies, then gemm_rs_run, then the copy back) is reported beside it.
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_step():
        op.run_streamed(A_pin, B_pin, C_pin, Y_pin, Ad, Bd, Cd, Y, stream, copy_stream)

    def e2e_serial_step():
        Ad.copy_(A_pin, non_blocking=True)
        Bd.copy_(B_pin, non_blocking=True)
        if Cd is not None:
            Cd.copy_(C_pin, non_blocking=True)
        op.run(Ad, Bd, Cd, Y, stream)
        Y_pin.copy_(Y, non_blocking=True)

    e2e_step()
    e2e_serial_step()
    torch.cuda.synchronize()
    if op.status(stream) != 0:
        raise RuntimeError("device timeout in the streamed call: " + binding.gemm_rs_last_error())
    barrier(dist, dev)
    e2e_ms = max_over_ranks(dist, time_loop(e2e_step, args.steps, stream), dev)
    e2e_serial_ms = time_loop(e2e_serial_step, args.steps, stream)
    if op.status(stream) != 0:
        raise RuntimeError("device timeout in the e2e region: " + binding.gemm_rs_last_error())
    h2d = A.numel() * 2 + B.numel() * 2 + (0 if C is None else C.numel() * 2)
    d2h = Y.numel() * Y.element_size()
    e2e_value = aggregate_throughput(w.flops, world, e2e_ms / 1e3) / 1e12

    # ---- unfused same-GPU baseline: batched per-rank cuBLAS GEMMs into fp32
    # partials, then the library's separate reduce kernel
    P = torch.empty((w.W, w.M, w.N), dtype=torch.float32, device=dev)
    p_dtype = binding.GEMM_RS_FP32
    try:
        torch.bmm(Ad, Bd, out_dtype=torch.float32, out=P)
        torch.cuda.synchronize()

        def gemms():
            torch.bmm(Ad, Bd, out_dtype=torch.float32, out=P)
        partials_note = "fp32 partials (torch.bmm out_dtype=float32)"
    except (TypeError, RuntimeError):
        P = torch.empty((w.W, w.M, w.N), dtype=torch.bfloat16, device=dev)
        p_dtype = binding.GEMM_RS_BF16

        def gemms():
            torch.bmm(Ad, Bd, out=P)
        partials_note = "bf16 partials (torch.bmm)"
    y_code = binding.GEMM_RS_BF16 if w.y_dtype == "bf16" else binding.GEMM_RS_FP32

    def reduce_only():
        binding.gemm_rs_reduce_partials(P.data_ptr(), p_dtype, 0 if Cd is None else Cd.data_ptr(),
                                        Y.data_ptr(), w.M, w.N, w.W, w.alpha, w.beta, y_code,
                                        stream.cuda_stream)

    def unfused():
        gemms()
        reduce_only()

    for _ in range(max(3, args.warmup)):
        unfused()
    # fused and unfused in interleaved rounds (the same clocks for both), each
    # call timed the way the fused arm's timed region times it: back to back,
    # or between its own events where an L2 flush separates the calls; the
    # other way is reported beside it
    rounds, per_round = 4, max(3, args.steps // 4)
    main_timer, other_timer = (time_loop, time_loop_b2b) if cold else (time_loop_b2b, time_loop)
    pair = interleaved({"fused": step, "unfused": unfused}, rounds, per_round, stream,
                       timer=main_timer)
    unfused_ms = pair["unfused"]
    gemms_ms = time_loop(gemms, args.steps, stream)
    reduce_ms = time_loop(reduce_only, args.steps, stream)
    other = interleaved({"fused": step, "unfused": unfused}, rounds, per_round, stream,
                        timer=other_timer)
    other = {"fused_ms": other["fused"], "unfused_ms": other["unfused"],
             "fused_speedup": other["unfused"] / other["fused"],
             "note": ("calls issued in a row with no events between them" if cold else
                      "each call between its own events, which keeps a call's prologue from "
                      "overlapping the previous call")}
    del P

    # chunked two-stream baseline (async-TP style)
    chunked = chunked_baseline(w.W, w.M, w.N, w.alpha, w.beta, y_code, Ad, Bd, Cd, Y, stream, dev)
    chunked_ms = chunked_fused_ms = None
    if p_dtype == binding.GEMM_RS_FP32:
        for _ in range(max(3, args.warmup)):
            chunked()
        cp = interleaved({"fused": step, "chunked": chunked}, rounds, per_round, stream,
                         timer=main_timer)
        chunked_ms, chunked_fused_ms = cp["chunked"], cp["fused"]
    del chunked

    # full-K GEMM of the same shape (no reduce-scatter at all): context
    A_full = Ad.permute(1, 0, 2).reshape(w.M, w.K).contiguous()
    B_full = Bd.reshape(w.K, w.N)
    for _ in range(3):
        torch.mm(A_full, B_full)
    fullk_ms = time_loop(lambda: torch.mm(A_full, B_full), args.steps, stream)
    del A_full

    # clear-kernel-sync ablation: counter clear + sync + kernel + sync per call
    def kernel_sync():
        step()
        torch.cuda.synchronize()

    def clear_kernel_sync():
        op.reset(stream)
        torch.cuda.synchronize()
        step()
        torch.cuda.synchronize()

    ks_ms = time_loop(kernel_sync, args.steps, stream)
    cks_ms = time_loop(clear_kernel_sync, args.steps, stream)

    # cold-L2 calls: a 256 MB write between calls, the calls' own event times
    n_cold = min(args.steps, 20)
    cs = [torch.cuda.Event(enable_timing=True) for _ in range(n_cold)]
    ce = [torch.cuda.Event(enable_timing=True) for _ in range(n_cold)]
    for i in range(n_cold):
        flush_l2()
        cs[i].record(stream)
        step()
        ce[i].record(stream)
    torch.cuda.synchronize()
    cold_ms = sorted(a.elapsed_time(b) for a, b in zip(cs, ce))

    # the library's other reductions: last-arriver (rank-order fold) and the
    # two-level fold (two rank groups, then their sums), each timed in
    # interleaved rounds with the default (every call leaves the tile state
    # words at 0, so the mode may change between calls)
    mode0 = op.plan["reduce_mode"]

    def with_mode(m):
        def run():
            binding.gemm_rs_set_reduce_mode(op.handle, m)
            step()
        return run
    modes = {"last_arriver": binding.GEMM_RS_REDUCE_LAST_ARRIVER,
             "chain": binding.GEMM_RS_REDUCE_CHAIN,
             "two_level": binding.GEMM_RS_REDUCE_TWO_LEVEL}
    arms = {"default": with_mode(mode0)}
    arms.update({name: with_mode(m) for name, m in modes.items() if m != mode0})
    for fn in arms.values():
        for _ in range(3):
            fn()
    res = interleaved(arms, rounds, per_round, stream, timer=main_timer)
    other_mode = {}
    for name, m in modes.items():
        if m == mode0:
            continue
        binding.gemm_rs_set_reduce_mode(op.handle, m)
        other_mode[name] = {"ms_per_step": res[name], "default_ms_interleaved": res["default"],
                            "plan": op.plan}
    binding.gemm_rs_set_reduce_mode(op.handle, mode0)
    if op.status(stream) != 0:
        raise RuntimeError("device timeout in the reduce-mode comparison: " +
                           binding.gemm_rs_last_error())
    clocks_rest = sampler.stop()

    # ---- roofline of the fused kernel (the only kernel of the step)
    flops_per_launch = float(w.flops)
    bytes_per_launch = float(algorithmic_bytes(w))
    t_tensor = flops_per_launch / (peaks["bf16_tflops"] * 1e12)
    t_hbm = bytes_per_launch / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = flops_per_launch / (kernel_avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
                "peak_sustained": peaks["bf16_tflops_sustained"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = bytes_per_launch / (kernel_avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} copy"}
    roof["kernel"] = kernel_name(op.plan)
    roof["traffic"] = recorded_traffic(roof["kernel"], w.name, op.plan)
    roof["algorithmic_bytes"] = int(bytes_per_launch)
    roof["algorithmic_flops"] = int(flops_per_launch)
    roof["kernel_ms"] = kernel_avg_ms

    # ---- CPU baseline: the oracle on a bounded row sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        rows, _ = calibrate_rows(w, A, B, C, cores, target_s=args.cpu_seconds)
        sec, n = oracle_sample(w, A, B, C, rows, cores)
        cpu = {"value": 2.0 * n * w.N * w.K / sec / 1e12, "unit": "TFLOP/s", "cores": cores,
               "cpu": host_cpu_model(),
               "kind": "oracle", "seconds": sec,
               "sample": f"{n} of {w.M} output rows (all N columns, all W ranks), evenly spaced"}

    plan = op.plan
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(w),
            "pct_of_peak": 100.0 * (flops_per_launch / (kernel_avg_ms / 1e3) / 1e12) / peaks["bf16_tflops"],
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "call": "gemm_rs_run_streamed (per-rank H2D on a copy stream, overlapped "
                            "with the kernel; Y back on the kernel's stream)",
                    "serial": {"ms_per_step": e2e_serial_ms,
                               "value": w.flops / (e2e_serial_ms / 1e3) / 1e12,
                               "note": "H2D of A, B, C, then gemm_rs_run, then D2H of Y"}},
            "gpu_launches": args.steps,
            "clocks": dict(clocks, region="the timed steps and the sustained run after them"),
            "sustained": sustained,
            "clocks_rest": clocks_rest,
            "cpu_baseline": cpu,
            "unfused": {"ms_per_step": unfused_ms,
                        "value": w.flops / (unfused_ms / 1e3) / 1e12,
                        "gemms_ms": gemms_ms, "reduce_ms": reduce_ms, "partials": partials_note,
                        "fused_ms_interleaved": pair["fused"],
                        "fused_speedup": unfused_ms / pair["fused"],
                        "note": f"fused and unfused timed in {rounds} interleaved rounds of "
                                f"{per_round} calls each, order reversed every round, "
                                + ("each call between its own events" if cold else
                                   "the calls of a round back to back")},
            "unfused_chunked": None if chunked_ms is None else {
                "ms_per_step": chunked_ms, "value": w.flops / (chunked_ms / 1e3) / 1e12,
                "chunks": w.W, "fused_speedup": chunked_ms / chunked_fused_ms,
                "note": "per chunk: W per-rank bmm (fp32 out) on one stream, reduce of the "
                        "previous chunk on a second stream, two chunk buffers"},
            "full_k_gemm": {"ms": fullk_ms, "value": w.flops / (fullk_ms / 1e3) / 1e12,
                            "note": "torch.mm [M,K]x[K,N], no reduce-scatter (context)"},
            "kernel_ms_median": kernel_median_ms, "kernel_ms_min": kernel_min_ms,
            "kernel_ms_note": kernel_note,
            "cold_l2": {"kernel_ms_median": cold_ms[len(cold_ms) // 2], "kernel_ms_min": cold_ms[0],
                        "calls": n_cold, "flush_bytes": FLUSH_BYTES},
            "ablation": {"kernel_batched_ms": ms_step, "kernel_sync_ms": ks_ms,
                         "clear_kernel_sync_ms": cks_ms},
            "other_reduce_mode": other_mode,
            "other_timing": other,
            "plan": plan,
        }
        print(json.dumps(line))
    op.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


AG_METRIC = "fused AG+GEMM TFLOP/s and % of GB300 bf16 tensor peak vs unfused, 1 GPU"


def run_ag(args):
    """The AG+GEMM half of the FFN (the first GEMM, all-gathered rows): one JSON
    line with the fused kernel's throughput, the unfused same-GPU baseline
    (the all-gather as W*(W-1) chunk copies into per-rank buffers, then one
    batched cuBLAS GEMM) and a plain batched GEMM without any gather."""
    import torch
    from tensor_gemm_reduce_tcgen05_gb300 import binding
    from tensor_gemm_reduce_tcgen05_gb300.inputs import AG_WORKLOADS, bf16_bits, make_ag_inputs

    w = AG_WORKLOADS[args.workload if args.workload in AG_WORKLOADS else "ag_ffn_w8_m4096"]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    X, B1 = make_ag_inputs(w.W, w.M, w.N, w.K, w.x_dist, w.b_dist)
    Xd, Bd = X.to(dev), B1.to(dev)
    op = binding.AgGemm(w.M, w.N, w.K, w.W, w.alpha, w.y_dtype, device=dev)
    H = op.new_output()

    def step():
        op.run(Xd, Bd, H, stream)

    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if op.status(stream) != 0:
        raise RuntimeError("device timeout during warm-up: " + binding.gemm_rs_last_error())
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if op.status(stream) != 0:
        raise RuntimeError("device timeout in the timed region: " + binding.gemm_rs_last_error())
    ms_step = t0.elapsed_time(t1) / args.steps
    kernel_ms = sorted(a.elapsed_time(b) for a, b in zip(starts, ends))
    kernel_avg = sum(kernel_ms) / len(kernel_ms)
    value = w.flops / (ms_step / 1e3) / 1e12
    if args.skip_extras:
        print(json.dumps({"metric": AG_METRIC, "value": value, "unit": "TFLOP/s",
                          "ms_per_step": ms_step, "kernel_ms": kernel_avg, "plan": op.plan,
                          "clocks": sampler.stop(), "note": "profiling run: fused kernel only"}))
        op.close()
        return 0

    # unfused: the all-gather as chunk copies into per-rank buffers, then bmm
    R = w.M // w.W
    G = torch.empty((w.W, w.M, w.K), dtype=torch.bfloat16, device=dev)
    Hu = torch.empty((w.W, w.M, w.N), dtype=torch.bfloat16 if w.y_dtype == "bf16" else torch.float32,
                     device=dev)

    def gemm():
        torch.bmm(G, Bd, out=Hu) if Hu.dtype == torch.bfloat16 else \
            torch.bmm(G, Bd, out_dtype=torch.float32, out=Hu)

    def gather():
        G.copy_(Xd.unsqueeze(0).expand(w.W, w.M, w.K))  # one copy kernel for all ranks

    def gather_chunks():
        for r in range(w.W):
            for c in range(w.W):
                if c != r:
                    G[r, c * R:(c + 1) * R].copy_(Xd[c * R:(c + 1) * R])

    def unfused():
        gather()
        gemm()

    def unfused_chunks():
        gather_chunks()
        gemm()

    def plain():
        torch.matmul(Xd, Bd, out=Hu)

    for _ in range(3):
        unfused()
        unfused_chunks()
        plain()
    rounds, per_round = 4, max(3, args.steps // 4)
    pair = interleaved({"fused": step, "unfused": unfused}, rounds, per_round, stream)
    unfused_ms = pair["unfused"]
    gather_ms = time_loop(gather, args.steps, stream)
    chunks_ms = time_loop(unfused_chunks, args.steps, stream)
    plain_ms = time_loop(plain, args.steps, stream)
    clocks = sampler.stop()
    del G, Hu

    cpu = None
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        cores = host_cores()
        rows = np.linspace(0, w.M - 1, 8).astype(np.int64)
        t = time.perf_counter()
        oracle.ag_gemm(bf16_bits(X), bf16_bits(B1), w.alpha, w.y_dtype, rows=rows, threads=cores)
        sec = time.perf_counter() - t
        cpu = {"value": 2.0 * len(rows) * w.W * w.N * w.K / sec / 1e12, "unit": "TFLOP/s",
               "cores": cores, "cpu": host_cpu_model(), "kind": "oracle", "seconds": sec,
               "sample": f"{len(rows)} of {w.M} rows of every rank's output, evenly spaced"}

    achieved = w.flops / (kernel_avg / 1e3) / 1e12
    line = {
        "metric": AG_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "W": w.W, "M": w.M, "N_per_rank": w.N, "K": w.K,
                   "alpha": w.alpha, "y_dtype": w.y_dtype,
                   "inputs": f"X {w.x_dist}, B1 {w.b_dist}",
                   "l2": "inputs larger than L2: gather buffers "
                         f"{w.W * w.M * w.K * 2 / 1e6:.0f} MB, no flush between steps"},
        "pct_of_peak": 100.0 * achieved / peaks["bf16_tflops"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
                     "kernel": "ag_gemm_pair_kernel", "kernel_ms": kernel_avg,
                     "traffic": recorded_traffic("ag_gemm_pair_kernel", w.name, op.plan,
                                                 AG_KERNEL_SOURCES)},
        "kernel_ms_median": kernel_ms[len(kernel_ms) // 2], "kernel_ms_min": kernel_ms[0],
        "gpu_launches": args.steps, "clocks": clocks, "cpu_baseline": cpu,
        "unfused": {"ms_per_step": unfused_ms, "value": w.flops / (unfused_ms / 1e3) / 1e12,
                    "gather_ms": gather_ms, "fused_ms_interleaved": pair["fused"],
                    "fused_speedup": unfused_ms / pair["fused"],
                    "note": "the all-gather as one copy of X into every rank's buffer, then "
                            "torch.bmm; fused and unfused timed in interleaved rounds"},
        "unfused_chunk_copies": {"ms_per_step": chunks_ms,
                                 "value": w.flops / (chunks_ms / 1e3) / 1e12,
                                 "note": "W*(W-1) chunk copies (one per rank and remote chunk), "
                                         "then torch.bmm"},
        "plain_gemm": {"ms": plain_ms, "value": w.flops / (plain_ms / 1e3) / 1e12,
                       "note": "torch.matmul X [M,K] x B1 [W,K,N], no gather (context)"},
        "plan": op.plan,
    }
    print(json.dumps(line))
    op.close()
    return 0


FFN_METRIC = "fused TP FFN (AG+GEMM then GEMM+RS) TFLOP/s vs unfused, 1 GPU"


def run_ffn(args):
    """The tensor-parallel FFN chain: AG+GEMM (X -> H) then GEMM+RS (H -> Y), on
    the shapes of the default GEMM+RS workload, through ffn_tp_run; against
    the unfused chain and against the two fused kernels timed alone."""
    import torch
    from tensor_gemm_reduce_tcgen05_gb300 import binding
    from tensor_gemm_reduce_tcgen05_gb300.inputs import AG_WORKLOADS, WORKLOADS, make_ag_inputs

    wa = AG_WORKLOADS["ag_ffn_w8_m4096"]
    wr = WORKLOADS["ffn_w8_m4096"]
    assert wr.W == wa.W and wr.M == wa.M and wr.Kpr == wa.N
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    X, B1 = make_ag_inputs(wa.W, wa.M, wa.N, wa.K, wa.x_dist, wa.b_dist)
    g = torch.Generator().manual_seed(2)
    B2 = (torch.randn((wr.W, wr.Kpr, wr.N), generator=g) * 0.02).to(torch.bfloat16)
    Xd, B1d, B2d = X.to(dev), B1.to(dev), B2.to(dev)
    ag = binding.AgGemm(wa.M, wa.N, wa.K, wa.W, wa.alpha, "bf16", device=dev)
    rs = binding.GemmRS(wr.M, wr.N, wr.K, wr.W, wr.alpha, wr.beta, wr.y_dtype, device=dev)
    H = ag.new_output()
    Y = rs.new_output()
    flops = wa.flops + wr.flops

    def chain():
        binding.ffn_tp_run(ag.handle, rs.handle, Xd.data_ptr(), B1d.data_ptr(), H.data_ptr(),
                           B2d.data_ptr(), 0, Y.data_ptr(), stream.cuda_stream)

    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(args.warmup):
        chain()
    torch.cuda.synchronize()
    if ag.status(stream) != 0 or rs.status(stream) != 0:
        raise RuntimeError("device timeout during warm-up: " + binding.gemm_rs_last_error())
    ms_step = time_loop(chain, args.steps, stream)
    ag_ms = time_loop(lambda: ag.run(Xd, B1d, H, stream), args.steps, stream)
    rs_ms = time_loop(lambda: rs.run(H, B2d, None, Y, stream), args.steps, stream)
    if ag.status(stream) != 0 or rs.status(stream) != 0:
        raise RuntimeError("device timeout in the timed region: " + binding.gemm_rs_last_error())
    if args.skip_extras:
        print(json.dumps({"metric": FFN_METRIC, "value": flops / (ms_step / 1e3) / 1e12,
                          "unit": "TFLOP/s", "ms_per_step": ms_step,
                          "stages": {"ag_gemm_ms": ag_ms, "gemm_rs_ms": rs_ms},
                          "clocks": sampler.stop(),
                          "note": "profiling run: the fused chain only"}))
        ag.close()
        rs.close()
        return 0

    # unfused chain: gather copy, bmm, bmm into fp32 partials, the reduce kernel
    G = torch.empty((wa.W, wa.M, wa.K), dtype=torch.bfloat16, device=dev)
    Hu = torch.empty((wa.W, wa.M, wa.N), dtype=torch.bfloat16, device=dev)
    P = torch.empty((wr.W, wr.M, wr.N), dtype=torch.float32, device=dev)
    y_code = binding.GEMM_RS_BF16 if wr.y_dtype == "bf16" else binding.GEMM_RS_FP32

    def unfused():
        G.copy_(Xd.unsqueeze(0).expand(wa.W, wa.M, wa.K))
        torch.bmm(G, B1d, out=Hu)
        torch.bmm(Hu, B2d, out_dtype=torch.float32, out=P)
        binding.gemm_rs_reduce_partials(P.data_ptr(), binding.GEMM_RS_FP32, 0, Y.data_ptr(), wr.M,
                                        wr.N, wr.W, wr.alpha, wr.beta, y_code, stream.cuda_stream)

    for _ in range(3):
        unfused()
    rounds, per_round = 4, max(3, args.steps // 4)
    pair = interleaved({"fused": chain, "unfused": unfused}, rounds, per_round, stream)
    unfused_ms = pair["unfused"]
    clocks = sampler.stop()
    del G, Hu, P

    line = {
        "metric": FFN_METRIC, "value": flops / (ms_step / 1e3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "ffn_tp_w8_m4096", "W": wa.W, "M": wa.M, "hidden": wa.K,
                   "ffn_per_rank": wa.N, "y_dtype": wr.y_dtype, "activation": "none",
                   "l2": "inputs larger than L2, no flush between steps"},
        "pct_of_peak": 100.0 * flops / (ms_step / 1e3) / 1e12 / peaks["bf16_tflops"],
        "gpu_launches": 2 * args.steps, "clocks": clocks,
        "stages": {"ag_gemm_ms": ag_ms, "gemm_rs_ms": rs_ms},
        "unfused": {"ms_per_step": unfused_ms, "value": flops / (unfused_ms / 1e3) / 1e12,
                    "fused_ms_interleaved": pair["fused"],
                    "fused_speedup": unfused_ms / pair["fused"],
                    "note": "gather copy, bmm, bmm into fp32 partials, separate reduce kernel; "
                            "fused and unfused timed in interleaved rounds"},
    }
    print(json.dumps(line))
    ag.close()
    rs.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ffn_w8_m8192_bias")
    ap.add_argument("--path", choices=["gemm_rs", "ag", "ffn"], default="gemm_rs",
                    help="gemm_rs: the fused GEMM + reduce-scatter (the default line); "
                         "ag: the fused all-gather + GEMM; ffn: both, chained")
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--reduce-mode", choices=sorted(REDUCE_MODES), default=None,
                    help="run the fused kernel in this reduction instead of the library's "
                         "default (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sustain-seconds", type=float, default=None,
                    help="after the timed steps, run the same calls back to back for at least "
                         "this long and report their throughput and clock (0: skip; default 3, "
                         "or 0 with --skip-extras)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused-only", action="store_true",
                    help="run only the unfused arm (cuBLAS bmm into fp32 partials + reduce "
                         "kernel); used for profiling runs")
    ap.add_argument("--skip-extras", action="store_true",
                    help="time only the fused kernel (no e2e, baselines, ablation or CPU oracle); "
                         "used for profiling runs")
    args = ap.parse_args(argv)
    # At least three warm-up steps are always run; the JSON line reports the number run.
    args.warmup = max(3, args.warmup)
    args.steps = max(1, args.steps)
    if args.sustain_seconds is None:
        args.sustain_seconds = 0.0 if args.skip_extras else 3.0
    if args.impl == "reference":
        return run_reference(args)
    if args.path == "ag":
        return run_ag(args)
    if args.path == "ffn":
        return run_ffn(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
