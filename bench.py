"""Benchmark of the AdamW optimizer step on one or more GPUs of one node.

One "step" is one optimizer step over the whole tensor list of the workload
(default: the OPT-1.3b-shaped list, 388 tensors, 1,315,758,080 parameters,
pure-bf16 AnyPrecisionAdamW with Kahan compensation: 18 bytes moved per
parameter).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on host cores

With N > 1 (torchrun) every rank runs an independent replica of the same
workload on its own GPU (the step has no data exchange); value = parameters
updated by all ranks / the slowest rank's time.
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
from concurrent.futures import ThreadPoolExecutor

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from adamw_optimizer_step_sm_gb300 import adamw_sm as A  # noqa: E402
from adamw_optimizer_step_sm_gb300 import workloads as W  # noqa: E402

METRIC = "params updated/s & achieved HBM GB/s (% of peak), OPT-1.3b-shaped bf16 Kahan step"
UNIT = "params/s"
DEFAULT_WORKLOAD = "opt1.3b_bf16_kahan"
L2_BYTES = 129 << 20
L2_FLUSH_THRESHOLD = 2 * L2_BYTES


def bytes_per_param(w: W.Workload) -> int:
    """Algorithmic HBM bytes per parameter per step.
    bf16 Kahan: read p, g, m, v, c (10) + write p, m, v, c (8) = 18.
    mixed: read master, m, v (12) + g (2), write master, m, v (12) + p_out (2)
    = 28.  remainder: read p, r (4) + m, v (8) + g (2), write p, r, m, v (12)
    = 26.  bf16 plain: read p, g, m, v (8), write p, m, v (6) = 14.  bf16
    Kahan with fp32 v: read 12, write 10 = 22.  Any precision: p and g (read
    4, write 2) plus each of m, v, c read and written in its own width, so
    6 + 2 * (m + v + c) bytes, c = 0 without Kahan summation (all-fp32 state:
    30).  With clipping the norm pass reads g once more: +2."""
    if w.mode >= W.MODE_ANYPREC:
        f = w.mode - W.MODE_ANYPREC
        mvc = (4 if f & 1 else 2) + (4 if f & 2 else 2) + (0 if f & 8 else (4 if f & 4 else 2))
        base = 6 + 2 * mvc
    else:
        base = {W.MODE_BF16_KAHAN: 18, W.MODE_MIXED: 28, W.MODE_REMAINDER: 26,
                W.MODE_BF16_PLAIN: 14, W.MODE_BF16_KAHAN_V32: 22}[w.mode]
    return base + (2 if w.max_grad_norm > 0 else 0)


def workload_of(args) -> W.Workload:
    """The named workload, in the storage mode --mode asks for (renamed
    <list>_mode<N>, same tensors, hyperparameters and inputs)."""
    w = W.WORKLOADS[args.workload]
    mode = getattr(args, "mode", None)
    if mode is None or mode == w.mode:
        return w
    if mode not in W.MODE_DTYPES:
        raise SystemExit(f"unknown storage mode {mode}")
    import dataclasses
    base = w.name.split("_")[0]
    return dataclasses.replace(w, name=f"{base}_mode{mode}", mode=mode,
                               description=f"{w.description}; run in storage mode {mode} "
                                           f"({mode_name(mode)[1]})")


def mode_name(mode: int) -> tuple[str, str]:
    """Name and buffer layout of a storage mode, for the JSON line."""
    named = {0: ("bf16_kahan", "bf16 p/g/m/v/c"),
             1: ("mixed_fp32_master", "fp32 master/m/v, bf16 g and param out"),
             2: ("mixed_bf16_remainder", "bf16 p + int16 remainder, fp32 m/v, bf16 g"),
             3: ("bf16_plain", "bf16 p/g/m/v, no compensation"),
             4: ("bf16_kahan_fp32_variance", "bf16 p/g/m/c, fp32 v")}
    if mode in named:
        return named[mode]
    f = mode - W.MODE_ANYPREC
    m, v = ("fp32" if f & 1 else "bf16"), ("fp32" if f & 2 else "bf16")
    c = "no compensation" if f & 8 else ("fp32" if f & 4 else "bf16") + " c"
    return (f"anyprecision_{f}", f"bf16 p/g, {m} m, {v} v, {c}")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


KERNEL_SOURCES = ("adamw_internal.h", "device_common.cuh", "kernels.cuh", "launch.h",
                  "adamw_sm.cu", "plan_build.cpp",
                  "update_mode.inc", "update_m0.cu", "update_m1.cu", "update_m2.cu",
                  "update_m3.cu", "update_m4.cu", "update_m17.cu", "update_m19.cu",
                  "update_m20.cu", "update_m21.cu", "update_m22.cu", "update_m23.cu",
                  "update_m25.cu", "update_m26.cu", "update_m27.cu")


def _code_only(text: str) -> str:
    """C/C++ source with its comments removed and whitespace runs collapsed,
    string and character literals kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(read=None) -> str:
    """Hash of the code (comments and layout left out) of the files that
    define the kernels, their launches and the partition: what decides the
    DRAM traffic of a launch.  `read(name)` gives a file's text (default:
    the working tree's)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "adamw_optimizer_step_sm_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as fh:
                return fh.read()
    for f in KERNEL_SOURCES:
        h.update(_code_only(read(f)).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the update kernel from a committed ncu summary,
    or None when none exists or the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        busy = [x for x in sm if x > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle --

def oracle_throughput(w: W.Workload, n_elems: int, steps: int, threads: int, arrays=None):
    """The oracle as it stands on host cores, over the first n_elems elements
    of the workload; returns (params/s, seconds, threads).  ``arrays`` may hold
    host copies (param, exp_avg, exp_avg_sq, aux, grad, offsets) of the
    workload's freshly drawn state; otherwise the sample is drawn on the CPU."""
    import numpy as np
    import oracle as O
    o = O.load()
    to16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    if arrays is None:
        ws = W.truncated(w, n_elems)
        st = W.make_state(ws, "cpu")
        p, m, v, a = (host_array(x) for x in (st.param, st.exp_avg, st.exp_avg_sq, st.aux))
        grads = [to16(W.make_grad(ws, k + 1, "cpu")) for k in range(min(steps, 2))]
        offsets, numels = st.offsets, ws.numels
    else:
        ws = w
        p, m, v, a, g0, offsets = arrays
        grads, numels = [g0], w.numels
    hp = O.hparams(**ws.hparams())
    # split the elementwise work into contiguous pieces, several per thread
    pieces = []
    for off, n in zip(offsets, numels):
        step = max(1 << 16, -(-n // threads))
        for s in range(0, n, step):
            pieces.append((off + s, min(n - s, step)))
    clip = ws.max_grad_norm > 0
    t0 = time.perf_counter()
    for k in range(steps):
        g = grads[k % len(grads)]
        coef = 1.0
        if clip:
            sumsq, bad = o.grad_sumsq([g[off:off + n] for off, n in zip(offsets, numels)])
            coef, _ = o.clip_coef(sumsq, ws.max_grad_norm)

        def one(pc, t=k + 1):
            s, n = pc
            sl = slice(s, s + n)
            if ws.mode == W.MODE_BF16_KAHAN:
                o.bf16_kahan(p[sl], g[sl], m[sl], v[sl], a[sl], hp, t, coef)
            elif ws.mode == W.MODE_MIXED:
                o.mixed(p[sl], g[sl], m[sl], v[sl], a[sl], hp, t, coef)
            elif ws.mode == W.MODE_REMAINDER:
                o.remainder(p[sl], g[sl], m[sl], v[sl], a[sl], hp, t, coef)
            elif ws.mode == W.MODE_BF16_PLAIN:
                o.bf16_plain(p[sl], g[sl], m[sl], v[sl], hp, t, coef)
            elif ws.mode == W.MODE_BF16_KAHAN_V32:
                o.bf16_kahan_v32(p[sl], g[sl], m[sl], v[sl], a[sl], hp, t, coef)
            else:
                o.anyprec(p[sl], g[sl], m[sl], v[sl], None if a is None else a[sl],
                          ws.mode - W.MODE_ANYPREC, hp, t, coef)

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, pieces))
    dt = time.perf_counter() - t0
    return sum(numels) * steps / dt, dt, threads


def host_array(t: torch.Tensor | None):
    """Host numpy copy with the oracle's dtype (bf16 as uint16 bits)."""
    import numpy as np
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------- distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """Largest x over ranks (the slowest replica sets the time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# -------------------------------------------------------------- GPU arm --

def copy_ceiling(device, nbytes: int = 4 << 30, reps: int = 5) -> dict:
    """Device-to-device copy bandwidth: cudaMemcpyAsync and the library's
    16-byte copy kernel (bytes = read + write)."""
    src = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    src.fill_(1)
    stream = torch.cuda.current_stream(device)
    out = {}
    for name, fn in (("memcpy", lambda: dst.copy_(src)),
                     ("kernel", lambda: A.adamw_copy_probe(dst.data_ptr(), src.data_ptr(), nbytes,
                                                           stream.cuda_stream))):
        fn()
        torch.cuda.synchronize(device)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        out[name] = 2 * nbytes / best / 1e9
    del src, dst
    torch.cuda.empty_cache()
    out["ceiling"] = max(out["memcpy"], out["kernel"])
    return out


def host_link_ceiling(device, nbytes: int, reps: int = 3) -> dict:
    """Host-to-device bandwidth over the CPU-GPU link for nbytes from pinned
    host memory: cudaMemcpyAsync, and the library's copy kernel reading the
    pinned buffer in place (zero copy).  Bytes = nbytes (what crosses the
    link); best of reps."""
    nbytes = (nbytes + 15) // 16 * 16
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    out = {}
    for name, fn in (("memcpy_h2d", lambda: dst.copy_(host, non_blocking=True)),
                     ("zero_copy_read", lambda: A.adamw_copy_probe(dst.data_ptr(), host.data_ptr(),
                                                                   nbytes, stream.cuda_stream))):
        fn()
        torch.cuda.synchronize(device)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        out[name] = nbytes / best / 1e9
    del host, dst
    torch.cuda.empty_cache()
    out["ceiling"] = max(out["memcpy_h2d"], out["zero_copy_read"])
    out["bytes"] = nbytes
    return out


def run_e2e(args, w, st, grads, plans, hp, clip, t, world, device) -> dict:
    """The same metric end to end: every step copies that step's bf16
    gradients from pinned host memory, runs the step and reads the non-finite
    flag (4 bytes) back to the host, which decides whether the step counted.

    Paths, all through the library's C ABI:
      overlapped  two device gradient buffers; step k+1's host-to-device copy
                  runs on a side stream while step k updates (the reported e2e)
      serial      copy, then step, on one stream
      zero_copy   the plan's gradient pointers are the pinned host buffer
                  itself; the kernels read it over NVLink-C2C
    """
    N = w.total
    # as many steps as the timed region (at most 50): the overlapped path's
    # first copy and last step are not hidden, and a window of more steps
    # spreads them the way a training run does
    k_e2e = max(2, min(args.steps, 50))
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)
    host_g = [torch.empty(grads[0].numel(), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    host_g[0].copy_(grads[0])
    host_g[1].copy_(grads[1 % len(grads)])
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    host_flag = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    norm = torch.zeros(1, dtype=torch.float64, device=device)
    state = {"t": t}
    bufs = [grads[0], grads[1 % len(grads)]]
    bplans = [plans[0], plans[1 % len(plans)]]

    def finish_step():
        host_flag.copy_(flag, non_blocking=True)
        stream.synchronize()
        if not (clip and int(host_flag.item())):
            state["t"] += 1

    def serial(i):
        bufs[0].copy_(host_g[i % 2], non_blocking=True)
        bplans[0].step(hp, state["t"] + 1, grad_norm=norm if clip else None, nonfinite=flag)
        finish_step()

    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]

    def overlap_prime():
        used[1].record(stream)
        with torch.cuda.stream(side):
            bufs[0].copy_(host_g[0], non_blocking=True)
            copied[0].record(side)

    def overlapped(i):
        b, nb = i % 2, 1 - i % 2
        side.wait_event(used[nb])            # buffer nb is free once step i-1 ended
        with torch.cuda.stream(side):
            bufs[nb].copy_(host_g[nb], non_blocking=True)
            copied[nb].record(side)
        stream.wait_event(copied[b])
        bplans[b].step(hp, state["t"] + 1, grad_norm=norm if clip else None, nonfinite=flag)
        used[b].record(stream)
        finish_step()

    v = st.views
    zc_plan = A.Plan(v(st.param), v(host_g[0]), v(st.exp_avg), v(st.exp_avg_sq), v(st.aux),
                     w.mode, norm=clip)

    def zero_copy(i):
        zc_plan.step(hp, state["t"] + 1, grad_norm=norm if clip else None, nonfinite=flag)
        finish_step()

    # each path: args.reps repetitions of k_e2e steps, the median repetition
    # reported (the host-to-device copies now and then stall for tens of
    # milliseconds on this host; the median keeps one stall from deciding)
    out = {}
    for name, fn, prime in (("overlapped", overlapped, overlap_prime), ("serial", serial, None),
                            ("zero_copy", zero_copy, None)):
        reps = []
        for _ in range(args.reps):
            torch.cuda.synchronize(device)
            barrier(world)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if prime:
                prime()
            for i in range(k_e2e):
                fn(i)
            e1.record(stream)
            e1.synchronize()
            reps.append(reduce_max(e0.elapsed_time(e1) / 1e3, world, device))
        secs = statistics.median(reps)
        out[name] = {"value": world * N * k_e2e / secs, "ms_per_step": secs / k_e2e * 1e3,
                     "ms_per_step_min": min(reps) / k_e2e * 1e3,
                     "ms_per_step_max": max(reps) / k_e2e * 1e3}
    zc_plan.close()
    torch.cuda.synchronize(device)
    described = {
        "overlapped": "bf16 grads in pinned host memory, copied to the device on a side stream "
                      "while the previous step runs (double-buffered); flag read back every step",
        "serial": "bf16 grads in pinned host memory copied to the device, then the step; flag "
                  "read back every step",
        "zero_copy": "bf16 grads in pinned host memory read by the kernels over NVLink-C2C; "
                     "flag read back every step",
    }
    name = max(out, key=lambda k: out[k]["value"])
    best = out[name]
    link = host_link_ceiling(device, int(N * 2))
    link_gbs = N * 2 / (best["ms_per_step"] / 1e3) / 1e9
    return {"value": best["value"], "unit": UNIT, "h2d_bytes_per_step": int(N * 2),
            "d2h_bytes_per_step": 4, "ms_per_step": best["ms_per_step"], "steps": k_e2e,
            "repetitions": args.reps,
            "path": described[name], "paths": out,
            "link_gbs": link_gbs, "link_ceiling_gbs": link,
            "frac_of_link": link_gbs / link["ceiling"], "_t": state["t"]}


def run_gpu(args):
    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    A.load()
    w = workload_of(args)
    from dataclasses import replace
    w_bench = replace(w, inf_at=None)   # timing steps carry no injected inf
    clip = w.max_grad_norm > 0
    bpp = bytes_per_param(w)
    N = w.total

    ceiling = copy_ceiling(device) if not args.no_ceiling else None

    st = W.make_state(w_bench, device)
    n_grad = max(1, min(args.steps + args.warmup, args.grad_buffers))
    grads = [W.make_grad(w_bench, k + 1, device) for k in range(n_grad)]
    cpu_arrays = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # host copy of the freshly drawn inputs (before any step runs), for
        # the CPU oracle baseline
        cpu_arrays = (host_array(st.param), host_array(st.exp_avg), host_array(st.exp_avg_sq),
                      host_array(st.aux), host_array(grads[0]), list(st.offsets))
    v = st.views
    plans = [A.Plan(v(st.param), v(g), v(st.exp_avg), v(st.exp_avg_sq), v(st.aux), w.mode,
                    norm=clip, fuse=not args.no_fuse) for g in grads]
    hp = A.hparams(**w.hparams())
    stream = torch.cuda.current_stream(device)
    norm = torch.zeros(1, dtype=torch.float64, device=device)
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    launches_per_step = (1 if plans[0].info.fused else 3) if clip else 1

    t = 0
    for i in range(args.warmup):
        plans[i % n_grad].step(hp, t + 1, grad_norm=norm if clip else None,
                               nonfinite=flag if clip else None)
        t += 1
    torch.cuda.synchronize(device)
    barrier(world)

    # Inputs larger than L2 stream back to back; smaller ones get a 256 MiB
    # write before every timed step (outside the step's events) so that each
    # step starts from a cold L2.
    flush = bpp * N < L2_FLUSH_THRESHOLD
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=device) if flush else None

    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    # args.reps repetitions of args.steps steps each.  Large lists: the steps
    # of a repetition run back to back between two events (no event between
    # steps, so consecutive launches may overlap their ramp as they do in
    # training).  L2-resident lists: each step between its own events, after
    # the flush.
    rep_s = []
    torch.cuda.synchronize(device)
    barrier(world)
    wall0 = time.perf_counter()
    for r in range(args.reps):
        if flush:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.steps):
                flush_buf.fill_(i & 0xFF)
                ev[i][0].record(stream)
                plans[(args.warmup + i) % n_grad].step(hp, t + 1, grad_norm=norm if clip else None,
                                                       nonfinite=flag if clip else None)
                ev[i][1].record(stream)
                t += 1
            torch.cuda.synchronize(device)
            rep_s.append(sum(a.elapsed_time(b) / 1e3 for a, b in ev))
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(args.steps):
                plans[(args.warmup + i) % n_grad].step(hp, t + 1, grad_norm=norm if clip else None,
                                                       nonfinite=flag if clip else None)
                t += 1
            e1.record(stream)
            e1.synchronize()
            rep_s.append(e0.elapsed_time(e1) / 1e3)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    barrier(world)
    clk = clocks.stop()

    # the slowest rank's time of each repetition, then the median repetition
    rep_s = [reduce_max(x, world, device) for x in rep_s]
    span_max = statistics.median(rep_s)
    ms_per_step = span_max / args.steps * 1e3
    value = world * N * args.steps / span_max
    # one update launch per step (or one norm + update sequence with
    # clipping): the average launch is the step time
    avg_launch = span_max / args.steps
    achieved = bpp * N / avg_launch / 1e9
    repetitions = {"n": len(rep_s), "ms_per_step_median": ms_per_step,
                   "ms_per_step_min": min(rep_s) / args.steps * 1e3,
                   "ms_per_step_max": max(rep_s) / args.steps * 1e3}

    extra = {}
    if flush:
        # the same steps back to back with a warm L2, and as one CUDA graph of
        # device-resident steps (no launch gaps), for context; both on one
        # plan (one gradient buffer), as a training loop runs them: its
        # device-step memo then holds each next step's scalars (median of
        # the repetitions for both; the graph replayed once untimed first,
        # which uploads it to the device)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        warm_s = []
        for _ in range(max(1, args.reps)):
            e0.record(stream)
            for i in range(args.steps):
                plans[0].step(hp, t + 1, grad_norm=norm if clip else None,
                              nonfinite=flag if clip else None)
                t += 1
            e1.record(stream)
            e1.synchronize()
            warm_s.append(e0.elapsed_time(e1) / 1e3)
        warm = statistics.median(warm_s)
        extra["warm_l2"] = {"ms_per_step": warm / args.steps * 1e3,
                            "value": N * args.steps / warm,
                            "how": f"median of {len(warm_s)} x {args.steps} steps of one plan "
                                   "launched from Python"}
        d_hp = A.device_hparams(hp, device)
        d_step = torch.full((1,), t, dtype=torch.int64, device=device)
        flags = A.STEP_CLIP if clip else 0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                plans[0].step_device(d_hp, d_step, flags, grad_norm=norm if clip else None)
        graph.replay()
        torch.cuda.synchronize(device)
        g_all = []
        for _ in range(max(1, args.reps)):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            g_all.append(e0.elapsed_time(e1) / 1e3)
        g_s = statistics.median(g_all)
        t = int(d_step.item())
        extra["graph_warm_l2"] = {"ms_per_step": g_s / args.steps * 1e3,
                                  "value": N * args.steps / g_s,
                                  "how": f"{args.steps} device-resident steps of one plan in one "
                                         f"CUDA graph, median of {len(g_all)} replays"}
        del graph

    # end to end through the public API, gradients arriving in pinned host
    # memory every step and the non-finite flag read back every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, st, grads, plans, hp, clip, t, world, device)
        t = e2e.pop("_t")

    peaks = load_peaks()
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": w.name, "description": w.description, "n_params": N,
            "n_tensors": w.n_tensors,
            "mode": mode_name(w.mode)[0],
            "storage": mode_name(w.mode)[1],
            "clip": clip, "bytes_per_param": bpp, "hparams": w.hparams(),
            "l2": (f"256 MiB written before every timed step (L2 flushed; {bpp * N / 1e6:.1f} MB "
                   "moved per step)") if flush else
                  f"inputs larger than L2 ({bpp * N / 1e9:.2f} GB moved per step)",
            "grads": f"{n_grad} resident grad buffers drawn before timing, cycled",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "fused_clipped_step": bool(plans[0].info.fused),
        },
        "repetitions": repetitions,
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                     "traffic": recorded_traffic(w.name),
                     "kernel": "adamw_update_kernel" if not clip else "whole step (norm + update)",
                     "algorithmic_bytes_per_launch": bpp * N,
                     "avg_launch_ms": avg_launch * 1e3},
        "copy_ceiling_gbs": ceiling,
        **extra,
        "frac_of_copy_ceiling": (achieved / ceiling["ceiling"]) if ceiling else None,
        "e2e": e2e,
        "gpu_launches": args.reps * args.steps * launches_per_step,
        "clocks": clk,
        "wall_s_timed": wall,
    }
    if cpu_arrays is not None:
        thr = host_threads()
        val, secs, used = oracle_throughput(w_bench, N, 1, thr, cpu_arrays)
        n1 = min(N, args.ref_sample // 4)
        val1, secs1, _ = oracle_throughput(w_bench, n1, 1, 1)
        out["cpu_baseline"] = {"value": val, "unit": UNIT, "cores": used, "kind": "oracle",
                               "sample": f"one step over the whole {w.name} list "
                                         f"({N} params, the same drawn inputs), {secs:.2f} s "
                                         f"on {used} threads",
                               "single_thread": {"value": val1, "unit": UNIT, "cores": 1,
                                                 "sample": f"one step over the first {n1} "
                                                           f"params of the list, {secs1:.2f} s"}}
    for p in plans:
        p.close()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as it stands, on host cores, each step a bounded sample
    (the first elements of the same list)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = workload_of(args)
    thr = host_threads()
    n = min(args.ref_sample, w.total)
    oracle_throughput(w, min(n, 1 << 20), max(1, min(args.warmup, 3)), thr)  # warm-up
    val, secs, used = oracle_throughput(w, n, args.steps, thr)
    out = {
        "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": w.name, "n_params": w.total, "n_tensors": w.n_tensors,
                   "bytes_per_param": bytes_per_param(w), "sample_elems_per_step": n},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"first {n} elements of the {w.name} list per step"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--grad-buffers", type=int, default=4)
    ap.add_argument("--reps", type=int, default=5,
                    help="timed repetitions of --steps steps; the median is reported")
    ap.add_argument("--ref-sample", type=int, default=1 << 28)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ceiling", action="store_true")
    ap.add_argument("--no-fuse", action="store_true",
                    help="run clipped steps as three launches even where one fused launch fits")
    ap.add_argument("--mode", type=int, default=None,
                    help="run the workload's tensor list in another storage mode (0-4, or "
                         "16 + any-precision flags)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
