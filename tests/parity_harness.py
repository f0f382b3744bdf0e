"""Runs a workload through the CUDA library and through the CPU oracle on the
same seeded bytes, and compares the results element by element.

Tolerances (checked in ``compare``):
  * bf16 state (p, m, v, c, bf16 param out): at most 1 bf16 ulp apart; NaN
    only where the other side has NaN;
  * fp32 state (master, m, v): relative error <= 1e-6, with an absolute floor
    of 1e-6 * max|x| of the finite values of the tensor for values near
    zero; NaN and +-inf at the same places on both sides;
  * the non-finite flag: identical.
Both sides evaluate the same fp32 operation sequence, so the results are
expected to be bit-identical; the report counts exact matches (a NaN on both
sides counts as a match whatever its payload).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle as O
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import workloads as W

THREADS = max(1, min(16, os.cpu_count() or 1))


def to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


def to_np(t: torch.Tensor | None) -> np.ndarray | None:
    """Host copy with the oracle's dtype: bf16 -> uint16 bits, int16, fp32."""
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return to_u16(t)
    if t.dtype == torch.int16:
        return t.detach().contiguous().cpu().numpy()
    return to_f32(t)


def hp_pair(w: W.Workload):
    h = w.hparams()
    return A.hparams(**h), O.hparams(**h)


# ------------------------------------------------------------ comparing --

def _ordered(h: np.ndarray) -> np.ndarray:
    k = h.astype(np.int32)
    return np.where(k & 0x8000, -(k & 0x7FFF), k)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray):
    """(max ulp distance over non-NaN pairs, NaN positions agree, exact count)."""
    fa = (a.astype(np.uint32) << 16).view(np.float32)
    fb = (b.astype(np.uint32) << 16).view(np.float32)
    na, nb = np.isnan(fa), np.isnan(fb)
    ok = ~(na | nb)
    d = np.abs(_ordered(a[ok]) - _ordered(b[ok]))
    return (int(d.max()) if d.size else 0), bool(np.array_equal(na, nb)), int(np.sum(a == b) + np.sum(na & nb))


@dataclass
class Report:
    max_ulp: int = 0
    max_rel: float = 0.0
    n: int = 0
    exact: int = 0
    failures: list = field(default_factory=list)

    def ok(self):
        return not self.failures


def compare(rep: Report, name: str, gpu: np.ndarray, ref: np.ndarray):
    if gpu.dtype == np.int16:   # remainder of the master: must be exact
        rep.n += gpu.size
        rep.exact += int(np.sum(gpu == ref))
        if not np.array_equal(gpu, ref):
            rep.failures.append(f"{name}: {int(np.sum(gpu != ref))} remainders differ")
        return
    if gpu.dtype == np.uint16:
        mu, nan_ok, ex = bf16_ulp_diff(gpu, ref)
        rep.max_ulp = max(rep.max_ulp, mu)
        rep.n += gpu.size
        rep.exact += ex
        if mu > 1 or not nan_ok:
            rep.failures.append(f"{name}: max {mu} bf16 ulp, NaN positions agree={nan_ok}")
    else:
        g64, r64 = gpu.astype(np.float64), ref.astype(np.float64)
        nan_g, nan_r = np.isnan(g64), np.isnan(r64)
        # infinities must sit at the same places with the same sign
        inf_g, inf_r = np.isinf(g64), np.isinf(r64)
        inf_ok = np.array_equal(inf_g, inf_r) and np.array_equal(g64[inf_g], r64[inf_r])
        ok = ~(nan_g | nan_r | inf_g | inf_r)
        floor = 1e-6 * (np.max(np.abs(r64[ok])) if ok.any() else 0.0)
        err = np.abs(g64[ok] - r64[ok])
        tol = 1e-6 * np.abs(r64[ok]) + floor
        rel = float(np.max(err / np.maximum(np.abs(r64[ok]), floor if floor > 0 else 1e-300))) if err.size else 0.0
        rep.max_rel = max(rep.max_rel, rel)
        rep.n += gpu.size
        # a NaN's payload and sign are not part of the result (IEEE leaves the
        # payload of a generated NaN open; x86, Arm and CUDA differ): NaN
        # pairs count as matching, as in the bf16 comparison
        rep.exact += int(np.sum((gpu.view(np.uint32) == ref.view(np.uint32)) | (nan_g & nan_r)))
        if not np.array_equal(nan_g, nan_r) or not inf_ok or np.any(err > tol):
            rep.failures.append(f"{name}: max rel {rel:.3g} beyond 1e-6 (or NaN / inf mismatch)")


# -------------------------------------------------------------- the GPU side --

class GpuSide:
    """A workload's state on the GPU plus a plan over its tensor list."""

    def __init__(self, w: W.Workload, device="cuda", state: W.State | None = None):
        self.w = w
        self.st = state or W.make_state(w, device)
        self.g = torch.zeros(self.st.param.numel(), dtype=torch.bfloat16, device=self.st.param.device)
        v = self.st.views
        self.plan = A.Plan(v(self.st.param), v(self.g), v(self.st.exp_avg), v(self.st.exp_avg_sq),
                           v(self.st.aux), w.mode, norm=True)
        self.norm = torch.zeros(1, dtype=torch.float64, device=device)
        self.flag = torch.zeros(1, dtype=torch.int32, device=device)
        self.t = 0

    def set_grad(self, k: int):
        self.g.copy_(W.make_grad(self.w, k, self.g.device, self.st.offsets, self.g.numel()))

    def step(self, hp: A.adamw_hparams_t, want_flag: bool = True) -> bool:
        """One step at t = applied + 1; returns True when it was skipped."""
        clip = hp.max_grad_norm > 0
        self.plan.step(hp, self.t + 1, grad_norm=self.norm if clip else None,
                       nonfinite=self.flag if (clip or want_flag) else None)
        skipped = clip and bool(self.flag.item())
        if not skipped:
            self.t += 1
        return skipped


# ----------------------------------------------------------- the CPU side --

class OracleRun:
    """The same list as host numpy arrays, stepped by the oracle."""

    def __init__(self, w: W.Workload, arrays: dict, numels: list[int], offsets: list[int]):
        self.w, self.o = w, O.load()
        self.a = arrays
        self.numels, self.offsets = numels, offsets
        self.t = 0

    @classmethod
    def from_state(cls, st: W.State):
        w = st.workload
        arrays = dict(param=to_np(st.param), exp_avg=to_np(st.exp_avg),
                      exp_avg_sq=to_np(st.exp_avg_sq), aux=to_np(st.aux))
        return cls(w, arrays, w.numels, st.offsets)

    def step_arrays(self, p, g, m, v, a, t, coef, hp):
        if self.w.mode == W.MODE_BF16_KAHAN:
            self.o.bf16_kahan(p, g, m, v, a, hp, t, coef)
        elif self.w.mode == W.MODE_MIXED:
            self.o.mixed(p, g, m, v, a, hp, t, coef)
        elif self.w.mode == W.MODE_REMAINDER:
            self.o.remainder(p, g, m, v, a, hp, t, coef)
        elif self.w.mode == W.MODE_BF16_PLAIN:
            self.o.bf16_plain(p, g, m, v, hp, t, coef)
        elif self.w.mode == W.MODE_BF16_KAHAN_V32:
            self.o.bf16_kahan_v32(p, g, m, v, a, hp, t, coef)
        else:
            self.o.anyprec(p, g, m, v, a, self.w.mode - W.MODE_ANYPREC, hp, t, coef)

    def views(self, name, k):
        o, n = self.offsets[k], self.numels[k]
        return None if self.a[name] is None else self.a[name][o:o + n]

    def step(self, g_flat: np.ndarray, hp: O.Hparams):
        """Returns (skipped, norm, nonfinite)."""
        o = self.o
        gs = [g_flat[off:off + n] for off, n in zip(self.offsets, self.numels)]
        sumsq, bad = o.grad_sumsq(gs)
        coef, norm = o.clip_coef(sumsq, hp.max_grad_norm if hp.max_grad_norm > 0 else 1.0)
        clip = hp.max_grad_norm > 0
        if clip and bad:
            return True, norm, bad
        if not clip:
            coef = 1.0
        t = self.t + 1

        def one(k):
            if self.numels[k] == 0:
                return
            p, m, v, a = (self.views(x, k) for x in ("param", "exp_avg", "exp_avg_sq", "aux"))
            self.step_arrays(p, gs[k], m, v, a, t, coef, hp)

        order = sorted(range(len(self.numels)), key=lambda k: -self.numels[k])
        with ThreadPoolExecutor(THREADS) as ex:
            list(ex.map(one, order))
        self.t = t
        return False, norm, bad


def compare_state(gpu: GpuSide, ref: OracleRun, rep: Report | None = None) -> Report:
    rep = rep or Report()
    st = gpu.st
    got = dict(param=to_np(st.param), exp_avg=to_np(st.exp_avg), exp_avg_sq=to_np(st.exp_avg_sq),
               aux=to_np(st.aux))
    for k, (o, n) in enumerate(zip(ref.offsets, ref.numels)):
        if n == 0:
            continue
        for name in ("param", "exp_avg", "exp_avg_sq", "aux"):
            if got[name] is not None:
                compare(rep, f"tensor {k} {name}", got[name][o:o + n], ref.a[name][o:o + n])
    return rep


def run_parity(w: W.Workload, steps: int | None = None, device="cuda",
               align_elems: int = 8, skew: int = 0) -> tuple[Report, list]:
    """Full-list parity: every element of every tensor after every step."""
    steps = steps or w.steps
    gpu = GpuSide(w, device, W.make_state(w, device, align_elems, skew))
    ref = OracleRun.from_state(gpu.st)
    hp_g, hp_o = hp_pair(w)
    log = []
    rep = Report()
    for k in range(1, steps + 1):
        gpu.set_grad(k)
        skipped = gpu.step(hp_g)
        oskipped, onorm, obad = ref.step(to_u16(gpu.g), hp_o)
        flag = bool(gpu.flag.item())
        log.append((k, skipped, oskipped, flag, obad, float(gpu.norm.item()), onorm))
        if skipped != oskipped or flag != obad:
            rep.failures.append(f"step {k}: skip/flag gpu=({skipped},{flag}) oracle=({oskipped},{obad})")
    compare_state(gpu, ref, rep)
    gpu.plan.close()
    return rep, log


# --------------------------------------------------- sampled (full size) --

def sample_indices(gpu: GpuSide, per_tensor: int, seed: int = 0) -> np.ndarray:
    """Flat-buffer indices to check: per tensor its first and last 9
    elements, ``per_tensor`` random ones, and the elements around every chunk
    boundary of the plan (where CTAs hand over and vector bodies start)."""
    w, st = gpu.w, gpu.st
    rng = np.random.default_rng(seed)
    idx = []
    for o, n in zip(st.offsets, w.numels):
        if n == 0:
            continue
        idx.append(o + np.arange(min(n, 9)))
        idx.append(o + np.arange(max(0, n - 9), n))
        idx.append(o + rng.integers(0, n, min(n, per_tensor)))
    entries = []
    v = st.views
    for tensors in zip(v(st.param), v(gpu.g), v(st.exp_avg), v(st.exp_avg_sq), v(st.aux)):
        entries.append(tuple(t.data_ptr() if t is not None else 0 for t in tensors)
                       + (tensors[0].numel(),))
    for c in A.adamw_plan_chunks(entries, w.mode, gpu.plan.info.grid):
        o = st.offsets[c.tensor] + c.offset
        for d in (0, 1, 7, 8, c.len - 9, c.len - 8, c.len - 1):
            if 0 <= d < c.len:
                idx.append(np.array([o + d]))
    return np.unique(np.concatenate(idx))


def run_sampled(w: W.Workload, per_tensor: int = 2048, steps: int | None = None,
                device="cuda") -> tuple[Report, list]:
    """Full-size parity on sampled elements: the update is elementwise, so the
    oracle steps only the sampled elements (with the clip coefficient from its
    own norm over the full gradient) and the GPU's values at those elements
    must match."""
    steps = steps or w.steps
    gpu = GpuSide(w, device)
    idx = sample_indices(gpu, per_tensor)
    it = torch.from_numpy(idx).to(device)
    st = gpu.st
    take = lambda x: None if x is None else to_np(x[it])
    arrays = dict(param=take(st.param), exp_avg=take(st.exp_avg),
                  exp_avg_sq=take(st.exp_avg_sq), aux=take(st.aux))
    ref = OracleRun(w, arrays, [idx.size], [0])
    o = ref.o
    hp_g, hp_o = hp_pair(w)
    clip = w.max_grad_norm > 0
    log, rep = [], Report()
    for k in range(1, steps + 1):
        gpu.set_grad(k)
        skipped = gpu.step(hp_g)
        flag = bool(gpu.flag.item())
        g_s = to_u16(gpu.g[it])
        # the oracle's own global norm and flag over the full gradient
        g_full = to_u16(gpu.g)
        sumsq, bad = o.grad_sumsq([g_full[off:off + n] for off, n in zip(st.offsets, w.numels)])
        del g_full
        coef, norm = o.clip_coef(sumsq, w.max_grad_norm if clip else 1.0)
        oskipped = clip and bad
        if not oskipped:
            ref.t += 1
            p, m, v, a = (ref.a[x] for x in ("param", "exp_avg", "exp_avg_sq", "aux"))
            ref.step_arrays(p, g_s, m, v, a, ref.t, coef if clip else 1.0, hp_o)
        gnorm = float(gpu.norm.item()) if clip else float("nan")
        log.append((k, skipped, oskipped, flag, bad, gnorm, norm))
        if skipped != oskipped or flag != bad:
            rep.failures.append(f"step {k}: skip/flag gpu=({skipped},{flag}) oracle=({oskipped},{bad})")
        if clip and abs(gnorm - norm) > 1e-12 * norm:
            rep.failures.append(f"step {k}: norm gpu {gnorm!r} oracle {norm!r}")
    got = dict(param=take(st.param), exp_avg=take(st.exp_avg),
               exp_avg_sq=take(st.exp_avg_sq), aux=take(st.aux))
    for name in ("param", "exp_avg", "exp_avg_sq", "aux"):
        if got[name] is not None:
            compare(rep, f"sampled {name}", got[name], ref.a[name])
    gpu.plan.close()
    return rep, log
