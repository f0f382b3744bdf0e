"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` function takes a loaded oracle (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with:
  * a library routine (torch's fp32->bf16 conversion, ``torch.optim.AdamW`` in
    fp32 and fp64, ``torch.nn.utils.clip_grad_norm_``, ``math.fsum``);
  * a closed form (first step from zero moments, constant-gradient
    trajectory, norm of a constant vector);
  * an invariant (Kahan-compensated bf16 tracks the exact trajectory where
    plain bf16 stalls; a skipped step writes nothing).
They are plain functions so that ``test_oracle_mutants`` can run every pin
against deliberately broken copies of the oracle and check that each broken
copy fails at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O

F32 = np.float32
EPS32 = 2.0 ** -24


# ------------------------------------------------------------------ helpers --

def torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 by torch (a library routine, round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=F32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (np.asarray(h).astype(np.uint32) << 16).view(F32).astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


def ulp_f32(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 23)


def f32(x) -> float:
    return float(np.float32(x))


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------- bf16 RNE ------

def _special_patterns() -> np.ndarray:
    pats = []
    for sign in (0, 0x80000000):
        for exp in range(0, 256):
            base = sign | (exp << 23)
            for mant_hi in (0x000000, 0x010000, 0x7E0000, 0x7F0000, 0x550000):
                for low in (0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
                    pats.append(base | mant_hi | low)
    pats += [0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x7F800000,
             0xFF800000, 0x7FC00000, 0x7F800001, 0xFFFFFFFF, 0x7FFFFFFF,
             0x00000001, 0x80000001, 0x00008000, 0x00018000, 0x00007FFF]
    return np.array(pats, dtype=np.uint32)


def pin_bf16_rne_vs_torch(o: O.Oracle, n_random: int = 1 << 22):
    pats = np.concatenate([_special_patterns(),
                           _rng(1).integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)])
    x = pats.view(F32)
    ours = o.f32_to_bf16(x)
    ref = torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.all(np.isnan(bf16_to_f64(ours[nan]))), "NaN must stay NaN"
    bad = np.nonzero((ours != ref) & ~nan)[0]
    assert bad.size == 0, f"bf16 RNE differs from torch at {pats[bad[:5]]}"
    # round trip of every bf16 pattern is the identity (finite and inf)
    allh = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    back = o.f32_to_bf16(o.bf16_to_f32(allh))
    fin = ~np.isnan(bf16_to_f64(allh))
    assert np.array_equal(back[fin], allh[fin])


def pin_bf16_rne_definition(o: O.Oracle, n: int = 1 << 18):
    """For finite x inside the bf16 range the result is the nearest bf16, ties
    to an even last mantissa bit; checked in fp64 against both neighbours."""
    r = _rng(2)
    x = (r.standard_normal(n) * np.exp2(r.integers(-120, 120, n))).astype(F32)
    h = o.f32_to_bf16(x)
    y = bf16_to_f64(h)
    xd = x.astype(np.float64)
    lo = bf16_to_f64((x.view(np.uint32) >> 16).astype(np.uint16))            # truncation
    hi_bits = ((x.view(np.uint32) >> 16) + 1).astype(np.uint16)
    hi = bf16_to_f64(hi_bits)
    assert np.all((y == lo) | (y == hi)), "result is not a neighbour of x"
    dlo, dhi = np.abs(xd - lo), np.abs(xd - hi)
    pick_lo = (dlo < dhi) | ((dlo == dhi) & (((x.view(np.uint32) >> 16) & 1) == 0))
    want = np.where(pick_lo, lo, hi)
    assert np.array_equal(y, want), "not nearest-even"


# ------------------------------------------------------ closed-form step 1 --

def _first_step_inputs(n=4096, seed=3):
    r = _rng(seed)
    g = (r.standard_normal(n) * 1e-2).astype(F32)
    g[:8] = [1e-8, -1e-8, 3e-8, 0.0, -0.0, 10.0, -7.5, 2.5e-9]
    g[8:16] = r.standard_normal(8).astype(F32) * 1e-6
    p = r.uniform(-4, 4, n).astype(F32)
    return p, g


def pin_first_step_mixed(o: O.Oracle):
    """t = 1 from m = v = 0: m_hat = g and v_hat = g^2, so the update is
    lr*g/(|g|+eps) + lr*wd*p in exact arithmetic."""
    p, g32 = _first_step_inputs()
    gh = torch_bf16_bits(g32)
    hp = O.hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    master, m, v = p.copy(), np.zeros_like(p), np.zeros_like(p)
    pout = np.zeros(p.size, np.uint16)
    o.mixed(master, gh, m, v, pout, hp, 1)
    g = bf16_to_f64(gh)
    lr, eps, wd = f32(1e-3), f32(1e-8), f32(0.1)
    adam = lr * g / (np.abs(g) + eps)
    want = p.astype(np.float64) - adam - lr * wd * p.astype(np.float64)
    err = np.abs(master - want)
    tol = ulp_f32(want) + 1e-6 * (np.abs(adam) + lr * wd * np.abs(p))
    assert np.all(err <= tol), f"master off by {np.max(err / tol):.3g} x tol"
    assert np.all(np.abs(m - (1 - f32(0.9)) * g) <= 2 * EPS32 * np.abs(m) + 1e-45)
    assert np.all(np.abs(v - (1 - f32(0.95)) * g * g) <= 4 * EPS32 * np.abs(v) + 1e-45)
    assert np.array_equal(pout, torch_bf16_bits(master)), "p_out must be bf16(master')"


def pin_first_step_bf16(o: O.Oracle):
    p32, g32 = _first_step_inputs(seed=4)
    ph, gh = torch_bf16_bits(p32), torch_bf16_bits(g32)
    hp = O.hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    p, m, v, c = ph.copy(), np.zeros_like(ph), np.zeros_like(ph), np.zeros_like(ph)
    o.bf16_kahan(p, gh, m, v, c, hp, 1)
    g, p0 = bf16_to_f64(gh), bf16_to_f64(ph)
    lr, eps, wd = f32(1e-3), f32(1e-8), f32(0.1)
    adam = lr * g / (np.abs(g) + eps)
    want = p0 - adam - lr * wd * p0
    pn, cn = bf16_to_f64(p), bf16_to_f64(c)
    # m_s, v_s are the bf16-rounded moments (8 significant bits: relative
    # rounding <= 2^-8 each, halved through the square root)
    tol = 6e-3 * np.abs(adam) + 0.5 * ulp_bf16(cn) * (cn != 0) + 8 * ulp_f32(p0)
    err = np.abs(pn + cn - want)
    assert np.all(err <= tol), f"p+c off by {np.max(err / tol):.3g} x tol"
    assert np.all(np.abs(pn - want) <= ulp_bf16(want) * 0.5 + tol), "p' not nearest bf16"
    mm, vv = bf16_to_f64(m), bf16_to_f64(v)
    assert np.all(np.abs(mm - (1 - f32(0.9)) * g) <= 2.0 ** -8 * np.abs(mm) + 1e-45)
    assert np.all(np.abs(vv - (1 - f32(0.95)) * g * g) <= 2.0 ** -8 * np.abs(vv) + 1e-45)


# ------------------------------------------- constant-gradient trajectory --

def pin_constant_grad_trajectory_mixed(o: O.Oracle, steps: int = 30):
    """Constant g keeps m_hat = g, v_hat = g^2 at every t, so
    p_t = (1-a) p_{t-1} - b with a = lr*wd, b = lr*g/(|g|+eps): a geometric
    closed form."""
    r = _rng(5)
    n = 2048
    gh = torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32))
    p = r.uniform(-1, 1, n).astype(F32)
    hp = O.hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    master, m, v = p.copy(), np.zeros_like(p), np.zeros_like(p)
    pout = np.zeros(n, np.uint16)
    for t in range(1, steps + 1):
        o.mixed(master, gh, m, v, pout, hp, t)
    g = bf16_to_f64(gh)
    lr, eps, wd = f32(1e-3), f32(1e-8), f32(0.1)
    a, b = lr * wd, lr * g / (np.abs(g) + eps)
    k = (1 - a) ** steps
    want = k * p.astype(np.float64) - b * (1 - k) / a
    err = np.abs(master - want)
    tol = steps * ulp_f32(np.maximum(np.abs(want), np.abs(p))) + 100 * EPS32 * steps * np.abs(b)
    assert np.all(err <= tol), f"trajectory off by {np.max(err / tol):.3g} x tol"


def pin_constant_grad_trajectory_bf16(o: O.Oracle, steps: int = 30):
    r = _rng(6)
    n = 2048
    gh = torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32))
    ph = torch_bf16_bits(r.uniform(-1, 1, n).astype(F32))
    hp = O.hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    p, m, v, c = ph.copy(), np.zeros_like(ph), np.zeros_like(ph), np.zeros_like(ph)
    for t in range(1, steps + 1):
        o.bf16_kahan(p, gh, m, v, c, hp, t)
    g, p0 = bf16_to_f64(gh), bf16_to_f64(ph)
    lr, eps, wd = f32(1e-3), f32(1e-8), f32(0.1)
    a, b = lr * wd, lr * g / (np.abs(g) + eps)
    k = (1 - a) ** steps
    want = k * p0 - b * (1 - k) / a
    got = bf16_to_f64(p) + bf16_to_f64(c)
    # bf16 moments: m_hat, v_hat off by O(2^-8) relative per step
    tol = 8e-3 * steps * np.abs(b) + ulp_bf16(bf16_to_f64(c)) + steps * ulp_f32(p0)
    err = np.abs(got - want)
    assert np.all(err <= tol), f"bf16 trajectory off by {np.max(err / tol):.3g} x tol"


# ------------------------------------------------ library special cases --

def _torch_adamw(params64_or_32, grads_per_step, lr, betas, eps, wd, max_norm=0.0):
    p = torch.nn.Parameter(params64_or_32.clone())
    opt = torch.optim.AdamW([p], lr=lr, betas=betas, eps=eps, weight_decay=wd,
                            foreach=False, fused=False)
    for g in grads_per_step:
        p.grad = g.clone()
        if max_norm > 0:
            torch.nn.utils.clip_grad_norm_([p], max_norm, foreach=False)
        opt.step()
    st = opt.state[p]
    return p.detach(), st["exp_avg"], st["exp_avg_sq"]


def _close(a, b, rel, name):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    floor = rel * np.max(np.abs(b))
    err = np.abs(a - b)
    tol = rel * np.abs(b) + floor
    assert np.all(err <= tol), f"{name}: off by {np.max(err / tol):.3g} x tol"


def pin_torch_adamw_mixed(o: O.Oracle, steps: int = 10, max_norm: float = 0.0):
    """Mixed mode equals torch.optim.AdamW (fp32, CPU) on the bf16-rounded
    gradients; with clipping, torch.nn.utils.clip_grad_norm_ first."""
    r = _rng(7 if max_norm == 0 else 8)
    n = 5000
    p = (r.standard_normal(n) * 0.02).astype(F32)
    grads_h = [torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32)) for _ in range(steps)]
    b1, b2 = f32(0.9), f32(0.95)
    hp = O.hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                   max_grad_norm=max_norm)
    master, m, v = p.copy(), np.zeros_like(p), np.zeros_like(p)
    pout = np.zeros(n, np.uint16)
    for t, gh in enumerate(grads_h, 1):
        coef = 1.0
        if max_norm > 0:
            coef, _ = o.clip_coef(o.grad_sumsq([gh])[0], max_norm)
        o.mixed(master, gh, m, v, pout, hp, t, coef)
    tg = [torch.from_numpy(bf16_to_f64(gh).astype(F32)) for gh in grads_h]
    tp, tm, tv = _torch_adamw(torch.from_numpy(p), tg, f32(2e-4), (b1, b2), f32(1e-8),
                              f32(0.1), max_norm)
    _close(master, tp.numpy(), 1e-6, "master")
    _close(m, tm.numpy(), 2e-6 if max_norm else 1e-6, "exp_avg")
    _close(v, tv.numpy(), 2e-6 if max_norm else 1e-6, "exp_avg_sq")


def pin_torch_adamw_mixed_clipped(o: O.Oracle):
    pin_torch_adamw_mixed(o, steps=10, max_norm=0.3)


def pin_torch_adamw_fp64_vs_bf16(o: O.Oracle, steps: int = 10):
    """Brute force: torch.optim.AdamW in fp64 on the same bf16 inputs.  The
    bf16 mode stores m and v in bf16, so they sit within a few bf16 ulps of the
    fp64 moments, and p + c within the accumulated moment rounding of the fp64
    parameter."""
    r = _rng(9)
    n = 64
    ph = torch_bf16_bits((r.standard_normal(n) * 0.02).astype(F32))
    grads_h = [torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32)) for _ in range(steps)]
    hp = O.hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    p, m, v, c = ph.copy(), np.zeros_like(ph), np.zeros_like(ph), np.zeros_like(ph)
    for t, gh in enumerate(grads_h, 1):
        o.bf16_kahan(p, gh, m, v, c, hp, t)
    tg = [torch.from_numpy(bf16_to_f64(gh)) for gh in grads_h]
    tp, tm, tv = _torch_adamw(torch.from_numpy(bf16_to_f64(ph)), tg, f32(2e-4),
                              (f32(0.9), f32(0.95)), f32(1e-8), f32(0.1))
    tp, tm, tv = tp.numpy(), tm.numpy(), tv.numpy()
    mm, vv = bf16_to_f64(m), bf16_to_f64(v)
    assert np.max(np.abs(mm - tm)) <= 0.02 * np.max(np.abs(tm)), "exp_avg vs fp64"
    assert np.max(np.abs(vv - tv)) <= 0.03 * np.max(np.abs(tv)), "exp_avg_sq vs fp64"
    got = bf16_to_f64(p) + bf16_to_f64(c)
    tol = 0.02 * steps * f32(2e-4) + ulp_bf16(bf16_to_f64(c))
    assert np.all(np.abs(got - tp) <= tol), "p + c vs fp64 parameter"
    assert np.all(np.abs(bf16_to_f64(p) - tp) <= ulp_bf16(tp) + tol), "p vs fp64"


# ------------------------------------------------------- Kahan invariant --

def pin_kahan_tracks_where_plain_stalls(o: O.Oracle, steps: int = 1000):
    """p = 1 in bf16 (ulp 2^-7) with lr = 1e-4: every update is below half an
    ulp.  Plain bf16 never moves; the compensated p + c follows the exact
    trajectory 1 - t*lr*g/(|g|+eps).

    The compensation is itself bf16: each step rounds c' once, and while p
    stays in [0.5, 1] the compensation is at most half an ulp of p (2^-9), so
    one rounding costs at most 2^-17 and 1000 steps at most 1000 * 2^-17
    (0.0076, against 0.1 of total movement that plain bf16 loses entirely).
    With b1 = b2 = 0 the moments are g and g^2 exactly (g has few significant
    bits) and that is the whole error budget.  With b1 = 0.9, b2 = 0.95 the
    bf16 moment EMAs stop short of g and g^2 by a few ulps (a known effect of
    bf16 state), which bends the trajectory by up to a few percent more."""
    n = 16
    gh = torch_bf16_bits(np.array([0.5, -0.5, 0.25, -0.125, 1.0, 3.0, -2.0, 0.75] * 2, F32))
    ph = torch_bf16_bits(np.ones(n, F32))
    g = bf16_to_f64(gh)
    lr, eps = f32(1e-4), f32(1e-8)
    want = 1.0 - steps * lr * g / (np.abs(g) + eps)
    for (b1, b2, rel) in ((0.0, 0.0, 0.0), (0.9, 0.95, 0.03)):
        hp = O.hparams(lr=1e-4, beta1=b1, beta2=b2, eps=1e-8, weight_decay=0.0)
        p, m, v, c = ph.copy(), np.zeros_like(ph), np.zeros_like(ph), np.zeros_like(ph)
        q, mq, vq = ph.copy(), np.zeros_like(ph), np.zeros_like(ph)
        for t in range(1, steps + 1):
            o.bf16_kahan(p, gh, m, v, c, hp, t)
            o.bf16_plain(q, gh, mq, vq, hp, t)
        assert np.array_equal(q, ph), "plain bf16 should stall at p0"
        got = bf16_to_f64(p) + bf16_to_f64(c)
        tol = rel * steps * lr + steps * 2.0 ** -17 + steps * 4 * EPS32 * lr
        err = np.abs(got - want)
        assert np.all(err <= tol), f"Kahan sum off by {np.max(err / tol):.3g} x tol (b={b1},{b2})"
        # and the bf16 parameter itself is within an ulp of the true value
        assert np.all(np.abs(bf16_to_f64(p) - want) <= ulp_bf16(want) + tol)


# ----------------------------------------------------------- norm / clip --

def pin_norm(o: O.Oracle):
    a = 0.375  # exact in bf16; a*a = 9/64 exact in fp64
    n = 1_000_000
    gh = np.full(n, torch_bf16_bits(np.array([a], F32))[0], np.uint16)
    s, bad = o.grad_sumsq([gh[:400_000], gh[400_000:]])
    assert s == n * a * a and not bad
    coef, norm = o.clip_coef(s, 1.0)
    assert norm == a * math.sqrt(n)
    assert coef == f32(min(1.0, 1.0 / (a * math.sqrt(n) + 1e-6)))
    # random values vs the exactly rounded sum of squares
    r = _rng(10)
    parts = [torch_bf16_bits((r.standard_normal(k) * 1e-2).astype(F32)) for k in (1, 7, 1000, 333_333)]
    s, bad = o.grad_sumsq(parts)
    exact = math.fsum(float(x) ** 2 for gp in parts for x in bf16_to_f64(gp))
    assert not bad and abs(s - exact) <= 1e-12 * exact
    ref = torch.linalg.vector_norm(torch.from_numpy(np.concatenate([bf16_to_f64(x) for x in parts])))
    _, norm = o.clip_coef(s, 1.0)
    assert abs(norm - float(ref)) <= 1e-12 * float(ref)
    # a long heavy-tailed list: the compensated fp64 sum equals the exactly
    # rounded sum (a plain running sum drifts low by ~1e-10 here)
    n_long = 20_000_000
    g32 = (r.standard_normal(n_long) * 1e-2).astype(F32)
    g32[r.random(n_long) < 0.01] *= 100.0
    gl = torch_bf16_bits(g32)
    s, bad = o.grad_sumsq([gl[:7_000_001], gl[7_000_001:]])
    x = bf16_to_f64(gl)
    exact = math.fsum(x * x)
    assert not bad and abs(s - exact) <= 4e-16 * exact, (s, exact)
    # no clipping below max_norm
    assert o.clip_coef(0.25, 1.0)[0] == 1.0
    assert o.clip_coef(4.0, 1.0)[0] == f32(1.0 / (2.0 + 1e-6))
    # non-finite flag
    for bad_val in (np.inf, -np.inf, np.nan):
        g = parts[3].copy()
        g[12345] = torch_bf16_bits(np.array([bad_val], F32))[0]
        _, flag = o.grad_sumsq([parts[0], g])
        assert flag, f"{bad_val} not flagged"


def pin_skip_on_nonfinite(o: O.Oracle):
    """With clipping on, a non-finite gradient anywhere in the list makes the
    step write nothing and report the skip."""
    r = _rng(11)
    sizes = [100, 37, 2048]
    hp = O.hparams(max_grad_norm=1.0)
    for mode in (0, 1):
        tens = []
        for n in sizes:
            g = torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32))
            if mode == 0:
                p = torch_bf16_bits((r.standard_normal(n) * 0.02).astype(F32))
                tens.append([p, g, torch_bf16_bits(r.standard_normal(n).astype(F32) * 1e-3),
                             torch_bf16_bits(np.abs(r.standard_normal(n)).astype(F32) * 1e-6),
                             np.zeros(n, np.uint16)])
            else:
                tens.append([(r.standard_normal(n) * 0.02).astype(F32), g,
                             np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)])
        tens[2][1][777] = torch_bf16_bits(np.array([np.inf], F32))[0]
        before = [[a.copy() for a in t] for t in tens]
        skipped, _ = o.list_step(tens, mode, hp, 1)
        assert skipped
        for t, b in zip(tens, before):
            for a, a0 in zip(t, b):
                assert np.array_equal(a.view(np.uint8), a0.view(np.uint8))
        tens[2][1][777] = 0
        skipped, _ = o.list_step(tens, mode, hp, 1)
        assert not skipped
        changed = any(not np.array_equal(t[0].view(np.uint8), b[0].view(np.uint8))
                      for t, b in zip(tens, before))
        assert changed


def pin_list_step_clipped_equals_torch(o: O.Oracle, steps: int = 5):
    """The list step with clipping: one coefficient from the global norm over
    every tensor of the list (torch.nn.utils.clip_grad_norm_ over the
    parameter list), then the mixed-mode step on each tensor
    (torch.optim.AdamW over the list), and the norm it reports is the square
    root of the sum of squares over all tensors."""
    r = _rng(24)
    sizes = [100, 37, 2048]
    ps = [(r.standard_normal(n) * 0.02).astype(F32) for n in sizes]
    grads = [[torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32)) for n in sizes]
             for _ in range(steps)]
    hp = O.hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_grad_norm=0.05)
    tens = [[p.copy(), None, np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)]
            for p, n in zip(ps, sizes)]
    for t, gs in enumerate(grads, 1):
        for e, g in zip(tens, gs):
            e[1] = g
        skipped, norm = o.list_step([tuple(e) for e in tens], 1, hp, t)
        assert not skipped
        want = math.sqrt(math.fsum(float(x) ** 2 for g in gs for x in bf16_to_f64(g)))
        assert abs(norm - want) <= 1e-14 * want, (norm, want)
        assert want > 0.05, "the clip must be active"
    tp = [torch.nn.Parameter(torch.from_numpy(p.copy())) for p in ps]
    opt = torch.optim.AdamW(tp, lr=f32(2e-4), betas=(f32(0.9), f32(0.95)), eps=f32(1e-8),
                            weight_decay=f32(0.1), foreach=False, fused=False)
    for gs in grads:
        for q, g in zip(tp, gs):
            q.grad = torch.from_numpy(bf16_to_f64(g).astype(F32))
        torch.nn.utils.clip_grad_norm_(tp, 0.05, foreach=False)
        opt.step()
    for e, q in zip(tens, tp):
        st = opt.state[q]
        _close(e[0], q.detach().numpy(), 1e-6, "master")
        _close(e[2], st["exp_avg"].numpy(), 2e-6, "exp_avg")
        _close(e[3], st["exp_avg_sq"].numpy(), 2e-6, "exp_avg_sq")
        assert np.array_equal(e[4], torch_bf16_bits(e[0])), "p_out must be bf16(master')"


def pin_bias_correction_powers(o: O.Oracle):
    """The per-step scalars against the closed forms with the library's fp64
    pow: step_size = lr/(1-b1^t), sbc2 = sqrt(1-b2^t), 1-b1, 1-b2, lr*wd,
    each rounded once to fp32.  Binary exponentiation is within a few fp64
    ulps of pow, so the fp32 scalars agree to at most one fp32 ulp (and
    exactly at t = 1, 2 where both are exact products)."""
    for b1, b2 in ((0.9, 0.95), (0.9, 0.999), (0.5, 0.25), (0.0, 0.0), (0.99, 0.9999)):
        hp = O.hparams(lr=2e-4, beta1=b1, beta2=b2, weight_decay=0.1)
        fb1, fb2, lr, wd = f32(b1), f32(b2), f32(2e-4), f32(0.1)
        for t in (1, 2, 3, 7, 10, 100, 1000, 12345, 10**6, 10**9):
            got = o.step_scalars(hp, t).astype(np.float64)
            want = np.array([lr / (1 - math.pow(fb1, t)), math.sqrt(1 - math.pow(fb2, t)),
                             1 - fb1, 1 - fb2, lr * wd], dtype=np.float32).astype(np.float64)
            tol = np.zeros(5) if t <= 2 else ulp_f32(want)
            assert np.all(np.abs(got - want) <= tol), (b1, b2, t, got, want)


# ------------------------------------------- other AnyPrecision options --

def pin_first_step_bf16_plain_and_v32(o: O.Oracle):
    """t = 1 closed form for the two other storage options: without
    compensation p' is the nearest bf16 to p - upd; with fp32 variance only
    the bf16 momentum rounds (half the error budget of the all-bf16 mode)."""
    p32, g32 = _first_step_inputs(seed=14)
    ph, gh = torch_bf16_bits(p32), torch_bf16_bits(g32)
    hp = O.hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    g, p0 = bf16_to_f64(gh), bf16_to_f64(ph)
    lr, eps, wd = f32(1e-3), f32(1e-8), f32(0.1)
    adam = lr * g / (np.abs(g) + eps)
    want = p0 - adam - lr * wd * p0
    # no compensation
    p, m, v = ph.copy(), np.zeros_like(ph), np.zeros_like(ph)
    o.bf16_plain(p, gh, m, v, hp, 1)
    err = np.abs(bf16_to_f64(p) - want)
    assert np.all(err <= 0.5 * ulp_bf16(want) + 6e-3 * np.abs(adam) + 8 * ulp_f32(p0))
    # fp32 variance: v exact to fp32, p + c within the bf16-momentum error
    p, m, c = ph.copy(), np.zeros_like(ph), np.zeros_like(ph)
    v32 = np.zeros(ph.size, F32)
    o.bf16_kahan_v32(p, gh, m, v32, c, hp, 1)
    assert np.all(np.abs(v32 - (1 - f32(0.95)) * g * g) <= 4 * EPS32 * np.abs(v32) + 1e-45)
    got = bf16_to_f64(p) + bf16_to_f64(c)
    cn = bf16_to_f64(c)
    tol = 4.1e-3 * np.abs(adam) + 0.5 * ulp_bf16(cn) * (cn != 0) + 8 * ulp_f32(p0)
    assert np.all(np.abs(got - want) <= tol), f"v32 first step off by {np.max(np.abs(got - want) / tol):.3g}"


def pin_torch_adamw_fp64_vs_v32(o: O.Oracle, steps: int = 10):
    """fp32 variance mode against fp64 torch.optim.AdamW: the variance agrees
    to fp32 rounding (1e-5 relative after 10 steps), unlike the bf16 variance
    of the all-bf16 mode; momentum within its bf16 storage error."""
    r = _rng(15)
    n = 64
    ph = torch_bf16_bits((r.standard_normal(n) * 0.02).astype(F32))
    grads_h = [torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32)) for _ in range(steps)]
    hp = O.hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    p, m, c = ph.copy(), np.zeros_like(ph), np.zeros_like(ph)
    v = np.zeros(n, F32)
    for t, gh in enumerate(grads_h, 1):
        o.bf16_kahan_v32(p, gh, m, v, c, hp, t)
    tg = [torch.from_numpy(bf16_to_f64(gh)) for gh in grads_h]
    tp, tm, tv = _torch_adamw(torch.from_numpy(bf16_to_f64(ph)), tg, f32(2e-4),
                              (f32(0.9), f32(0.95)), f32(1e-8), f32(0.1))
    tp, tm, tv = tp.numpy(), tm.numpy(), tv.numpy()
    # v is fed by the exact bf16 gradients; only m's bf16 rounding differs
    assert np.all(np.abs(v - tv) <= 1e-5 * np.abs(tv) + 1e-30), "fp32 variance vs fp64"
    assert np.max(np.abs(bf16_to_f64(m) - tm)) <= 0.02 * np.max(np.abs(tm))
    got = bf16_to_f64(p) + bf16_to_f64(c)
    assert np.all(np.abs(got - tp) <= 0.02 * steps * f32(2e-4) + ulp_bf16(bf16_to_f64(c)))


def pin_lr_linear_warmup(o: O.Oracle):
    """The recipe's linear schedule with 500 warm-up steps (here over 1000
    training steps): lr 0 on the first update, half at 250 applied steps,
    the peak at 500, half again at 750, 0 from 1000 on; linear in between."""
    base, W_, T_ = f32(2e-4), 500, 1000
    lr = lambda t: o.lr_linear_warmup(base, t, W_, T_)
    assert lr(1) == 0.0
    assert lr(251) == f32(base * 0.5) and lr(501) == base and lr(751) == f32(base * 0.5)
    assert lr(1001) == 0.0 and lr(5000) == 0.0
    up = [lr(t) for t in range(1, 502)]
    down = [lr(t) for t in range(501, 1002)]
    assert all(a <= b for a, b in zip(up, up[1:])) and all(a >= b for a, b in zip(down, down[1:]))
    assert abs(lr(101) - base * 100 / 500) <= 2 * EPS32 * base
    # no warm-up: the peak from the first update
    assert o.lr_linear_warmup(base, 1, 0, 1000) == base


# ------------------------------------------------------- remainder mode --

def pin_remainder_split_roundtrip(o: O.Oracle, n_random: int = 1 << 22):
    """bf16 high half + int16 remainder hold an fp32 value exactly, and the
    high half is the nearest bf16 (torch's RNE) except at exact ties, which
    go away from zero."""
    pats = np.concatenate([_special_patterns(),
                           _rng(12).integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)])
    x = pats.view(F32)
    p16, r16 = o.split_master(x)
    back = o.join_master(p16, r16)
    assert np.array_equal(back.view(np.uint32), pats), "split/join is not exact"
    nan = np.isnan(x)
    tie = (pats & 0xFFFF) == 0x8000
    ref = torch_bf16_bits(x)
    ok = ~nan & ~tie
    assert np.array_equal(p16[ok], ref[ok]), "high half is not the nearest bf16"
    assert np.array_equal(p16[tie & ~nan], ((pats[tie & ~nan] >> 16) + 1).astype(np.uint16))
    assert np.all(np.abs(r16.astype(np.int32)) <= 0x8000)


def pin_remainder_equals_mixed_master(o: O.Oracle, steps: int = 12):
    """Remainder mode stores the same fp32 master as the mixed mode, so its
    trajectory is the mixed mode's bit for bit (itself pinned to
    torch.optim.AdamW), and the bf16 parameter is that master's high half."""
    r = _rng(13)
    n = 5000
    p0 = torch_bf16_bits((r.standard_normal(n) * 0.02).astype(F32))   # bf16-exact start
    hp = O.hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_grad_norm=0.5)
    master = bf16_to_f64(p0).astype(F32)
    m, v, pout = np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)
    p16, r16 = p0.copy(), np.zeros(n, np.int16)
    m2, v2 = np.zeros(n, F32), np.zeros(n, F32)
    for t in range(1, steps + 1):
        gh = torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32))
        coef, _ = o.clip_coef(o.grad_sumsq([gh])[0], 0.5)
        o.mixed(master, gh, m, v, pout, hp, t, coef)
        o.remainder(p16, gh, m2, v2, r16, hp, t, coef)
    joined = o.join_master(p16, r16)
    assert np.array_equal(joined.view(np.uint32), master.view(np.uint32)), "master differs"
    assert np.array_equal(m2.view(np.uint32), m.view(np.uint32))
    assert np.array_equal(v2.view(np.uint32), v.view(np.uint32))
    hi, _ = o.split_master(master)
    assert np.array_equal(hi, p16)
    assert np.any(r16 != 0), "updates must leave a remainder"
    # the bf16 parameter is within half a bf16 ulp of the master
    assert np.all(np.abs(bf16_to_f64(p16) - joined) <= 0.5 * ulp_bf16(joined))


# ---------------------------------------------- any-precision storage --

# Every valid combination of the any-precision flags (1: fp32 exp_avg, 2: fp32
# exp_avg_sq, 4: fp32 compensation, 8: no Kahan summation; 4 needs Kahan).
ANY_FLAGS = [f for f in range(16) if (f & 12) != 12]


# Half a bf16 ulp, with room for the fp64 evaluation of the expected value.
HALF_ULP = 0.5 * (1.0 + 2.0 ** -10)


def _anyprec_state(flags: int, ph: np.ndarray):
    dm, dv, dc = O.anyprec_dtypes(flags)
    n = ph.size
    return (ph.copy(), np.zeros(n, dm), np.zeros(n, dv),
            None if dc is None else np.zeros(n, dc))


def _f64(a: np.ndarray) -> np.ndarray:
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def _anyprec_params(r, n: int) -> np.ndarray:
    """Half of the elements in [0.5, 2) in magnitude, where updates of about
    lr = 3e-3 are below half a bf16 ulp and only the compensation moves them;
    half around N(0, 0.02), where every update moves the bf16 parameter."""
    big = r.uniform(0.5, 2.0, n // 2) * r.choice([-1.0, 1.0], n // 2)
    small = r.standard_normal(n - n // 2) * 0.02
    return torch_bf16_bits(np.concatenate([big, small]).astype(F32))


def pin_anyprec_matches_named_modes(o: O.Oracle, steps: int = 20):
    """Flags 0, 2 and 8 store exactly what the all-bf16 Kahan step, the
    fp32-variance Kahan step and the uncompensated step store (each pinned on
    its own above), with and without a clip coefficient."""
    r = _rng(21)
    n = 257
    ph = _anyprec_params(r, n)
    grads = [torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32)) for _ in range(steps)]
    for coef, max_norm in ((1.0, 0.0), (0.37, 1.0)):
        hp = O.hparams(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                       max_grad_norm=max_norm)
        for flags in (0, 2, 8):
            a = _anyprec_state(flags, ph)
            b = _anyprec_state(flags, ph)
            for t, gh in enumerate(grads, 1):
                o.anyprec(a[0], gh, a[1], a[2], a[3], flags, hp, t, coef)
                if flags == 0:
                    o.bf16_kahan(b[0], gh, b[1], b[2], b[3], hp, t, coef)
                elif flags == 2:
                    o.bf16_kahan_v32(b[0], gh, b[1], b[2], b[3], hp, t, coef)
                else:
                    o.bf16_plain(b[0], gh, b[1], b[2], hp, t, coef)
            for x, y in zip(a, b):
                if x is not None:
                    assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), \
                        f"flags {flags} differ from the named mode"


def pin_anyprec_step_definition(o: O.Oracle, steps: int = 40):
    """Every combination, every step, against the textbook update in fp64
    evaluated on the values the step stored:
      m_t = b1 m_{t-1} + (1-b1) g,  v_t = b2 v_{t-1} + (1-b2) g^2
      upd = lr/(1-b1^t) * m_t / (sqrt(v_t)/sqrt(1-b2^t) + eps) + lr wd p_{t-1}
    Kahan: p_t + c_t = p_{t-1} + c_{t-1} - upd; otherwise p_t is the nearest
    bf16 to p_{t-1} - upd.  Allowed error: the fp32 roundings of the step (a
    few units of 2^-24 relative) plus half a bf16 ulp for each value stored
    as bf16 (attained at ties, hence HALF_ULP a hair above 1/2, against a
    full ulp for a wrong rounding) -- so a buffer stored in the wrong type, a
    wrong sign or a dropped term fails."""
    r = _rng(22)
    n = 64
    ph = _anyprec_params(r, n)
    grads = []
    for _ in range(steps):
        g = r.standard_normal(n) * 1e-2
        g[r.random(n) < 0.05] *= 100.0
        grads.append(torch_bf16_bits(g.astype(F32)))
    lr, b1, b2, eps, wd = f32(3e-3), f32(0.9), f32(0.95), f32(1e-8), f32(0.1)
    hp = O.hparams(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    for flags in ANY_FLAGS:
        p, m, v, c = _anyprec_state(flags, ph)
        m32, v32, c32, kahan = flags & 1, flags & 2, flags & 4, not flags & 8
        for t, gh in enumerate(grads, 1):
            p0, m0, v0 = _f64(p), _f64(m), _f64(v)
            c0 = _f64(c) if kahan else None
            o.anyprec(p, gh, m, v, c, flags, hp, t)
            g = bf16_to_f64(gh)
            m1, v1 = _f64(m), _f64(v)
            # moments, each in its own storage type
            want = b1 * m0 + (1.0 - b1) * g
            tol = 4 * EPS32 * (np.abs(b1 * m0) + np.abs((1.0 - b1) * g))
            tol = tol + (0.0 if m32 else HALF_ULP * ulp_bf16(m1))
            assert np.all(np.abs(m1 - want) <= tol + 1e-45), f"exp_avg, flags {flags}, t {t}"
            want = b2 * v0 + (1.0 - b2) * g * g
            tol = 5 * EPS32 * (np.abs(b2 * v0) + np.abs((1.0 - b2) * g * g))
            tol = tol + (0.0 if v32 else HALF_ULP * ulp_bf16(v1))
            assert np.all(np.abs(v1 - want) <= tol + 1e-45), f"exp_avg_sq, flags {flags}, t {t}"
            # the update from the stored moments
            bc1 = 1.0 - float(b1) ** t
            bc2 = 1.0 - float(b2) ** t
            adam = (lr / bc1) * m1 / (np.sqrt(v1) / math.sqrt(bc2) + eps)
            decay = lr * wd * p0
            upd = adam + decay
            tol_upd = 12 * EPS32 * (np.abs(adam) + np.abs(decay))
            p1 = bf16_to_f64(p)
            if kahan:
                c1 = _f64(c)
                y = c0 - upd
                err = np.abs((p1 + c1) - (p0 + c0 - upd))
                tol = (tol_upd + 2 * EPS32 * np.abs(y) + 2 * EPS32 * np.abs(p1 - p0)
                       + (2 * ulp_f32(c1) if c32 else HALF_ULP * ulp_bf16(c1) + ulp_f32(c1)))
                assert np.all(err <= tol), \
                    f"p + c, flags {flags}, t {t}: off by {np.max(err / tol):.3g} x tol"
            else:
                err = np.abs(p1 - (p0 - upd))
                tol = HALF_ULP * ulp_bf16(p1) + ulp_f32(p0 - upd) + tol_upd
                assert np.all(err <= tol), \
                    f"p, flags {flags}, t {t}: off by {np.max(err / tol):.3g} x tol"


def pin_anyprec_fp32_state_vs_torch(o: O.Oracle, steps: int = 200):
    """fp32 momentum, variance and compensation on a bf16 parameter behave as
    an fp32-master AdamW: over 200 steps p + c follows torch.optim.AdamW in
    fp64 (no weight decay, so the bf16 parameter's decay term cannot differ
    from the master's) to within the fp32 rounding of the update, although
    no update is large enough to move a bf16 parameter of magnitude >= 0.5
    by itself -- the same step without Kahan summation never moves them."""
    r = _rng(23)
    n = 64
    mag = r.uniform(0.5, 2.0, n) * r.choice([-1.0, 1.0], n)
    ph = torch_bf16_bits(mag.astype(F32))
    grads = [torch_bf16_bits((r.standard_normal(n) * 1e-2).astype(F32)) for _ in range(steps)]
    hp = O.hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)
    p, m, v, c = _anyprec_state(7, ph)
    q, mq, vq, _ = _anyprec_state(8 | 3, ph)
    for t, gh in enumerate(grads, 1):
        o.anyprec(p, gh, m, v, c, 7, hp, t)
        o.anyprec(q, gh, mq, vq, None, 8 | 3, hp, t)
    assert np.array_equal(q, ph), "without compensation the bf16 parameters stall"
    assert np.array_equal(m, mq) and np.array_equal(v, vq), "moments do not depend on p"
    tg = [torch.from_numpy(bf16_to_f64(gh)) for gh in grads]
    tp, tm, tv = _torch_adamw(torch.from_numpy(bf16_to_f64(ph)), tg, f32(1e-3),
                              (f32(0.9), f32(0.95)), f32(1e-8), 0.0)
    tp, tm, tv = tp.numpy(), tm.numpy(), tv.numpy()
    _close(m, tm, 2e-5, "fp32 exp_avg vs fp64")
    _close(v, tv, 2e-5, "fp32 exp_avg_sq vs fp64")
    got = bf16_to_f64(p) + c.astype(np.float64)
    moved = np.abs(tp - bf16_to_f64(ph))
    assert np.min(moved) > 0.0 and np.max(moved) > 0.02, "the trajectory must move"
    err = np.abs(got - tp)
    tol = steps * f32(1e-3) * 2e-5
    assert np.all(err <= tol), f"p + c vs fp64 master: off by {np.max(err / tol):.3g} x tol"


ALL_PINS = [
    pin_list_step_clipped_equals_torch,
    pin_anyprec_matches_named_modes,
    pin_anyprec_step_definition,
    pin_anyprec_fp32_state_vs_torch,
    pin_first_step_bf16_plain_and_v32,
    pin_torch_adamw_fp64_vs_v32,
    pin_lr_linear_warmup,
    pin_remainder_split_roundtrip,
    pin_remainder_equals_mixed_master,
    pin_bias_correction_powers,
    pin_bf16_rne_vs_torch,
    pin_bf16_rne_definition,
    pin_first_step_mixed,
    pin_first_step_bf16,
    pin_constant_grad_trajectory_mixed,
    pin_constant_grad_trajectory_bf16,
    pin_torch_adamw_mixed,
    pin_torch_adamw_mixed_clipped,
    pin_torch_adamw_fp64_vs_bf16,
    pin_kahan_tracks_where_plain_stalls,
    pin_norm,
    pin_skip_on_nonfinite,
]
