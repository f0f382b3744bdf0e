"""GPU parity at the edges of the method and of the sizes, through the C ABI,
against the oracle: a tensor longer than 2^31 elements, tens of thousands of
tiny tensors, degenerate hyperparameters (betas 0, lr 0, a variance decay
next to 1, eps 1, t near 10^9) and degenerate gradients (all zero, bf16
subnormals, magnitudes whose squares overflow fp32, signed zeros).  Same
tolerances as the other parity tests; every case here is bit-identical and
the tests assert it."""
import numpy as np
import pytest
import torch

import parity_harness as H
from adamw_optimizer_step_sm_gb300 import workloads as W
from test_gpu_parity import _assert, _small

pytestmark = pytest.mark.gpu


def _run_custom(w, grad_fn, steps, t0=0, state=None):
    """Full parity over ``steps`` steps whose gradients ``grad_fn(k, g)``
    writes into the flat bf16 buffer ``g``; both sides start at t = t0."""
    gpu = H.GpuSide(w, "cuda", state)
    ref = H.OracleRun.from_state(gpu.st)
    gpu.t = ref.t = t0
    hp_g, hp_o = H.hp_pair(w)
    rep, log = H.Report(), []
    for k in range(1, steps + 1):
        grad_fn(k, gpu.g)
        skipped = gpu.step(hp_g)
        oskipped, onorm, obad = ref.step(H.to_u16(gpu.g), hp_o)
        flag = bool(gpu.flag.item())
        log.append((k, skipped, oskipped, flag, obad, float(gpu.norm.item()), onorm))
        if skipped != oskipped or flag != obad:
            rep.failures.append(f"step {k}: skip/flag gpu=({skipped},{flag}) oracle=({oskipped},{obad})")
        if w.max_grad_norm > 0 and not skipped and abs(float(gpu.norm.item()) - onorm) > 1e-13 * onorm:
            rep.failures.append(f"step {k}: norm gpu {float(gpu.norm.item())!r} oracle {onorm!r}")
    H.compare_state(gpu, ref, rep)
    gpu.plan.close()
    return rep, log


def _normal_grads(w, st):
    def fill(k, g):
        g.copy_(W.make_grad(w, k, g.device, st.offsets, g.numel()))
    return fill


HPARAM_CASES = {
    "betas_zero": dict(beta1=0.0, beta2=0.0),
    "lr_zero": dict(lr=0.0),
    "no_weight_decay": dict(weight_decay=0.0),
    "variance_decay_next_to_one": dict(beta2=0.9999999),
    "eps_one": dict(eps=1.0),
    "eps_tiny": dict(eps=1e-30),
    "clip_to_almost_nothing": dict(max_grad_norm=1e-30),
}


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_ANYPREC | 7])
@pytest.mark.parametrize("case", sorted(HPARAM_CASES))
def test_degenerate_hyperparameters(mode, case):
    w = _small("hp", mode=mode, steps=4, **HPARAM_CASES[case])
    st = W.make_state(w, "cuda")
    rep, log = _run_custom(w, _normal_grads(w, st), 4, state=st)
    _assert(rep, log)
    assert rep.exact == rep.n


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.0), (W.MODE_MIXED, 1.0),
                                       (W.MODE_REMAINDER, 0.0), (W.MODE_ANYPREC | 5, 1.0)])
def test_step_counter_near_a_billion(mode, clip):
    """Bias corrections at t ~ 1e9 are 1 to within fp32 (beta^t underflows);
    both sides evaluate beta^t by the same binary exponentiation."""
    w = _small("late", mode=mode, steps=3, max_grad_norm=clip)
    st = W.make_state(w, "cuda")
    rep, log = _run_custom(w, _normal_grads(w, st), 3, t0=999_999_998, state=st)
    _assert(rep, log)
    assert rep.exact == rep.n


def _bf16(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


GRAD_CASES = {
    # every gradient zero: the norm is 0 and the clip coefficient 1
    "all_zero": lambda n, gen: torch.zeros(n),
    # signed zeros only
    "negative_zero": lambda n, gen: torch.full((n,), -0.0),
    # bf16 subnormals: squares underflow to 0 in fp32, the momentum does not
    "subnormal": lambda n, gen: torch.randint(1, 0x80, (n,), generator=gen).float()
    * _bf16(0x0001) * torch.where(torch.rand(n, generator=gen) < 0.5, -1.0, 1.0),
    # near the bf16 maximum: g^2 overflows fp32 (v = inf where unclipped);
    # the largest draws round to +-inf in bf16 (inf / inf = NaN downstream)
    "overflowing_squares": lambda n, gen: torch.randn(n, generator=gen) * 1e38,
    # mostly ordinary values with a few huge ones
    "few_huge": lambda n, gen: torch.where(torch.rand(n, generator=gen) < 1e-3,
                                           torch.full((n,), 3.0e38), torch.randn(n, generator=gen) * 1e-2),
}


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_BF16_PLAIN,
                                  W.MODE_ANYPREC | 7])
@pytest.mark.parametrize("clip", [0.0, 1.0])
@pytest.mark.parametrize("case", sorted(GRAD_CASES))
def test_degenerate_gradients(mode, clip, case):
    w = _small("g", mode=mode, steps=3, max_grad_norm=clip)
    st = W.make_state(w, "cuda")
    gen = torch.Generator().manual_seed(7)

    def fill(k, g):
        g.copy_(GRAD_CASES[case](g.numel(), gen).to(torch.bfloat16).to(g.device))

    rep, log = _run_custom(w, fill, 3, state=st)
    _assert(rep, log)
    assert rep.exact == rep.n


def test_many_tiny_tensors():
    """40,000 tensors of 1 to 64 elements (every one shorter than a vector
    run or just one): the table, the partition and the element paths at
    scale; every element checked, with clipping."""
    rng = np.random.default_rng(11)
    sizes = [int(x) for x in rng.integers(1, 65, 40_000)]
    w = _small("tiny", mode=W.MODE_MIXED, sizes=sizes, max_grad_norm=0.5, steps=3)
    rep, log = H.run_parity(w, align_elems=1, skew=1)
    _assert(rep, log)
    assert rep.exact == rep.n


def test_tensor_longer_than_2_to_the_31():
    """One bf16 Kahan tensor of 2^31 + 1003 elements (21.5 GB of state):
    offsets, chunk lengths and per-thread indices beyond int32, sampled at
    the first and last elements, at random and around every chunk boundary,
    with the oracle's own norm over the whole gradient and clipping on."""
    n = (1 << 31) + 1003
    w = W.Workload("huge", W.MODE_BF16_KAHAN, (W.TensorSpec("t", n),), 2, lr=2e-4, beta1=0.9,
                   beta2=0.95, eps=1e-8, weight_decay=0.1, max_grad_norm=1.0, heavy_tail=True)
    rep, log = H.run_sampled(w, per_tensor=1 << 16)
    _assert(rep, log)
    assert rep.exact == rep.n


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_ANYPREC | 7])
def test_two_hundred_clipped_steps_stay_bit_identical(mode):
    """A long run with clipping on: 200 steps of a ragged 1.2M-element list,
    an inf injected at step 77 (skipped on both sides), fresh gradients every
    step.  The clip coefficient is an fp32 rounding of a norm both sides sum
    exactly, so no step may flip a bit, and nothing may drift."""
    w = _small("long_run", mode=mode, steps=200, max_grad_norm=0.5, inf_at=(77, 8, 4321))
    rep, log = H.run_parity(w)
    _assert(rep, log)
    assert rep.exact == rep.n
    assert [k for (k, s, *_r) in log if s] == [77]
