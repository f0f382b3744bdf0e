"""AnyPrecisionAdamW (the torch.optim front end) against the oracle: every
step of its device-resident path bit-identical to the oracle's list step on
the same bytes, for each buffer-type option, with clipping and a skipped
step, with an LR scheduler, through real backward passes, and across a
checkpoint."""
import io

import numpy as np
import pytest
import torch

import oracle as O
import parity_harness as H
from adamw_optimizer_step_sm_gb300 import optim as OPT

pytestmark = pytest.mark.gpu

SHAPES = [(256, 96), (96,), (7,), (1000, 33), (1,), (4097,), (64, 64, 3)]
OPTIONS = {
    "recipe_bf16_kahan": dict(),
    "fp32_state": dict(momentum_dtype=torch.float32, variance_dtype=torch.float32,
                       compensation_buffer_dtype=torch.float32),
    "fp32_momentum_no_kahan": dict(momentum_dtype=torch.float32, use_kahan_summation=False),
    "fp32_variance": dict(variance_dtype=torch.float32),
}


def _params(seed=3):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    return [(torch.randn(s, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            .requires_grad_() for s in SHAPES]


def _grad(k, seed=5, inf_at=None):
    gen = torch.Generator(device="cuda").manual_seed(seed * 1000 + k)
    gs = [(torch.randn(s, generator=gen, device="cuda") * 1e-2).to(torch.bfloat16) for s in SHAPES]
    if inf_at == k:
        gs[3].view(-1)[77] = float("inf")
    return gs


class _OracleSide:
    """The same parameters and state as host arrays, stepped by the oracle."""

    def __init__(self, params, mode):
        self.o = O.load()
        self.mode = mode
        dm, dv, dc = O.anyprec_dtypes(mode - O.ANYPREC)
        self.p = [H.to_u16(p.detach()).reshape(-1).copy() for p in params]
        self.m = [np.zeros(p.numel(), dm) for p in params]
        self.v = [np.zeros(p.numel(), dv) for p in params]
        self.c = [None if dc is None else np.zeros(p.numel(), dc) for p in params]
        self.t = 0

    def step(self, grads, hp):
        gs = [H.to_u16(g).reshape(-1).copy() for g in grads]
        tens = [(p, g, m, v, c) for p, g, m, v, c in zip(self.p, gs, self.m, self.v, self.c)]
        skipped, norm = self.o.list_step(tens, self.mode, hp, self.t + 1)
        if not skipped:
            self.t += 1
        return skipped, norm

    def check(self, opt, params):
        for k, p in enumerate(params):
            st = opt.state[p]
            assert np.array_equal(H.to_u16(p.detach()).reshape(-1), self.p[k]), f"param {k}"
            for name, ref in (("exp_avg", self.m[k]), ("exp_avg_sq", self.v[k]),
                              ("compensation", self.c[k])):
                if ref is None:
                    assert name not in st
                    continue
                got = H.to_np(st[name]).reshape(-1)
                assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), f"{name} {k}"


def _hp(group):
    return O.hparams(lr=group["lr"], beta1=group["betas"][0], beta2=group["betas"][1],
                     eps=group["eps"], weight_decay=group["weight_decay"],
                     max_grad_norm=group["max_grad_norm"])


@pytest.mark.parametrize("option", sorted(OPTIONS))
@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_optimizer_steps_match_the_oracle(option, clip):
    params = _params()
    opt = OPT.AnyPrecisionAdamW(params, max_grad_norm=clip, **OPTIONS[option])
    ref = _OracleSide(params, opt.mode)
    for k in range(1, 6):
        opt.zero_grad()
        gs = _grad(k, inf_at=3 if clip else None)
        for p, g in zip(params, gs):
            p.grad.copy_(g)
        opt.step()
        skipped, norm = ref.step(gs, _hp(opt.param_groups[0]))
        torch.cuda.synchronize()
        assert int(opt.last_nonfinite[0].item()) == int(skipped)
        assert skipped == (clip > 0 and k == 3)
        if clip:
            assert abs(opt.last_grad_norm[0].item() - norm) <= 1e-13 * norm or skipped
        assert int(opt.state[params[0]]["step"].item()) == ref.t
    ref.check(opt, params)


def test_lr_scheduler_and_two_groups():
    """A LambdaLR changes lr every step (uploaded to the device between
    steps); two groups with different weight decay step independently."""
    params = _params()
    opt = OPT.AnyPrecisionAdamW([{"params": params[:3]},
                                 {"params": params[3:], "weight_decay": 0.0}])
    sched = torch.optim.lr_scheduler.LambdaLR(opt, lambda s: 1.0 / (1 + s))
    refs = [_OracleSide(params[:3], opt.mode), _OracleSide(params[3:], opt.mode)]
    for k in range(1, 5):
        gs = _grad(k)
        for p, g in zip(params, gs):
            p.grad.copy_(g)
        opt.step()
        refs[0].step(gs[:3], _hp(opt.param_groups[0]))
        refs[1].step(gs[3:], _hp(opt.param_groups[1]))
        sched.step()
    torch.cuda.synchronize()
    refs[0].check(opt, params[:3])
    refs[1].check(opt, params[3:])


def test_backward_accumulates_into_the_optimizer_buffer():
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(64, 128), torch.nn.GELU(),
                                torch.nn.Linear(128, 8)).cuda().to(torch.bfloat16)
    params = list(model.parameters())
    opt = OPT.AnyPrecisionAdamW(params, momentum_dtype=torch.float32)
    ptrs = [p.grad.data_ptr() for p in params]
    ref = _OracleSide(params, opt.mode)
    for k in range(3):
        x = torch.randn(32, 64, device="cuda", dtype=torch.bfloat16)
        opt.zero_grad()
        model(x).float().pow(2).mean().backward()
        model(x * 0.5).float().pow(2).mean().backward()   # accumulates
        assert [p.grad.data_ptr() for p in params] == ptrs, "gradients moved out of the buffer"
        gs = [p.grad.detach().clone() for p in params]
        opt.step()
        ref.step(gs, _hp(opt.param_groups[0]))
    torch.cuda.synchronize()
    ref.check(opt, params)


def test_checkpoint_round_trip_continues_identically():
    pa, pb = _params(), _params()
    opt_a = OPT.AnyPrecisionAdamW(pa, max_grad_norm=1.0, momentum_dtype=torch.float32)
    opt_b = OPT.AnyPrecisionAdamW(pb, max_grad_norm=1.0, momentum_dtype=torch.float32)
    for k in range(1, 3):
        for p, g in zip(pa, _grad(k)):
            p.grad.copy_(g)
        opt_a.step()
    buf = io.BytesIO()
    torch.save({"params": [p.detach().clone() for p in pa], "opt": opt_a.state_dict()}, buf)
    buf.seek(0)
    ck = torch.load(buf, weights_only=False)
    with torch.no_grad():
        for p, q in zip(pb, ck["params"]):
            p.copy_(q)
    opt_b.load_state_dict(ck["opt"])
    for k in range(3, 6):
        for p, q, g in zip(pa, pb, _grad(k)):
            p.grad.copy_(g)
            q.grad.copy_(g)
        opt_a.step()
        opt_b.step()
    torch.cuda.synchronize()
    for p, q in zip(pa, pb):
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))
        for name in ("exp_avg", "exp_avg_sq", "compensation"):
            assert torch.equal(opt_a.state[p][name].view(torch.uint8),
                               opt_b.state[q][name].view(torch.uint8))
    assert opt_a.state[pa[0]]["step"].item() == opt_b.state[pb[0]]["step"].item() == 5


@pytest.mark.parametrize("clip", [0.0, 1.0])
def test_step_replays_from_a_cuda_graph(clip):
    """The step needs no host synchronisation, so it can be captured once and
    replayed: replays of the captured step (new gradients copied into the
    optimizer's gradient buffer before each) give the same bytes as eager
    steps of a twin optimizer, including the step counter."""
    pa, pb = _params(), _params()
    kw = dict(max_grad_norm=clip, variance_dtype=torch.float32)
    opt_a, opt_b = OPT.AnyPrecisionAdamW(pa, **kw), OPT.AnyPrecisionAdamW(pb, **kw)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in (1, 2):                       # warm-up steps, eager on both
            for p, q, g in zip(pa, pb, _grad(k)):
                p.grad.copy_(g)
                q.grad.copy_(g)
            opt_a.step()
            opt_b.step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        opt_a.step()
    for k in (3, 4, 5):
        for p, q, g in zip(pa, pb, _grad(k)):
            p.grad.copy_(g)
            q.grad.copy_(g)
        graph.replay()
        opt_b.step()
    torch.cuda.synchronize()
    for p, q in zip(pa, pb):
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))
        for name in ("exp_avg", "exp_avg_sq", "compensation"):
            assert torch.equal(opt_a.state[p][name].view(torch.uint8),
                               opt_b.state[q][name].view(torch.uint8))
    assert opt_a.state[pa[0]]["step"].item() == opt_b.state[pb[0]]["step"].item() == 5


def test_tensor_lr_works_and_out_of_range_values_are_refused():
    """A scheduler may keep lr as a 0-d tensor: the step takes its value.
    An out-of-range value set between steps is refused on the host (on the
    device it could only make the step skip)."""
    from adamw_optimizer_step_sm_gb300 import adamw_sm as A
    params = _params()
    opt = OPT.AnyPrecisionAdamW(params)
    ref = _OracleSide(params, opt.mode)
    opt.param_groups[0]["lr"] = torch.tensor(1e-4)
    gs = _grad(1)
    for p, g in zip(params, gs):
        p.grad.copy_(g)
    opt.step()
    ref.step(gs, O.hparams(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1))
    torch.cuda.synchronize()
    ref.check(opt, params)
    opt.param_groups[0]["lr"] = -1.0
    with pytest.raises(A.AdamWError):
        opt.step()
    opt.param_groups[0]["lr"] = 1e-4
    opt.param_groups[0]["betas"] = (0.9, 1.0)
    with pytest.raises(A.AdamWError):
        opt.step()


class _MasterOracle:
    """The same parameters as host arrays for the fp32-master (mode 1) or
    bf16 + remainder (mode 2) oracle steps."""

    def __init__(self, params, remainder: bool):
        self.o = O.load()
        self.mode = 2 if remainder else 1
        p16 = [H.to_u16(p.detach()).reshape(-1).copy() for p in params]
        n = [p.numel() for p in params]
        if remainder:
            self.tens = [[q, None, np.zeros(k, np.float32), np.zeros(k, np.float32),
                          np.zeros(k, np.int16)] for q, k in zip(p16, n)]
        else:
            self.tens = [[(q.astype(np.uint32) << 16).view(np.float32).copy(), None,
                          np.zeros(k, np.float32), np.zeros(k, np.float32), q.copy()]
                         for q, k in zip(p16, n)]
        self.t = 0

    def step(self, grads, hp):
        for e, g in zip(self.tens, grads):
            e[1] = H.to_u16(g).reshape(-1).copy()
        skipped, norm = self.o.list_step([tuple(e) for e in self.tens], self.mode, hp, self.t + 1)
        if not skipped:
            self.t += 1
        return skipped, norm

    def check(self, opt, params):
        for k, p in enumerate(params):
            st, e = opt.state[p], self.tens[k]
            model = e[0] if self.mode == 2 else e[4]
            assert np.array_equal(H.to_u16(p.detach()).reshape(-1), model), f"param {k}"
            assert np.array_equal(H.to_np(st["exp_avg"]).reshape(-1).view(np.uint8), e[2].view(np.uint8))
            assert np.array_equal(H.to_np(st["exp_avg_sq"]).reshape(-1).view(np.uint8), e[3].view(np.uint8))
            if self.mode == 1:
                assert np.array_equal(H.to_np(st["master"]).reshape(-1).view(np.uint8), e[0].view(np.uint8))
            else:
                assert np.array_equal(H.to_np(st["remainder"]).reshape(-1), e[4])


@pytest.mark.parametrize("master", ["fp32", "remainder"])
@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_master_weight_optimizer_matches_the_oracle(master, clip):
    params = _params()
    opt = OPT.MasterWeightAdamW(params, master=master, max_grad_norm=clip, lr=2e-4,
                                betas=(0.9, 0.95), weight_decay=0.1)
    ref = _MasterOracle(params, master == "remainder")
    for k in range(1, 6):
        opt.zero_grad()
        gs = _grad(k, inf_at=3 if clip else None)
        for p, g in zip(params, gs):
            p.grad.copy_(g)
        opt.step()
        skipped, norm = ref.step(gs, _hp(opt.param_groups[0]))
        torch.cuda.synchronize()
        assert int(opt.last_nonfinite[0].item()) == int(skipped)
        assert skipped == (clip > 0 and k == 3)
        assert int(opt.state[params[0]]["step"].item()) == ref.t
    ref.check(opt, params)


def test_master_weight_modes_keep_the_same_trajectory():
    """The bf16 + remainder master is the fp32 master exactly: after the same
    steps the fp32 master of one optimizer equals (bf16 parameter, remainder)
    of the other, joined."""
    pa, pb = _params(), _params()
    oa = OPT.MasterWeightAdamW(pa, master="fp32", max_grad_norm=1.0)
    ob = OPT.MasterWeightAdamW(pb, master="remainder", max_grad_norm=1.0)
    for k in range(1, 6):
        for p, q, g in zip(pa, pb, _grad(k)):
            p.grad.copy_(g)
            q.grad.copy_(g)
        oa.step()
        ob.step()
    torch.cuda.synchronize()
    o = O.load()
    for p, q in zip(pa, pb):
        joined = o.join_master(H.to_u16(q.detach()).reshape(-1), H.to_np(ob.state[q]["remainder"]).reshape(-1))
        master = H.to_np(oa.state[p]["master"]).reshape(-1)
        assert np.array_equal(joined.view(np.uint32), master.view(np.uint32))
        for name in ("exp_avg", "exp_avg_sq"):
            assert torch.equal(oa.state[p][name], ob.state[q][name])


@pytest.mark.parametrize("master", ["fp32", "remainder"])
def test_master_weight_backward_and_checkpoint(master):
    """Real backward passes accumulate into the optimizer's gradient buffer,
    and a checkpoint taken after two steps continues bit for bit in a fresh
    optimizer over a copy of the model."""
    torch.manual_seed(1)
    make = lambda: torch.nn.Sequential(torch.nn.Linear(64, 96), torch.nn.GELU(),
                                       torch.nn.Linear(96, 8)).cuda().to(torch.bfloat16)
    ma = make()
    mb = make()
    mb.load_state_dict(ma.state_dict())
    oa = OPT.MasterWeightAdamW(ma.parameters(), master=master, max_grad_norm=1.0)
    xs = [torch.randn(16, 64, device="cuda", dtype=torch.bfloat16) for _ in range(5)]
    ptrs = [p.grad.data_ptr() for p in ma.parameters()]
    for x in xs[:2]:
        oa.zero_grad()
        ma(x).float().pow(2).mean().backward()
        assert [p.grad.data_ptr() for p in ma.parameters()] == ptrs
        oa.step()
    buf = io.BytesIO()
    torch.save({"model": ma.state_dict(), "opt": oa.state_dict()}, buf)
    buf.seek(0)
    ck = torch.load(buf, weights_only=False)
    mb.load_state_dict(ck["model"])
    ob = OPT.MasterWeightAdamW(mb.parameters(), master=master, max_grad_norm=1.0)
    ob.load_state_dict(ck["opt"])
    for x in xs[2:]:
        for m, o in ((ma, oa), (mb, ob)):
            o.zero_grad()
            m(x).float().pow(2).mean().backward()
            o.step()
    torch.cuda.synchronize()
    for p, q in zip(ma.parameters(), mb.parameters()):
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))
        for name in oa.state[p]:
            if name != "step":
                assert torch.equal(oa.state[p][name].view(torch.uint8), ob.state[q][name].view(torch.uint8))
    assert oa.state[next(ma.parameters())]["step"].item() == ob.state[next(mb.parameters())]["step"].item() == 5


@pytest.mark.parametrize("master", ["fp32", "remainder"])
def test_master_follows_weights_loaded_after_the_optimizer(master):
    """Build the optimizer, then load other weights into the model (as a
    model load_state_dict does, in place): the next step starts from the
    loaded weights, exactly as the oracle started from them."""
    params = _params(seed=3)
    opt = OPT.MasterWeightAdamW(params, master=master, lr=2e-4, betas=(0.9, 0.95),
                                weight_decay=0.1, max_grad_norm=1.0)
    loaded = _params(seed=11)
    with torch.no_grad():
        for p, q in zip(params, loaded):
            p.copy_(q)
    ref = _MasterOracle(loaded, master == "remainder")
    for k in range(1, 4):
        gs = _grad(k)
        for p, g in zip(params, gs):
            p.grad.copy_(g)
        opt.step()
        ref.step(gs, _hp(opt.param_groups[0]))
    torch.cuda.synchronize()
    ref.check(opt, params)


@pytest.mark.parametrize("master", ["fp32", "remainder"])
def test_state_without_a_master_rederives_it_from_the_model(master):
    """A checkpoint whose state has no master (saved by an optimizer without
    one) loads its moments and step count; the master is taken from the
    model's parameters as they are then."""
    params = _params(seed=3)
    opt = OPT.MasterWeightAdamW(params, master=master, lr=2e-4, betas=(0.9, 0.95),
                                weight_decay=0.1)
    for k in range(1, 3):
        for p, g in zip(params, _grad(k)):
            p.grad.copy_(g)
        opt.step()
    sd = opt.state_dict()
    key = "master" if master == "fp32" else "remainder"
    sd["state"] = {i: {n: (v.clone() if torch.is_tensor(v) else v) for n, v in st.items() if n != key}
                   for i, st in sd["state"].items()}
    other = _params(seed=17)
    with torch.no_grad():
        for p, q in zip(params, other):
            p.copy_(q)
    opt.load_state_dict(sd)
    ref = _MasterOracle(other, master == "remainder")
    for kk, p in enumerate(params):
        ref.tens[kk][2] = H.to_np(opt.state[p]["exp_avg"]).reshape(-1).copy()
        ref.tens[kk][3] = H.to_np(opt.state[p]["exp_avg_sq"]).reshape(-1).copy()
    ref.t = int(opt.state[params[0]]["step"].item())
    assert ref.t == 2
    for k in range(3, 5):
        gs = _grad(k)
        for p, g in zip(params, gs):
            p.grad.copy_(g)
        opt.step()
        ref.step(gs, _hp(opt.param_groups[0]))
    torch.cuda.synchronize()
    ref.check(opt, params)


def test_fp32_master_survives_loading_the_model_after_the_optimizer():
    """Restoring a checkpoint in the other order (optimizer state first, then
    the same checkpoint's model weights) keeps the loaded fp32 master: the
    model's bf16 values are its rounding, so nothing is re-derived and the
    run continues bit for bit."""
    torch.manual_seed(2)
    make = lambda: torch.nn.Linear(96, 80).cuda().to(torch.bfloat16)
    ma = make()
    oa = OPT.MasterWeightAdamW(ma.parameters(), master="fp32")
    xs = [torch.randn(16, 96, device="cuda", dtype=torch.bfloat16) for _ in range(4)]
    for x in xs[:2]:
        oa.zero_grad()
        ma(x).float().pow(2).mean().backward()
        oa.step()
    ck = {"model": {k: v.clone() for k, v in ma.state_dict().items()}, "opt": oa.state_dict()}
    mb = make()
    ob = OPT.MasterWeightAdamW(mb.parameters(), master="fp32")
    ob.load_state_dict(ck["opt"])
    mb.load_state_dict(ck["model"])
    for x in xs[2:]:
        for m, o in ((ma, oa), (mb, ob)):
            o.zero_grad()
            m(x).float().pow(2).mean().backward()
            o.step()
    torch.cuda.synchronize()
    for p, q in zip(ma.parameters(), mb.parameters()):
        assert torch.equal(oa.state[p]["master"], ob.state[q]["master"])
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))
