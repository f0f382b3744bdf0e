"""GPU parity of the any-precision storage modes (MODE_ANYPREC | flags:
momentum, variance and compensation each bf16 or fp32, Kahan summation on or
off) against the oracle's any-precision step, through the C ABI.  Same
tolerances as the other parity tests (<= 1 bf16 ulp, <= 1e-6 relative on
fp32 state, identical flags); bit-identical results are expected and
checked."""
import pytest
import torch

import parity_harness as H
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import workloads as W
from test_gpu_parity import _assert, _same_state, _small, _twin

pytestmark = pytest.mark.gpu

MODES = list(W.ANYPREC_MODES)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("clip", [0.0, 0.5])
@pytest.mark.parametrize("layout", [(8, 0), (1, 3)])
def test_anyprec_ragged_lists(mode, clip, layout):
    """Every combination over the ragged list: tails, empty and one-element
    tensors, bases that are not 16-byte aligned; clipped steps run fused."""
    w = _small("anyprec", mode=mode, max_grad_norm=clip)
    rep, log = H.run_parity(w, align_elems=layout[0], skew=layout[1])
    _assert(rep, log)
    assert rep.exact == rep.n


@pytest.mark.parametrize("name", ["opt1.3b_anyprec_fp32_state", "opt1.3b_anyprec_m32"])
def test_anyprec_sampled_full_size(name):
    rep, log = H.run_sampled(W.WORKLOADS[name], per_tensor=512)
    _assert(rep, log)
    assert rep.exact == rep.n


@pytest.mark.parametrize("mode,clip", [(W.MODE_ANYPREC | 7, 0.5), (W.MODE_ANYPREC | 9, 0.0),
                                       (W.MODE_ANYPREC | 4, 1.0)])
def test_anyprec_device_step_matches_host_step(mode, clip):
    w = _small("anydev", mode=mode, max_grad_norm=clip, steps=5,
               inf_at=(3, 8, 777) if clip else None)
    a, b_state, b_plan = _twin(w)
    hp, _ = H.hp_pair(w)
    d_hp = A.device_hparams(hp)
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_b = torch.zeros(1, dtype=torch.float64, device="cuda")
    f_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in range(1, 6):
        a.set_grad(k)
        skipped = a.step(hp)
        b_plan.step_device(d_hp, d_step, A.STEP_CLIP if clip else 0,
                           grad_norm=n_b if clip else None, nonfinite=f_b)
        torch.cuda.synchronize()
        assert int(f_b.item()) == int(a.flag.item())
        assert int(d_step.item()) == a.t
        assert skipped == (clip > 0 and k == 3)
    _same_state(a.st, b_state)
    a.plan.close()
    b_plan.close()


@pytest.mark.parametrize("mode", [W.MODE_ANYPREC | 7, W.MODE_ANYPREC | 10])
def test_anyprec_fused_and_unfused_clipped_steps_agree(mode):
    w = _small("anyfuse", mode=mode, max_grad_norm=0.5, steps=4, inf_at=(3, 8, 99))
    a = H.GpuSide(w)
    b_state = W.make_state(w, "cuda")
    v = b_state.views
    b_plan = A.Plan(v(b_state.param), v(a.g), v(b_state.exp_avg), v(b_state.exp_avg_sq),
                    v(b_state.aux), mode, norm=True, fuse=False)
    assert a.plan.info.fused == 1 and b_plan.info.fused == 0
    hp, _ = H.hp_pair(w)
    nb = torch.zeros(1, dtype=torch.float64, device="cuda")
    fb = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb = 0
    for k in range(1, 5):
        a.set_grad(k)
        skipped = a.step(hp)
        b_plan.step(hp, tb + 1, grad_norm=nb, nonfinite=fb)
        torch.cuda.synchronize()
        if not fb.item():
            tb += 1
        assert skipped == bool(fb.item()) == (k == 3)
    _same_state(a.st, b_state)
    a.plan.close()
    b_plan.close()


@pytest.mark.parametrize("alias,named", [(W.MODE_ANYPREC, W.MODE_BF16_KAHAN),
                                         (W.MODE_ANYPREC | 2, W.MODE_BF16_KAHAN_V32),
                                         (W.MODE_ANYPREC | 8, W.MODE_BF16_PLAIN)])
def test_anyprec_aliases_run_the_named_modes(alias, named):
    """Modes 16, 18 and 24 are the named bf16 modes under other numbers: the
    plan reports the number it was given and writes the same bytes."""
    wa = _small("alias", mode=alias, steps=3)
    wn = _small("named", mode=named, steps=3)
    a, b = H.GpuSide(wa), H.GpuSide(wn)
    assert a.plan.info.mode == alias and b.plan.info.mode == named
    hp, _ = H.hp_pair(wa)
    for k in range(1, 4):
        a.set_grad(k)
        b.set_grad(k)
        a.step(hp)
        b.step(hp)
    torch.cuda.synchronize()
    _same_state(a.st, b.st)
    a.plan.close()
    b.plan.close()


@pytest.mark.parametrize("mode", MODES)
def test_anyprec_canaries_stay_untouched(mode):
    """Bytes outside every tensor (skew, gaps, a 4096-element tail) and the
    gradient are never written, whatever each stream's element size."""
    w = _small("anycanary", mode=mode, max_grad_norm=0.0, steps=3)
    st = W.make_state(w, "cuda", align_elems=8, skew=5, tail_pad=4096)
    gpu = H.GpuSide(w, "cuda", st)
    covered = torch.zeros(st.param.numel(), dtype=torch.bool, device="cuda")
    for o, n in zip(st.offsets, w.numels):
        covered[o:o + n] = True
    gaps = ~covered
    bufs = [b for b in (st.param, st.exp_avg, st.exp_avg_sq, st.aux) if b is not None]
    for b in bufs:
        b.view(torch.uint8).view(-1, b.element_size())[gaps] = 0xA5
    hp_plain, _ = H.hp_pair(w)
    hp_clip = A.hparams(**{**w.hparams(), "max_grad_norm": 0.5})
    for k in range(1, 4):
        gpu.set_grad(k)
        g_before = gpu.g.clone()
        gpu.plan.step(hp_clip if k == 2 else hp_plain, k, grad_norm=gpu.norm if k == 2 else None)
        torch.cuda.synchronize()
        assert torch.equal(gpu.g.view(torch.int16), g_before.view(torch.int16)), "grad written"
    for b in bufs:
        assert bool((b.view(torch.uint8).view(-1, b.element_size())[gaps] == 0xA5).all()), \
            f"a {b.dtype} canary changed"
    gpu.plan.close()


@pytest.mark.parametrize("mode", [W.MODE_ANYPREC | 7, W.MODE_ANYPREC | 9])
def test_anyprec_step_table_matches_a_plan(mode):
    """adamw_step_table with an any-precision mode (aux NULL without Kahan
    summation) updates exactly like an explicit plan, one cached plan."""
    w = _small("anytable", mode=mode, max_grad_norm=0.5, steps=3)
    a = H.GpuSide(w)
    b = W.make_state(w, "cuda")
    g = torch.zeros_like(a.g)
    v = b.views
    aux = v(b.aux) if b.aux is not None else [None] * len(w.numels)
    entries = [A.adamw_tensor_t(*(t.data_ptr() if t is not None else None for t in ts),
                                ts[0].numel())
               for ts in zip(v(b.param), v(g), v(b.exp_avg), v(b.exp_avg_sq), aux)]
    raw = bytes((A.adamw_tensor_t * len(entries))(*entries))
    d_table = torch.frombuffer(bytearray(raw), dtype=torch.uint8).cuda()
    hp, _ = H.hp_pair(w)
    A.adamw_step_table_cache_clear()
    norm_a = torch.zeros(1, dtype=torch.float64, device="cuda")
    norm_b = torch.zeros(1, dtype=torch.float64, device="cuda")
    flag_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for k in (1, 2, 3):
        a.set_grad(k)
        g.copy_(a.g)
        a.plan.step(hp, k, grad_norm=norm_a)
        A.adamw_step_table(d_table.data_ptr(), len(entries), w.mode, hp, k, norm_b.data_ptr(),
                           flag_b.data_ptr(), stream)
    torch.cuda.synchronize()
    assert A.adamw_step_table_cache_clear() == 1
    _same_state(a.st, b)
    assert norm_a.item() == norm_b.item()
    a.plan.close()
