"""GPU parity: the CUDA library, called through its C ABI, against the CPU
oracle on identical seeded bytes.  Tolerances are those stated in
``parity_harness``: <= 1 bf16 ulp on bf16 state, <= 1e-6 relative on fp32
state, identical non-finite flags (bit-identical results are expected)."""
import numpy as np
import pytest
import torch

import oracle as O
import parity_harness as H
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _assert(rep: H.Report, log=None):
    assert rep.ok(), "\n".join(rep.failures[:20]) + f"\nlog={log}"


def _small(name, **kw):
    """A small list with the shape mix of the workloads on the pages plus ragged
    sizes that span several CTAs and leave tails."""
    sizes = kw.pop("sizes", [1, 7, 8, 9, 4095, 65537, 0, 3, 1000003, 255, 256, 257, 3 * 768, 50272])
    mode = kw.pop("mode", W.MODE_BF16_KAHAN)
    tensors = tuple(W.TensorSpec(f"t{i}", n) for i, n in enumerate(sizes))
    base = dict(steps=6, lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, heavy_tail=True)
    base.update(kw)
    return W.Workload(name, mode, tensors, **base)


# ---------------------------------------------------- the pages' workloads --

def test_flat1m_bf16_kahan_bit_exact():
    rep, log = H.run_parity(W.WORKLOADS["flat1m_bf16_kahan"])
    _assert(rep, log)
    assert rep.exact == rep.n, f"{rep.n - rep.exact} of {rep.n} values not bit-identical"


def test_bert_shard_mixed():
    rep, log = H.run_parity(W.WORKLOADS["bert55m_shard_mixed"])
    _assert(rep, log)
    assert rep.exact == rep.n


def test_opt125m_bf16_kahan_full_list():
    rep, log = H.run_parity(W.WORKLOADS["opt125m_bf16_kahan"])
    _assert(rep, log)
    assert rep.exact == rep.n


def test_bert_shard_remainder():
    rep, log = H.run_parity(W.WORKLOADS["bert55m_shard_remainder"])
    _assert(rep, log)
    assert rep.exact == rep.n


def test_opt1_3b_remainder_clip_inf_skip_sampled_full_size():
    w = W.WORKLOADS["opt1.3b_remainder_clip"]
    rep, log = H.run_sampled(w, per_tensor=512)
    _assert(rep, log)
    assert [k for (k, s, *_r) in log if s] == [w.inf_at[0]], log
    assert rep.exact == rep.n


def test_remainder_mode_holds_the_mixed_mode_master():
    """On the GPU too, the remainder mode's (bf16 param, remainder) pair is
    the mixed mode's fp32 master bit for bit, step after step."""
    import oracle as O
    o = O.load()
    sizes = [70001, 4099, 1 << 20]
    wr = _small("rem", mode=W.MODE_REMAINDER, sizes=sizes, max_grad_norm=0.5, steps=5)
    wm = _small("mix", mode=W.MODE_MIXED, sizes=sizes, max_grad_norm=0.5, steps=5)
    r = H.GpuSide(wr)
    m = H.GpuSide(wm)
    m.st.param.copy_(r.st.param.float())           # same bf16-exact start
    hp, _ = H.hp_pair(wr)
    for k in range(1, 6):
        r.set_grad(k)
        m.g.copy_(r.g)
        r.step(hp)
        m.step(hp)
    joined = o.join_master(H.to_u16(r.st.param), H.to_np(r.st.aux))
    assert np.array_equal(joined.view(np.uint32), H.to_f32(m.st.param).view(np.uint32))
    assert torch.equal(r.st.exp_avg, m.st.exp_avg) and torch.equal(r.st.exp_avg_sq, m.st.exp_avg_sq)
    r.plan.close()
    m.plan.close()


@pytest.mark.parametrize("name", ["opt1.3b_bf16_plain", "opt1.3b_bf16_kahan_v32"])
def test_other_anyprecision_options_sampled_full_size(name):
    rep, log = H.run_sampled(W.WORKLOADS[name], per_tensor=512)
    _assert(rep, log)
    assert rep.exact == rep.n


def test_fused_clipped_shard_matches_oracle():
    """A 13.85M-element shard with clipping: each clipped step is one fused
    launch (norm, grid barrier, update); bit-identical to the oracle over 20
    steps including the skipped step 7."""
    w = W.WORKLOADS["bert55m_shard_mixed_clip"]
    gpu = H.GpuSide(w)
    assert gpu.plan.info.fused == 1
    gpu.plan.close()
    rep, log = H.run_parity(w)
    _assert(rep, log)
    assert [k for (k, s, *_r) in log if s] == [7]
    assert rep.exact == rep.n


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER])
def test_fused_and_unfused_clipped_steps_agree(mode):
    """The fused launch and the three-launch path give the same bytes, and
    norms equal to fp64 rounding: the fused launch's norm phase runs on the
    update's grid, the three-launch norm pass on a grid of its own, so the
    sums are grouped differently (each group is summed without error; the
    groups' fp64 total rounds)."""
    w = _small("fuse", mode=mode, max_grad_norm=0.5, steps=4, inf_at=(3, 8, 99))
    a = H.GpuSide(w)
    b_state = W.make_state(w, "cuda")
    v = b_state.views
    b_plan = A.Plan(v(b_state.param), v(a.g), v(b_state.exp_avg), v(b_state.exp_avg_sq),
                    v(b_state.aux), mode, norm=True, fuse=False)
    assert a.plan.info.fused == 1 and b_plan.info.fused == 0
    assert a.plan.info.norm_grid == a.plan.info.grid
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
        assert abs(a.norm.item() - nb.item()) <= 1e-13 * nb.item() or (k == 3)
    _same_state(a.st, b_state)
    assert A.adamw_plan_device_status(a.plan.handle) == 0
    a.plan.close()
    b_plan.close()


def test_fused_barrier_wait_runs_out_and_reports():
    """Failure detection without a GPU fault: with the barrier counter shifted
    by one, the last CTA to arrive waits for an arrival that never comes; its
    bounded wait (about half a second) runs out, it sets the device status and
    returns.  The host reads the status, which also realigns the counter, and
    the next steps run normally on the same context."""
    import time
    w = _small("stall", mode=W.MODE_MIXED, max_grad_norm=1.0, steps=3)
    gpu = H.GpuSide(w)
    assert gpu.plan.info.fused == 1
    hp, _ = H.hp_pair(w)
    gpu.set_grad(1)
    gpu.step(hp)
    assert A.adamw_plan_device_status(gpu.plan.handle) == 0
    A.adamw_plan_test_skew_barrier(gpu.plan.handle, 1)
    gpu.set_grad(2)
    t0 = time.perf_counter()
    gpu.plan.step(hp, 2, grad_norm=gpu.norm, nonfinite=gpu.flag)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert A.adamw_plan_device_status(gpu.plan.handle) == 1
    assert 0.05 < waited < 30
    # the context and the plan work again
    for k in (3, 4):
        gpu.set_grad(k)
        gpu.plan.step(hp, k, grad_norm=gpu.norm, nonfinite=gpu.flag)
    torch.cuda.synchronize()
    assert A.adamw_plan_device_status(gpu.plan.handle) == 0
    assert np.isfinite(gpu.norm.item())
    gpu.plan.close()


def test_opt1_3b_bf16_kahan_sampled_full_size():
    rep, log = H.run_sampled(W.WORKLOADS["opt1.3b_bf16_kahan"], per_tensor=1024)
    _assert(rep, log)
    assert rep.exact == rep.n


def test_opt1_3b_mixed_clip_inf_skip_sampled_full_size():
    w = W.WORKLOADS["opt1.3b_mixed_clip"]
    rep, log = H.run_sampled(w, per_tensor=1024)
    _assert(rep, log)
    skipped = [k for (k, s, os_, *_rest) in log if s]
    assert skipped == [w.inf_at[0]], log
    # both norms are the exact sum of squares up to fp64 rounding noise, so
    # the fp32 clip coefficient agrees and so does every stored bit
    for (k, s, _, flag, bad, gn, on) in log:
        if not s:
            assert abs(gn - on) <= 1e-13 * on
    assert rep.exact == rep.n


# ------------------------------------------------------------- edge cases --

@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER,
                                  W.MODE_BF16_PLAIN, W.MODE_BF16_KAHAN_V32])
@pytest.mark.parametrize("clip", [0.0, 0.5])
@pytest.mark.parametrize("layout", [(8, 0), (1, 3), (1, 1)])
def test_ragged_lists(mode, clip, layout):
    """Tails, empty tensors, one-element tensors and bases that are not 16-B
    aligned (element-path heads and whole element-path tensors)."""
    w = _small("ragged", mode=mode, max_grad_norm=clip)
    rep, log = H.run_parity(w, align_elems=layout[0], skew=layout[1])
    _assert(rep, log)
    assert rep.exact == rep.n


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.0), (W.MODE_MIXED, 0.5),
                                       (W.MODE_ANYPREC | 7, 0.0), (W.MODE_BF16_PLAIN, 0.5)])
@pytest.mark.parametrize("layout", [(8, 0), (1, 3)])
def test_interleaved_partition_over_ragged_tensors(mode, clip, layout):
    """A list long enough for the interleaved partition (at least two tiles
    per CTA) made of ragged tensors: tiles span tensor boundaries, cuts fall
    inside tensors, and with the skewed layout every tensor has an
    element-path head before its vector body.  Every element checked."""
    sizes = [3_000_001, 7, 2_500_003, 65_537, 1_999_999, 1, 4_194_304, 257, 1_048_583, 9]
    w = _small("interleaved", mode=mode, sizes=sizes, max_grad_norm=clip, steps=3)
    gpu = H.GpuSide(w)
    info = gpu.plan.info
    assert info.n_chunks >= 2 * info.grid, "list too short for the interleaved partition"
    gpu.plan.close()
    rep, log = H.run_parity(w, align_elems=layout[0], skew=layout[1])
    _assert(rep, log)
    assert rep.exact == rep.n


def _claimable(gpu: H.GpuSide) -> int:
    """Chunks of the plan's update partition that CTAs claim at run time."""
    v = gpu.st.views
    entries = [tuple(t.data_ptr() if t is not None else 0 for t in ts) + (ts[0].numel(),)
               for ts in zip(v(gpu.st.param), v(gpu.g), v(gpu.st.exp_avg), v(gpu.st.exp_avg_sq),
                             v(gpu.st.aux))]
    return sum(c.cta < 0 for c in A.adamw_plan_chunks(entries, gpu.w.mode, gpu.plan.info.grid))


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.0), (W.MODE_MIXED, 0.5),
                                       (W.MODE_REMAINDER, 0.0)])
def test_claimed_tiles_match_oracle_on_host_and_device_paths(mode, clip):
    """A list of more than 8 rounds of tiles, whose last rounds are not dealt
    to CTAs but claimed at run time (ragged tensors, so claimed tiles span
    tensor boundaries and the pieces shrink towards the end): every element
    against the oracle over three steps on the host path, and the
    device-resident step, whose claims share the word with its arrival
    count, bit-identical to the host path."""
    sizes = [30_000_001, 7, 6_500_003, 65_537, 1, 4_194_304, 1_048_583]
    w = _small("claimed", mode=mode, sizes=sizes, max_grad_norm=clip, steps=3)
    probe = H.GpuSide(w)
    assert _claimable(probe) > probe.plan.info.grid, "no claimable tiles"
    probe.plan.close()
    del probe
    rep, log = H.run_parity(w, align_elems=1, skew=3)
    _assert(rep, log)
    assert rep.exact == rep.n
    a, b_state, b_plan = _twin(w)
    hp, _ = H.hp_pair(w)
    d_hp = A.device_hparams(hp)
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_b = torch.zeros(1, dtype=torch.float64, device="cuda")
    f_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in range(1, 4):
        a.set_grad(k)
        a.step(hp)
        b_plan.step_device(d_hp, d_step, A.STEP_CLIP if clip else 0,
                           grad_norm=n_b if clip else None, nonfinite=f_b)
    torch.cuda.synchronize()
    assert int(d_step.item()) == a.t == 3 and int(f_b.item()) == 0
    _same_state(a.st, b_state)
    a.plan.close()
    b_plan.close()


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.5), (W.MODE_MIXED, 0.0),
                                       (W.MODE_ANYPREC | 7, 0.5)])
def test_claimed_tiles_over_thousands_of_small_tensors(mode, clip):
    """The claimed last rounds falling on 2500 small tensors (37 and 1000
    elements) at the end of a list of more than 8 rounds, on bases skewed so
    that every tensor has an element-path head: claimed tiles made of many
    chunks, element-path chunks and pieces shorter than a vector, every
    element against the oracle."""
    sizes = [30_000_000, 6_000_001] + [37] * 2000 + [1000] * 500 + [5]
    w = _small("claimsmall", mode=mode, sizes=sizes, max_grad_norm=clip, steps=2)
    probe = H.GpuSide(w, "cuda", W.make_state(w, "cuda", 1, 3))
    v = probe.st.views
    entries = [tuple(t.data_ptr() if t is not None else 0 for t in ts) + (ts[0].numel(),)
               for ts in zip(v(probe.st.param), v(probe.g), v(probe.st.exp_avg),
                             v(probe.st.exp_avg_sq), v(probe.st.aux))]
    chunks = A.adamw_plan_chunks(entries, mode, probe.plan.info.grid)
    claimed = {c.tensor for c in chunks if c.cta < 0}
    assert len(claimed) > 2000 and any(c.cta < 0 and not c.vec for c in chunks), \
        (len(claimed), "claimed chunks should span the small tensors, element paths included")
    probe.plan.close()
    del probe
    rep, log = H.run_parity(w, align_elems=1, skew=3)
    _assert(rep, log)
    assert rep.exact == rep.n


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER])
def test_clip_skips_step_with_inf_and_writes_nothing(mode):
    w = _small("skip", mode=mode, max_grad_norm=1.0, inf_at=(2, 8, 777), steps=4)
    rep, log = H.run_parity(w)
    _assert(rep, log)
    assert [k for (k, s, *_r) in log if s] == [2]
    # the skipped step itself wrote nothing
    gpu = H.GpuSide(w)
    hp, _ = H.hp_pair(w)
    gpu.set_grad(1)
    gpu.step(hp)
    before = [t.clone() for t in (gpu.st.param, gpu.st.exp_avg, gpu.st.exp_avg_sq, gpu.st.aux)]
    gpu.set_grad(2)
    assert gpu.step(hp) is True
    after = (gpu.st.param, gpu.st.exp_avg, gpu.st.exp_avg_sq, gpu.st.aux)
    for b, a in zip(before, after):
        assert torch.equal(b.view(torch.uint8), a.view(torch.uint8))
    gpu.plan.close()


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER])
@pytest.mark.parametrize("path", ["fused", "three_launches", "device"])
def test_clip_skips_step_with_nan_in_every_path(mode, path):
    """A NaN gradient under clipping (one element among a million, or the
    only non-zero one) sets the flag and skips the step in every path, as in
    the oracle, and the norm reads NaN; the next finite step goes on from the
    unchanged state."""
    w = _small("nanskip", mode=mode, max_grad_norm=1.0, steps=3)
    gpu = H.GpuSide(w)
    if path != "fused":
        gpu.plan.close()
        v = gpu.st.views
        gpu.plan = A.Plan(v(gpu.st.param), v(gpu.g), v(gpu.st.exp_avg), v(gpu.st.exp_avg_sq),
                          v(gpu.st.aux), mode, norm=True, fuse=False)
    assert gpu.plan.info.fused == (1 if path == "fused" else 0)
    ref = H.OracleRun.from_state(gpu.st)
    hp_g, hp_o = H.hp_pair(w)
    d_hp = A.device_hparams(hp_g)
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    for k in (1, 2, 3):
        gpu.set_grad(k)
        if k == 2:
            gpu.g[gpu.st.offsets[8] + 4242] = float("nan")
        if path == "device":
            gpu.plan.step_device(d_hp, d_step, A.STEP_CLIP, grad_norm=gpu.norm, nonfinite=gpu.flag)
            torch.cuda.synchronize()
            skipped = bool(gpu.flag.item())
        else:
            skipped = gpu.step(hp_g)
        oskipped, onorm, obad = ref.step(H.to_u16(gpu.g), hp_o)
        assert skipped == oskipped == obad == (k == 2), (k, skipped, oskipped, obad)
        if k == 2:
            assert np.isnan(gpu.norm.item())
    if path == "device":
        assert int(d_step.item()) == 2
    rep = H.compare_state(gpu, ref)
    _assert(rep)
    assert rep.exact == rep.n
    # a list whose only non-zero gradient is the NaN
    gpu.g.zero_()
    gpu.g[gpu.st.offsets[1] + 5] = float("nan")
    gpu.plan.grad_norm(gpu.norm, gpu.flag)
    torch.cuda.synchronize()
    assert int(gpu.flag.item()) == 1 and np.isnan(gpu.norm.item())
    gpu.plan.close()


@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")])
def test_nonfinite_reported_without_clip(bad):
    """Without clipping the step runs and NaN/inf propagate exactly as in the
    oracle; the flag reports them."""
    w = _small("report", steps=2)
    gpu = H.GpuSide(w)
    ref = H.OracleRun.from_state(gpu.st)
    hp_g, hp_o = H.hp_pair(w)
    for k in (1, 2):
        gpu.set_grad(k)
        if k == 2:
            gpu.g[gpu.st.offsets[8] + 12345] = bad
        gpu.step(hp_g)
        _, _, obad = ref.step(H.to_u16(gpu.g), hp_o)
        assert bool(gpu.flag.item()) == obad == (k == 2)
    rep = H.compare_state(gpu, ref)
    _assert(rep)
    gpu.plan.close()


def test_grad_norm_deterministic_and_matches_oracle():
    w = W.WORKLOADS["opt125m_bf16_kahan"]
    gpu = H.GpuSide(w)
    gpu.set_grad(1)
    norms = []
    for _ in range(3):
        gpu.plan.grad_norm(gpu.norm, gpu.flag)
        norms.append(float(gpu.norm.item()))
    assert norms[0] == norms[1] == norms[2]
    g = H.to_u16(gpu.g)
    o = O.load()
    sumsq, bad = o.grad_sumsq([g[off:off + n] for off, n in zip(gpu.st.offsets, w.numels)])
    _, onorm = o.clip_coef(sumsq, 1.0)
    assert not bad and gpu.flag.item() == 0
    # both sides sum the exact squares with fp64-level error
    assert abs(norms[0] - onorm) <= 1e-13 * onorm
    gpu.plan.close()


def test_grad_norm_with_huge_and_tiny_values():
    """Values whose squares leave fp32 range take the fp64 path."""
    w = _small("huge", sizes=[4096, 100])
    gpu = H.GpuSide(w)
    gpu.g.zero_()
    gpu.g[5] = 3.0e30
    gpu.g[6] = -2.0e19
    gpu.g[7] = 1.0e-30
    gpu.g[4096 + 8] = 0.5
    gpu.plan.grad_norm(gpu.norm, gpu.flag)
    g = H.to_u16(gpu.g)
    o = O.load()
    sumsq, bad = o.grad_sumsq([g[off:off + n] for off, n in zip(gpu.st.offsets, w.numels)])
    assert not bad and gpu.flag.item() == 0
    onorm = float(np.sqrt(sumsq))
    assert abs(gpu.norm.item() - onorm) <= 1e-12 * onorm
    gpu.plan.close()


def test_empty_plan_and_zero_length_tensors():
    z = torch.zeros(0, dtype=torch.bfloat16, device="cuda")
    plan = A.Plan([z], [z], [z], [z], [z], W.MODE_BF16_KAHAN, norm=True)
    norm = torch.full((1,), 7.0, dtype=torch.float64, device="cuda")
    flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    plan.step(A.hparams(max_grad_norm=1.0), 1, grad_norm=norm, nonfinite=flag)
    torch.cuda.synchronize()
    assert norm.item() == 0.0 and flag.item() == 0
    assert plan.info.grid == 0
    plan.close()
    empty = A.adamw_plan_create([], W.MODE_MIXED, 0)
    A.adamw_step(empty, A.hparams(), 1)
    A.adamw_plan_destroy(empty)


def test_api_errors_on_gpu():
    w = _small("err", sizes=[1000])
    st = W.make_state(w, "cuda")
    g = torch.zeros(st.aux.numel(), dtype=torch.bfloat16, device="cuda")
    v = st.views
    plan = A.Plan(v(st.param), v(g), v(st.exp_avg), v(st.exp_avg_sq), v(st.aux), w.mode, norm=False)
    with pytest.raises(A.AdamWError) as e:
        plan.step(A.hparams(max_grad_norm=1.0), 1)
    assert e.value.status == A.ADAMW_ERR_NO_NORM
    with pytest.raises(A.AdamWError) as e:
        plan.step(A.hparams(beta1=1.5), 1)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    with pytest.raises(A.AdamWError) as e:
        plan.step(A.hparams(), 0)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_create([(st.param.data_ptr() + 1, g.data_ptr(), st.exp_avg.data_ptr(),
                              st.exp_avg_sq.data_ptr(), st.aux.data_ptr(), 10)], w.mode)
    assert e.value.status == A.ADAMW_ERR_MISALIGNED
    plan.close()


@pytest.mark.parametrize("fuse", [True, False])
def test_clipped_step_without_a_flag_is_refused_before_any_launch(fuse):
    """A clipped step may be skipped, so it must report the non-finite flag:
    adamw_step refuses it without one (INVALID_ARG) and writes nothing; the
    Plan wrapper then supplies its own flag tensor."""
    w = _small("clipflag", sizes=[1000, 70001], mode=W.MODE_MIXED, max_grad_norm=1.0)
    gpu = H.GpuSide(w)
    if not fuse:
        gpu.plan.close()
        v = gpu.st.views
        gpu.plan = A.Plan(v(gpu.st.param), v(gpu.g), v(gpu.st.exp_avg), v(gpu.st.exp_avg_sq),
                          v(gpu.st.aux), w.mode, norm=True, fuse=False)
    assert gpu.plan.info.fused == (1 if fuse else 0)
    gpu.set_grad(1)
    before = [H.to_np(x).copy() for x in (gpu.st.param, gpu.st.exp_avg, gpu.st.exp_avg_sq, gpu.st.aux)]
    hp = A.hparams(**w.hparams())
    with pytest.raises(A.AdamWError) as e:
        A.adamw_step(gpu.plan.handle, hp, 1, gpu.norm.data_ptr(), 0,
                     torch.cuda.current_stream().cuda_stream)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    torch.cuda.synchronize()
    after = [H.to_np(x) for x in (gpu.st.param, gpu.st.exp_avg, gpu.st.exp_avg_sq, gpu.st.aux)]
    for a, b in zip(before, after):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    # the wrapper's default flag: a step with an inf is skipped and says so
    gpu.g[3] = float("inf")
    gpu.plan.step(hp, 1)
    torch.cuda.synchronize()
    assert gpu.plan.last_nonfinite is not None and int(gpu.plan.last_nonfinite.item()) == 1
    # without clipping the flag stays optional
    A.adamw_step(gpu.plan.handle, A.hparams(), 1, 0, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    gpu.plan.close()


def test_copy_probe_copies():
    src = torch.randint(-2**31, 2**31 - 1, (1 << 22,), dtype=torch.int32, device="cuda")
    dst = torch.zeros_like(src)
    A.adamw_copy_probe(dst.data_ptr(), src.data_ptr(), src.numel() * 4,
                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)
    with pytest.raises(A.AdamWError):
        A.adamw_copy_probe(dst.data_ptr() + 4, src.data_ptr(), 64)


def test_steps_on_a_side_stream_and_a_second_plan():
    """Two independent plans on two streams give the same bytes as one run."""
    w = _small("streams", sizes=[70000, 333])
    a, b = H.GpuSide(w), H.GpuSide(w)
    hp, _ = H.hp_pair(w)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for k in (1, 2, 3):
        a.set_grad(k)
        b.set_grad(k)
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            a.plan.step(hp, k)
        with torch.cuda.stream(s2):
            b.plan.step(hp, k)
    torch.cuda.synchronize()
    for x, y in zip((a.st.param, a.st.aux), (b.st.param, b.st.aux)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    a.plan.close()
    b.plan.close()


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.0), (W.MODE_MIXED, 1.0)])
def test_gradients_in_pinned_host_memory(mode, clip):
    """A plan whose gradients live in pinned host memory (read by the kernels
    over the CPU-GPU link) gives the same bytes as one with device gradients."""
    w = _small("hostgrad", mode=mode, max_grad_norm=clip, steps=3)
    a = H.GpuSide(w)
    b_state = W.make_state(w, "cuda")
    host_g = torch.zeros(a.g.numel(), dtype=torch.bfloat16, pin_memory=True)
    v = b_state.views
    plan_b = A.Plan(v(b_state.param), v(host_g), v(b_state.exp_avg), v(b_state.exp_avg_sq),
                    v(b_state.aux), mode, norm=True)
    hp, _ = H.hp_pair(w)
    norm_a = torch.zeros(1, dtype=torch.float64, device="cuda")
    norm_b = torch.zeros(1, dtype=torch.float64, device="cuda")
    for k in (1, 2, 3):
        a.set_grad(k)
        host_g.copy_(a.g)
        a.plan.step(hp, k, grad_norm=norm_a if clip else None)
        plan_b.step(hp, k, grad_norm=norm_b if clip else None)
    torch.cuda.synchronize()
    for x, y in zip((a.st.param, a.st.exp_avg, a.st.exp_avg_sq, a.st.aux),
                    (b_state.param, b_state.exp_avg, b_state.exp_avg_sq, b_state.aux)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    if clip:
        assert norm_a.item() == norm_b.item()
    a.plan.close()
    plan_b.close()


def test_buffers_of_another_kind_are_refused_before_any_launch():
    """Unpinned host memory on a device without pageable access, or any
    pointer the device cannot dereference, is an error code, not a fault.
    (On devices with pageable-memory access, unpinned host memory is valid.)"""
    st = W.make_state(_small("acc", sizes=[64]), "cuda")
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    cpu_g = torch.zeros(64, dtype=torch.bfloat16)          # pageable host memory
    entry = (st.param.data_ptr(), cpu_g.data_ptr(), st.exp_avg.data_ptr(),
             st.exp_avg_sq.data_ptr(), st.aux.data_ptr(), 64)
    pageable = getattr(torch.cuda.get_device_properties(0), "pageable_memory_access", None)
    try:
        plan = A.adamw_plan_create([entry], W.MODE_BF16_KAHAN)
        A.adamw_plan_destroy(plan)
        accepted = True
    except A.AdamWError as e:
        assert e.status == A.ADAMW_ERR_NOT_ACCESSIBLE
        accepted = False
    if pageable is not None:
        assert accepted == bool(pageable)
    del g


def test_step_table_over_a_device_table_matches_a_plan():
    """adamw_step_table takes the tensor table from device memory, caches one
    plan for it, and updates exactly like an explicit plan."""
    w = _small("table", mode=W.MODE_MIXED, max_grad_norm=0.5, steps=3)
    a = H.GpuSide(w)
    b = W.make_state(w, "cuda")
    g = torch.zeros_like(a.g)
    v = b.views
    entries = [A.adamw_tensor_t(*(t.data_ptr() for t in ts), ts[0].numel())
               for ts in zip(v(b.param), v(g), v(b.exp_avg), v(b.exp_avg_sq), v(b.aux))]
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
    for x, y in zip((a.st.param, a.st.exp_avg, a.st.exp_avg_sq, a.st.aux),
                    (b.param, b.exp_avg, b.exp_avg_sq, b.aux)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    assert norm_a.item() == norm_b.item()
    a.plan.close()


# ----------------------------------------------- device-resident step path --

def _twin(w):
    """Two identical states of workload w: one stepped by the host path, one
    by the device-resident path."""
    a = H.GpuSide(w)
    b_state = W.make_state(w, "cuda")
    v = b_state.views
    b_plan = A.Plan(v(b_state.param), v(a.g), v(b_state.exp_avg), v(b_state.exp_avg_sq),
                    v(b_state.aux), w.mode, norm=True)
    return a, b_state, b_plan


def _same_state(x, y):
    for p, q in zip((x.param, x.exp_avg, x.exp_avg_sq, x.aux), (y.param, y.exp_avg, y.exp_avg_sq, y.aux)):
        if p is not None:
            assert torch.equal(p.view(torch.uint8), q.view(torch.uint8))


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.0), (W.MODE_BF16_KAHAN, 0.5),
                                       (W.MODE_MIXED, 0.0), (W.MODE_MIXED, 1.0),
                                       (W.MODE_REMAINDER, 1.0)])
def test_device_step_matches_host_step(mode, clip):
    """Hyperparameters and the step counter in device memory give the same
    bytes as the host path, including a skipped step (inf at step 3)."""
    w = _small("dev", mode=mode, max_grad_norm=clip, steps=5,
               inf_at=(3, 8, 777) if clip else None)
    a, b_state, b_plan = _twin(w)
    hp, _ = H.hp_pair(w)
    d_hp = A.device_hparams(hp)
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_b = torch.zeros(1, dtype=torch.float64, device="cuda")
    f_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = A.STEP_CLIP if clip else 0
    for k in range(1, 6):
        a.set_grad(k)                  # the twin plan reads the same buffer
        skipped = a.step(hp)
        b_plan.step_device(d_hp, d_step, flags, grad_norm=n_b if clip else None, nonfinite=f_b)
        torch.cuda.synchronize()
        assert int(f_b.item()) == int(a.flag.item())
        assert int(d_step.item()) == a.t
        if clip:
            assert n_b.item() == a.norm.item()
        assert skipped == (clip > 0 and k == 3)
    _same_state(a.st, b_state)
    a.plan.close()
    b_plan.close()


@pytest.mark.parametrize("clip", [0.0, 1.0])
def test_device_step_memo_across_beta_changes_and_large_t(clip):
    """The memo of the next step's scalars (computed by CTA 0 from a table
    of the betas' squares, rebuilt when the betas change): device steps with
    the betas changed twice and the counter moved to large t (many set bits,
    so the table's squares up to 2^40 are used) give the bytes of the host
    path at the same t, every step; CTA 0 of this list has no elements."""
    w = _small("memo", max_grad_norm=clip, steps=1)
    a, b_state, b_plan = _twin(w)
    base = w.hparams()
    hps = {k: A.hparams(**{**base, **kw}) for k, kw in
           {"x": {}, "y": dict(beta1=0.8, beta2=0.99), "z": dict(beta1=0.95, beta2=0.9995)}.items()}
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_a = torch.zeros(1, dtype=torch.float64, device="cuda")
    f_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_b = torch.zeros(1, dtype=torch.float64, device="cuda")
    f_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    big = (1 << 40) + (1 << 33) + 12345
    plan_t = [(1, "x"), (2, "x"), (3, "x"), (4, "y"), (5, "y"), (6, "y"), (big, "y"), (big + 1, "y"),
              (big + 2, "z"), (big + 3, "z"), (7, "x"), (8, "x")]
    flags = A.STEP_CLIP if clip else 0
    for k, (t, key) in enumerate(plan_t):
        a.set_grad(k + 1)
        hp = hps[key]
        a.plan.step(hp, t, grad_norm=n_a if clip else None, nonfinite=f_a)
        if int(d_step.item()) != t - 1:
            d_step.fill_(t - 1)
        b_plan.step_device(A.device_hparams(hp), d_step, flags, grad_norm=n_b if clip else None,
                           nonfinite=f_b)
        torch.cuda.synchronize()
        assert int(d_step.item()) == t and int(f_b.item()) == int(f_a.item()) == 0
        _same_state(a.st, b_state)
    a.plan.close()
    b_plan.close()


def test_device_step_refuses_invalid_hparams_on_device():
    w = _small("devbad", sizes=[4096, 77], steps=1)
    a, b_state, b_plan = _twin(w)
    a.set_grad(1)
    before = [t.clone() for t in (b_state.param, b_state.exp_avg, b_state.exp_avg_sq, b_state.aux)]
    d_hp = A.device_hparams(A.hparams(beta1=1.5))
    d_step = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    b_plan.step_device(d_hp, d_step, 0, nonfinite=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == -1 and int(d_step.item()) == 7
    for x, y in zip(before, (b_state.param, b_state.exp_avg, b_state.exp_avg_sq, b_state.aux)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    a.plan.close()
    b_plan.close()


@pytest.mark.parametrize("mode,clip", [(W.MODE_BF16_KAHAN, 0.0), (W.MODE_MIXED, 1.0)])
def test_device_step_replayed_from_a_cuda_graph(mode, clip):
    """One device-resident step captured in a CUDA graph and replayed with a
    changing learning rate (written to the device hyperparameters between
    replays) equals the host path with the same per-step lr."""
    w = _small("graph", mode=mode, max_grad_norm=clip, steps=6)
    a, b_state, b_plan = _twin(w)
    flags = A.STEP_CLIP if clip else 0
    hps = [A.hparams(**{**w.hparams(), "lr": 2e-4 * (k + 1) / 6}) for k in range(6)]
    d_hp = A.device_hparams(hps[0])
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    norm = torch.zeros(1, dtype=torch.float64, device="cuda")
    # load the kernels once outside the capture (a throwaway list)
    warm = _small("warm", mode=mode, sizes=[64], steps=1)
    wa, wb_state, wb_plan = _twin(warm)
    wb_plan.step_device(A.device_hparams(hps[0]), torch.zeros(1, dtype=torch.int64, device="cuda"),
                        flags, grad_norm=norm if clip else None)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        b_plan.step_device(d_hp, d_step, flags, grad_norm=norm if clip else None)
    for k in range(6):
        a.set_grad(k + 1)
        a.step(hps[k], want_flag=False)
        d_hp.copy_(A.device_hparams(hps[k]))
        graph.replay()
    torch.cuda.synchronize()
    assert int(d_step.item()) == 6
    _same_state(a.st, b_state)
    for p in (a.plan, b_plan, wa.plan, wb_plan):
        p.close()


def test_schedule_and_step_replayed_from_a_cuda_graph():
    """The recipe's linear warm-up schedule and the step, both on the device,
    captured once and replayed: every update uses the schedule's lr for its
    own t, bit-identical to the host path fed the oracle's schedule."""
    import oracle as O
    o = O.load()
    w = _small("sched", steps=8)
    a, b_state, b_plan = _twin(w)
    base, warm, total = 2e-4, 3, 6
    d_hp = A.device_hparams(A.hparams(**w.hparams()))
    d_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    warm_state = _small("warm2", sizes=[64], steps=1)
    wa, wb_state, wb_plan = _twin(warm_state)
    scratch_hp = A.device_hparams(A.hparams())
    scratch_step = torch.zeros(1, dtype=torch.int64, device="cuda")
    A.adamw_lr_linear_warmup_device(scratch_hp.data_ptr(), scratch_step.data_ptr(), base, warm, total,
                                    torch.cuda.current_stream().cuda_stream)
    wb_plan.step_device(scratch_hp, scratch_step, 0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        A.adamw_lr_linear_warmup_device(d_hp.data_ptr(), d_step.data_ptr(), base, warm, total,
                                        torch.cuda.current_stream().cuda_stream)
        b_plan.step_device(d_hp, d_step, 0)
    for k in range(1, 9):
        a.set_grad(k)
        lr = o.lr_linear_warmup(np.float32(base), k, warm, total)
        a.step(A.hparams(**{**w.hparams(), "lr": lr}), want_flag=False)
        graph.replay()
    torch.cuda.synchronize()
    assert int(d_step.item()) == 8
    _same_state(a.st, b_state)
    for p in (a.plan, b_plan, wa.plan, wb_plan):
        p.close()


@pytest.mark.parametrize("mode", [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER,
                                  W.MODE_BF16_PLAIN, W.MODE_BF16_KAHAN_V32])
def test_canaries_around_tensors_stay_untouched(mode):
    """Bounds check without a sanitizer: every element of the flat buffers
    that belongs to no tensor (the skew, the gaps between tensors, a
    4096-element tail) holds a canary pattern, and the gradient buffer is
    read-only; after clipped and unclipped steps not one of those bytes may
    have changed."""
    w = _small("canary", mode=mode, max_grad_norm=0.0, steps=3)
    st = W.make_state(w, "cuda", align_elems=8, skew=5, tail_pad=4096)
    gpu = H.GpuSide(w, "cuda", st)
    covered = torch.zeros(st.param.numel(), dtype=torch.bool, device="cuda")
    for o, n in zip(st.offsets, w.numels):
        covered[o:o + n] = True
    gaps = ~covered
    bufs = [b for b in (st.param, st.exp_avg, st.exp_avg_sq, st.aux) if b is not None]
    for b in bufs:
        raw = b.view(torch.uint8).view(-1, b.element_size())
        raw[gaps] = 0xA5
    hp_plain, _ = H.hp_pair(w)
    hp_clip = A.hparams(**{**w.hparams(), "max_grad_norm": 0.5})
    for k in range(1, 4):
        gpu.set_grad(k)
        g_before = gpu.g.clone()
        gpu.plan.step(hp_clip if k == 2 else hp_plain, k, grad_norm=gpu.norm if k == 2 else None)
        torch.cuda.synchronize()
        assert torch.equal(gpu.g.view(torch.int16), g_before.view(torch.int16)), "grad written"
    for b in bufs:
        raw = b.view(torch.uint8).view(-1, b.element_size())
        assert bool((raw[gaps] == 0xA5).all()), f"a {b.dtype} canary changed"
    gpu.plan.close()
