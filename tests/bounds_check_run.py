"""Runs the main paths of a bounds-checked build of the library (loaded from
ADAMW_SM_LIBRARY, built with -DADAMW_CHECK_BOUNDS=1) and checks that no
chunk is ever refused, that every result is still bit-identical to the
oracle, and that a lengthened chunk is refused before any byte of it is
touched.  Run by tests/test_gpu_bounds_check.py in a child process (the
library a process loads is fixed for its lifetime); exits non-zero on any
failure."""
import sys

import numpy as np
import torch

import parity_harness as H
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import workloads as W

RAGGED = [1, 7, 8, 9, 4095, 65537, 0, 3, 1000003, 255, 256, 257, 3 * 768, 50272]
LONG = [3_000_001, 7, 2_500_003, 65_537, 1_999_999, 1, 4_194_304, 257, 1_048_583, 9]
# more than 8 rounds of tiles: the last rounds are claimed at run time
CLAIMED = [30_000_001, 7, 6_500_003, 65_537, 1, 4_194_304, 1_048_583]


def workload(name, mode, sizes, clip, steps=3):
    return W.Workload(name, mode, tuple(W.TensorSpec(f"t{i}", n) for i, n in enumerate(sizes)),
                      steps, lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                      max_grad_norm=clip, heavy_tail=True)


def parity_with_status(w, layout, device_step=False):
    gpu = H.GpuSide(w, "cuda", W.make_state(w, "cuda", *layout))
    ref = H.OracleRun.from_state(gpu.st)
    hp_g, hp_o = H.hp_pair(w)
    d_hp, d_step = A.device_hparams(hp_g), torch.zeros(1, dtype=torch.int64, device="cuda")
    for k in range(1, w.steps + 1):
        gpu.set_grad(k)
        if device_step:
            gpu.plan.step_device(d_hp, d_step, A.STEP_CLIP if w.max_grad_norm > 0 else 0,
                                 grad_norm=gpu.norm if w.max_grad_norm > 0 else None,
                                 nonfinite=gpu.flag)
        else:
            gpu.step(hp_g)
        ref.step(H.to_u16(gpu.g), hp_o)
    status = A.adamw_plan_device_status(gpu.plan.handle)
    rep = H.compare_state(gpu, ref)
    fused = gpu.plan.info.fused
    gpu.plan.close()
    assert status == 0, f"{w.name} mode {w.mode}: device status {status}"
    assert rep.ok() and rep.exact == rep.n, f"{w.name} mode {w.mode}: {rep.failures[:3]}"
    return fused


def refused_chunk_is_left_alone():
    """The last chunk of the list (the end of its last tensor, which is
    followed by 4096 elements of padding in every buffer, so the lengthened
    chunk would stay inside the allocations even unchecked) is lengthened by
    8 elements: the update must skip exactly that chunk and report it."""
    w = workload("corrupt", W.MODE_BF16_KAHAN, [5000, 30000], 0.0, steps=1)
    st = W.make_state(w, "cuda", align_elems=8, skew=0, tail_pad=4096)
    gpu = H.GpuSide(w, "cuda", st)
    v = st.views
    entries = [tuple(t.data_ptr() for t in ts) + (ts[0].numel(),)
               for ts in zip(v(st.param), v(gpu.g), v(st.exp_avg), v(st.exp_avg_sq), v(st.aux))]
    chunks = A.adamw_plan_chunks(entries, w.mode, gpu.plan.info.grid)
    last = [i for i, c in enumerate(chunks) if c.tensor == 1 and c.offset + c.len == 30000]
    assert len(last) == 1, "no unique last chunk"
    c = chunks[last[0]]
    lo, hi = st.offsets[1] + c.offset, st.offsets[1] + c.offset + c.len
    before = st.param.clone()
    A.adamw_plan_test_corrupt_chunk(gpu.plan.handle, last[0], 8)
    gpu.set_grad(1)
    gpu.step(A.hparams(**w.hparams()), want_flag=False)
    status = A.adamw_plan_device_status(gpu.plan.handle)
    assert status & A.STATUS_BOUNDS, f"lengthened chunk not reported (status {status})"
    assert torch.equal(st.param[lo:hi + 4096].view(torch.int16), before[lo:hi + 4096].view(torch.int16)), \
        "the refused chunk (or the padding after it) was written"
    assert not torch.equal(st.param[st.offsets[0]:st.offsets[0] + 5000].view(torch.int16),
                           before[st.offsets[0]:st.offsets[0] + 5000].view(torch.int16)), \
        "the other chunks were not updated"
    gpu.plan.close()


def main():
    assert A.adamw_build_flags() & A.BUILD_CHECK_BOUNDS, "not a bounds-checked build"
    n = 0
    for mode in list(range(5)) + list(W.ANYPREC_MODES):
        for clip in (0.0, 0.5):
            for layout in ((8, 0), (1, 3)):
                parity_with_status(workload("ragged", mode, RAGGED, clip), layout)
                n += 1
    for mode in (W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER, W.MODE_ANYPREC | 7):
        for clip in (0.0, 0.5):
            parity_with_status(workload("long", mode, LONG, clip), (1, 3))
            parity_with_status(workload("long", mode, LONG, clip), (8, 0), device_step=True)
            n += 2
    for mode in (W.MODE_BF16_KAHAN, W.MODE_MIXED):
        parity_with_status(workload("claimed", mode, CLAIMED, 0.5, steps=2), (1, 3))
        parity_with_status(workload("claimed", mode, CLAIMED, 0.0, steps=2), (8, 0), device_step=True)
        n += 2
    fused = parity_with_status(workload("fused", W.MODE_MIXED, [13_850_000], 1.0), (8, 0))
    assert fused == 1
    n += 1
    refused_chunk_is_left_alone()
    print(f"bounds-checked build: {n} parity runs without a refused chunk; a lengthened chunk "
          "was refused and left alone")
    return 0


if __name__ == "__main__":
    sys.exit(main())
