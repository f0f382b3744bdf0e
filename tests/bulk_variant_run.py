"""Runs the bf16 Kahan paths of the library built with its optional
cp.async.bulk staging of the update (loaded from ADAMW_SM_LIBRARY, built
with -DADAMW_BULK=1) against the oracle: contiguous and round-robin
partitions, ragged and misaligned lists, clipping with a skipped step,
every element bit-identical, and the plan's device status clean (a bounded
mbarrier wait that gave up would set it).  Run by
tests/test_gpu_bulk_variant.py in a child process (the library a process
loads is fixed for its lifetime); exits non-zero on any failure."""
import sys

import parity_harness as H
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import workloads as W

RAGGED = [1, 7, 8, 9, 4095, 65537, 0, 3, 1000003, 255, 256, 257, 3 * 768, 50272]
LONG = [3_000_001, 7, 2_500_003, 65_537, 1_999_999, 1, 4_194_304, 257, 1_048_583, 9]


def workload(name, sizes, clip, steps=3, inf_at=None):
    return W.Workload(name, W.MODE_BF16_KAHAN, tuple(W.TensorSpec(f"t{i}", n) for i, n in enumerate(sizes)),
                      steps, lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                      max_grad_norm=clip, heavy_tail=True, inf_at=inf_at)


def parity(w, layout, fuse=True):
    gpu = H.GpuSide(w, "cuda", W.make_state(w, "cuda", *layout))
    if not fuse:
        gpu.plan.close()
        v = gpu.st.views
        gpu.plan = A.Plan(v(gpu.st.param), v(gpu.g), v(gpu.st.exp_avg), v(gpu.st.exp_avg_sq),
                          v(gpu.st.aux), w.mode, norm=True, fuse=False)
    ref = H.OracleRun.from_state(gpu.st)
    hp_g, hp_o = H.hp_pair(w)
    skipped = []
    for k in range(1, w.steps + 1):
        gpu.set_grad(k)
        s = gpu.step(hp_g)
        os_, _, _ = ref.step(H.to_u16(gpu.g), hp_o)
        assert s == os_, f"{w.name}: step {k} skipped {s}, oracle {os_}"
        if s:
            skipped.append(k)
    status = A.adamw_plan_device_status(gpu.plan.handle)
    rep = H.compare_state(gpu, ref)
    gpu.plan.close()
    assert status == 0, f"{w.name}: device status {status}"
    assert rep.ok() and rep.exact == rep.n, f"{w.name}: {rep.failures[:3]}"
    return skipped


def main():
    assert A.adamw_build_flags() & A.BUILD_BULK_STAGING, "not the staging build"
    n = 0
    parity(W.WORKLOADS["flat1m_bf16_kahan"], (8, 0))
    n += 1
    for clip in (0.0, 0.5):
        for layout in ((8, 0), (1, 3)):
            parity(workload("ragged", RAGGED, clip), layout)
            parity(workload("long", LONG, clip), layout)
            n += 2
    skipped = parity(workload("skip", LONG, 1.0, steps=4, inf_at=(2, 3, 777)), (8, 0), fuse=False)
    assert skipped == [2], skipped
    n += 1
    print(f"staging build: {n} parity runs bit-identical to the oracle, device status clean")
    return 0


if __name__ == "__main__":
    sys.exit(main())
