"""adamw_grad_norm_noalloc: the global gradient norm for callers that cannot
allocate device memory (their device memory belongs to a caching allocator,
or they must not synchronise the device, as cudaMalloc/cudaFree may).  It
runs from a fixed file-scope scratch array in the library instead of a plan.

Checked through the C ABI against the plan-based adamw_grad_norm on the same
gradients, on two calls in a row (the second after the scratch holds the
first call's contents), within the norm tolerance the other GPU tests use
(1e-13 relative; both sum the exact squares), with identical non-finite
flags.  This file is collected last so that a run stopping at its first
failure has run every other test already."""
import math

import pytest
import torch

import parity_harness as H
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-13


def _list(align_elems, skew):
    sizes = [1, 7, 8, 9, 4095, 65537, 0, 3, 1000003, 255, 256, 257, 3 * 768, 50272, 4_000_000]
    w = W.Workload("noalloc", W.MODE_BF16_KAHAN, tuple(W.TensorSpec(f"t{i}", n) for i, n in enumerate(sizes)),
                   2, lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, heavy_tail=True)
    return H.GpuSide(w, "cuda", W.make_state(w, "cuda", align_elems, skew))


def _norms(gpu):
    dev = gpu.g.device
    ref_n = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    ref_f = torch.full((1,), -1, dtype=torch.int32, device=dev)
    na_n = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    na_f = torch.full((1,), -1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    gpu.plan.grad_norm(ref_n, ref_f)
    entries = [(0, g.data_ptr(), 0, 0, 0, g.numel()) for g in gpu.st.views(gpu.g)]
    A.adamw_grad_norm_noalloc(entries, na_n.data_ptr(), na_f.data_ptr(), stream)
    torch.cuda.synchronize()
    return float(ref_n.item()), int(ref_f.item()), float(na_n.item()), int(na_f.item())


@pytest.mark.parametrize("layout", [(8, 0), (1, 3)])
def test_noalloc_norm_matches_plan_norm_on_two_calls(layout):
    gpu = _list(*layout)
    # first call: finite gradients
    gpu.set_grad(1)
    r, rf, n, nf = _norms(gpu)
    assert rf == nf == 0
    assert r > 0 and abs(n - r) <= NORM_RTOL * r, (n, r)
    # second call, different gradients with one inf: same flag, both inf
    gpu.set_grad(2)
    gpu.g[gpu.st.offsets[8] + 4321] = float("inf")
    r2, rf2, n2, nf2 = _norms(gpu)
    assert rf2 == nf2 == 1
    assert math.isinf(r2) and math.isinf(n2)
    # third call back to finite values: the scratch's stale contents do not leak
    gpu.set_grad(2)
    r3, rf3, n3, nf3 = _norms(gpu)
    assert rf3 == nf3 == 0 and abs(n3 - r3) <= NORM_RTOL * r3 and r3 != r
    gpu.plan.close()


def test_noalloc_rejects_lists_beyond_its_maximum():
    g = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    entries = [(0, g.data_ptr(), 0, 0, 0, 16)] * (A.NOALLOC_MAX_TENSORS + 1)
    with pytest.raises(A.AdamWError) as e:
        A.adamw_grad_norm_noalloc(entries)
    assert e.value.status == A.ADAMW_ERR_TOO_LARGE
    with pytest.raises(A.AdamWError) as e:
        A.adamw_grad_norm_noalloc([(0, g.data_ptr() + 1, 0, 0, 0, 4)])
    assert e.value.status == A.ADAMW_ERR_MISALIGNED
    # an empty list is a norm of zero
    out = torch.full((1,), 5.0, dtype=torch.float64, device="cuda")
    A.adamw_grad_norm_noalloc([], out.data_ptr())
    torch.cuda.synchronize()
    assert out.item() == 0.0
