"""adamw_grad_norm_noalloc: the global gradient norm for callers that cannot
allocate device memory (their device memory belongs to a caching allocator,
or they must not synchronise the device, as cudaMalloc/cudaFree may).  It
runs from a fixed file-scope scratch array in the library instead of a plan.

Checked through the C ABI against the plan-based adamw_grad_norm on the same
gradients, on two calls in a row (the second after the scratch holds the
first call's contents), and against the oracle's compensated sum of squares
over the same bytes, within the norm tolerance the other GPU tests use
(1e-13 relative; all three sum the exact squares), with identical non-finite
flags -- for finite gradients, an inf, a NaN, and gradients so small that
their squares underflow fp32.  The caller's table is read during the call
only, also when it lives in pinned memory.  This file is collected last so
that a run stopping at its first failure has run every other test already."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle as O
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


def _entries(gpu):
    return [(0, g.data_ptr(), 0, 0, 0, g.numel()) for g in gpu.st.views(gpu.g)]


def _norms(gpu):
    dev = gpu.g.device
    ref_n = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    ref_f = torch.full((1,), -1, dtype=torch.int32, device=dev)
    na_n = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    na_f = torch.full((1,), -1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    gpu.plan.grad_norm(ref_n, ref_f)
    A.adamw_grad_norm_noalloc(_entries(gpu), na_n.data_ptr(), na_f.data_ptr(), stream)
    torch.cuda.synchronize()
    return float(ref_n.item()), int(ref_f.item()), float(na_n.item()), int(na_f.item())


def _oracle_norm(gpu):
    """The oracle's norm and flag over the same gradient bytes."""
    o = O.load()
    sumsq, bad = o.grad_sumsq([H.to_u16(g).reshape(-1).copy() for g in gpu.st.views(gpu.g)])
    return math.sqrt(sumsq), int(bad)


def _close(a, b):
    return abs(a - b) <= NORM_RTOL * abs(b)


@pytest.mark.parametrize("layout", [(8, 0), (1, 3)])
def test_noalloc_norm_matches_plan_norm_on_two_calls(layout):
    gpu = _list(*layout)
    # first call: finite gradients
    gpu.set_grad(1)
    r, rf, n, nf = _norms(gpu)
    on, of = _oracle_norm(gpu)
    assert rf == nf == of == 0
    assert r > 0 and _close(n, r) and _close(n, on), (n, r, on)
    # second call, different gradients with one inf: same flag, both inf
    gpu.set_grad(2)
    gpu.g[gpu.st.offsets[8] + 4321] = float("inf")
    r2, rf2, n2, nf2 = _norms(gpu)
    assert rf2 == nf2 == _oracle_norm(gpu)[1] == 1
    assert math.isinf(r2) and math.isinf(n2)
    # a NaN (the fp32 range check is false for NaN: the fp64 recount decides)
    gpu.set_grad(2)
    gpu.g[gpu.st.offsets[14] + 77] = float("nan")
    r3, rf3, n3, nf3 = _norms(gpu)
    assert rf3 == nf3 == _oracle_norm(gpu)[1] == 1
    assert math.isnan(r3) and math.isnan(n3)
    # back to finite values: the scratch's stale contents do not leak
    gpu.set_grad(2)
    r4, rf4, n4, nf4 = _norms(gpu)
    on4, of4 = _oracle_norm(gpu)
    assert rf4 == nf4 == of4 == 0 and _close(n4, r4) and _close(n4, on4) and r4 != r
    gpu.plan.close()


def test_noalloc_norm_of_gradients_whose_squares_underflow_fp32():
    """Every gradient near 1e-30 (squares about 1e-60, below fp32's range):
    the fp64 recount gives the exact sum, as the plan's norm and the oracle."""
    gpu = _list(8, 0)
    gen = torch.Generator(device="cuda").manual_seed(9)
    g = (torch.rand(gpu.g.numel(), generator=gen, device="cuda") + 0.5) * 1e-30
    gpu.g.copy_(g.to(torch.bfloat16))
    r, rf, n, nf = _norms(gpu)
    on, of = _oracle_norm(gpu)
    assert rf == nf == of == 0
    assert 0 < on < 1e-25 and _close(n, r) and _close(n, on), (n, r, on)
    gpu.plan.close()


def test_noalloc_table_may_change_as_soon_as_the_call_returns():
    """A caller's table in pinned host memory, rewritten right after the call
    returns (to another valid list: zero gradients of the same sizes): the
    norm is the one of the list as it was during the call."""
    gpu = _list(8, 0)
    gpu.set_grad(1)
    zeros = torch.zeros_like(gpu.g)
    views, zviews = gpu.st.views(gpu.g), gpu.st.views(zeros)
    n_t = len(views)
    raw = torch.empty(n_t * ctypes.sizeof(A.adamw_tensor_t), dtype=torch.uint8, pin_memory=True)
    table = (A.adamw_tensor_t * n_t).from_address(raw.data_ptr())
    for k, g in enumerate(views):
        table[k] = A.adamw_tensor_t(None, g.data_ptr(), None, None, None, g.numel())
    out = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # keep the GPU busy so the norm kernels are still queued when the table changes
    busy = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(20):
        busy.fill_(3)
    rc = A.load().adamw_grad_norm_noalloc(table, n_t, ctypes.c_void_p(out.data_ptr()),
                                          ctypes.c_void_p(flag.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == A.ADAMW_OK
    for k, z in enumerate(zviews):
        table[k] = A.adamw_tensor_t(None, z.data_ptr(), None, None, None, z.numel())
    torch.cuda.synchronize()
    on, of = _oracle_norm(gpu)
    assert int(flag.item()) == of == 0
    assert on > 0 and _close(float(out.item()), on), (float(out.item()), on)
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


def test_noalloc_accepts_its_largest_list():
    """4096 tensors (three launches' worth of list): the norm of every
    gradient, as the oracle sums it."""
    n_t = A.NOALLOC_MAX_TENSORS
    gen = torch.Generator(device="cuda").manual_seed(4)
    flat = (torch.randn(n_t * 40, generator=gen, device="cuda") * 1e-2).to(torch.bfloat16)
    sizes = [(k % 37) + 3 for k in range(n_t)]
    entries, offs, o = [], [], 0
    for n in sizes:
        entries.append((0, flat.data_ptr() + 2 * o, 0, 0, 0, n))
        offs.append(o)
        o += n
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    A.adamw_grad_norm_noalloc(entries, out.data_ptr(), flag.data_ptr())
    torch.cuda.synchronize()
    host = H.to_u16(flat)
    sumsq, bad = O.load().grad_sumsq([host[a:a + n].copy() for a, n in zip(offs, sizes)])
    assert int(flag.item()) == int(bad) == 0
    assert _close(float(out.item()), math.sqrt(sumsq))
