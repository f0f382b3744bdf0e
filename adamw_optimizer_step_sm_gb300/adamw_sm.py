"""Python binding of the adamw_sm C ABI (include/adamw_sm.h).

Argument marshalling only: every step of the optimizer runs in the library's
CUDA kernels.  The functions keep the C names; a non-zero status raises
``AdamWError``.  ``Plan`` is a small convenience wrapper that builds the
tensor table from torch tensors (torch supplies device memory and streams).

The library is built in-tree (``build.build``) on first use when its sources
are newer than the shared object (or taken from the path in the environment
variable ADAMW_SM_LIBRARY, for a build made with other tuning constants); if
it cannot be built or loaded, every call raises -- there is no fallback
implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MODE_BF16_KAHAN = 0
MODE_MIXED_FP32_MASTER = 1
MODE_MIXED_BF16_REMAINDER = 2
MODE_BF16_PLAIN = 3
MODE_BF16_KAHAN_FP32_VAR = 4
# AnyPrecisionAdamW storage: MODE_ANYPREC | ANYPREC_* flags (bf16 param and
# grad; each flag makes one optimizer buffer fp32, or drops the compensation).
MODE_ANYPREC = 16
ANYPREC_M_FP32 = 1
ANYPREC_V_FP32 = 2
ANYPREC_C_FP32 = 4
ANYPREC_NO_KAHAN = 8
ANYPREC_MODES = tuple(MODE_ANYPREC | f for f in range(16) if (f & 12) != 12)
PLAN_NORM = 1
BUILD_CHECK_BOUNDS = 1
BUILD_BULK_STAGING = 2
STATUS_WAIT_RAN_OUT = 1
STATUS_BOUNDS = 2
PLAN_NO_FUSE = 2
STEP_CLIP = 1
STEP_NORM = 2

ADAMW_OK = 0
ADAMW_ERR_INVALID_ARG = -1
ADAMW_ERR_MISALIGNED = -2
ADAMW_ERR_CUDA = -3
ADAMW_ERR_NO_NORM = -4
ADAMW_ERR_TOO_LARGE = -5
ADAMW_ERR_NOT_ACCESSIBLE = -6


class AdamWError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status}: {adamw_status_string(status)}")


class adamw_tensor_t(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("aux", ctypes.c_void_p), ("numel", ctypes.c_int64)]


class adamw_hparams_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("max_grad_norm", ctypes.c_float)]


class adamw_plan_info_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("n_tensors", ctypes.c_int32),
                ("total_elems", ctypes.c_int64), ("grid", ctypes.c_int32),
                ("block", ctypes.c_int32), ("n_chunks", ctypes.c_int64),
                ("scalar_elems", ctypes.c_int64), ("device", ctypes.c_int32),
                ("has_norm", ctypes.c_int32), ("norm_grid", ctypes.c_int32),
                ("fused", ctypes.c_int32)]


class adamw_chunk_t(ctypes.Structure):
    _fields_ = [("tensor", ctypes.c_int32), ("vec", ctypes.c_int32),
                ("offset", ctypes.c_int64), ("len", ctypes.c_int64),
                ("cta", ctypes.c_int32), ("pad_", ctypes.c_int32)]


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def load() -> ctypes.CDLL:
    """Build if needed and load the shared library (raises on failure)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ADAMW_SM_LIBRARY") or _build.build()
            L = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.adamw_plan_create.argtypes = [ctypes.POINTER(adamw_tensor_t), i32, i32, i32,
                                            ctypes.POINTER(vp)]
            L.adamw_step.argtypes = [vp, ctypes.POINTER(adamw_hparams_t), i64, vp, vp, vp]
            L.adamw_grad_norm.argtypes = [vp, vp, vp, vp]
            L.adamw_step_device.argtypes = [vp, vp, vp, i32, vp, vp, vp]
            L.adamw_plan_destroy.argtypes = [vp]
            L.adamw_plan_device_status.argtypes = [vp, ctypes.POINTER(i32)]
            L.adamw_plan_test_skew_barrier.argtypes = [vp, i64]
            L.adamw_plan_test_corrupt_chunk.argtypes = [vp, i64, i64]
            L.adamw_build_flags.argtypes = []
            L.adamw_build_flags.restype = i32
            L.adamw_lr_linear_warmup.argtypes = [ctypes.c_float, i64, i64, i64]
            L.adamw_lr_linear_warmup.restype = ctypes.c_float
            L.adamw_lr_linear_warmup_device.argtypes = [vp, vp, ctypes.c_float, i64, i64, vp]
            L.adamw_plan_get_info.argtypes = [vp, ctypes.POINTER(adamw_plan_info_t)]
            L.adamw_plan_chunks.argtypes = [ctypes.POINTER(adamw_tensor_t), i32, i32, i32,
                                            ctypes.POINTER(adamw_chunk_t), i64,
                                            ctypes.POINTER(i64)]
            L.adamw_step_scalars.argtypes = [ctypes.POINTER(adamw_hparams_t), i64,
                                             ctypes.POINTER(ctypes.c_float)]
            L.adamw_copy_probe.argtypes = [vp, vp, i64, vp]
            L.adamw_grad_norm_noalloc.argtypes = [ctypes.POINTER(adamw_tensor_t), i32, vp, vp, vp]
            L.adamw_step_table.argtypes = [vp, i32, i32, ctypes.POINTER(adamw_hparams_t), i64,
                                           vp, vp, vp]
            L.adamw_step_table_cache_clear.argtypes = []
            L.adamw_status_string.argtypes = [ctypes.c_int]
            L.adamw_status_string.restype = ctypes.c_char_p
            for name in ("adamw_plan_create", "adamw_step", "adamw_grad_norm", "adamw_step_device",
                         "adamw_plan_destroy", "adamw_plan_get_info", "adamw_plan_chunks",
                         "adamw_step_scalars", "adamw_copy_probe", "adamw_grad_norm_noalloc",
                         "adamw_step_table", "adamw_step_table_cache_clear",
                         "adamw_plan_device_status", "adamw_lr_linear_warmup_device",
                         "adamw_plan_test_skew_barrier", "adamw_plan_test_corrupt_chunk"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
        return _lib


def _check(rc: int, where: str):
    if rc != ADAMW_OK:
        raise AdamWError(rc, where)


def _table(entries) -> tuple[ctypes.Array, int]:
    entries = list(entries)
    arr = (adamw_tensor_t * max(1, len(entries)))()
    for i, e in enumerate(entries):
        arr[i] = e if isinstance(e, adamw_tensor_t) else adamw_tensor_t(*e)
    return arr, len(entries)


# ------------------------------------------------------------ C functions --

def adamw_status_string(status: int) -> str:
    return load().adamw_status_string(status).decode()


def adamw_plan_create(entries, mode: int, flags: int = 0) -> int:
    """entries: adamw_tensor_t or (param, grad, exp_avg, exp_avg_sq, aux, numel)
    tuples of device addresses.  Returns the plan handle."""
    arr, n = _table(entries)
    out = ctypes.c_void_p()
    _check(load().adamw_plan_create(arr, n, mode, flags, ctypes.byref(out)), "adamw_plan_create")
    return out.value


def adamw_step(plan: int, hp: adamw_hparams_t, step: int, d_grad_norm: int = 0,
               d_nonfinite: int = 0, stream: int = 0) -> None:
    _check(load().adamw_step(plan, ctypes.byref(hp), step, d_grad_norm or None,
                             d_nonfinite or None, stream or None), "adamw_step")


def adamw_step_device(plan: int, d_hp: int, d_step: int, flags: int = 0, d_grad_norm: int = 0,
                      d_nonfinite: int = 0, stream: int = 0) -> None:
    """A step whose hyperparameters (device adamw_hparams_t at d_hp) and
    applied-step counter (device int64 at d_step) live on the device."""
    _check(load().adamw_step_device(plan, d_hp, d_step, flags, d_grad_norm or None,
                                    d_nonfinite or None, stream or None), "adamw_step_device")


def adamw_grad_norm(plan: int, d_grad_norm: int = 0, d_nonfinite: int = 0,
                    stream: int = 0) -> None:
    _check(load().adamw_grad_norm(plan, d_grad_norm or None, d_nonfinite or None,
                                  stream or None), "adamw_grad_norm")


NOALLOC_MAX_TENSORS = 4096


def adamw_grad_norm_noalloc(entries, d_grad_norm: int = 0, d_nonfinite: int = 0,
                            stream: int = 0) -> None:
    """Global gradient norm of a tensor list without any device allocation
    (no plan; only .grad and .numel of each entry are read).  For callers
    that cannot call cudaMalloc; see include/adamw_sm.h."""
    arr, n = _table(entries)
    _check(load().adamw_grad_norm_noalloc(arr, n, d_grad_norm or None, d_nonfinite or None,
                                          stream or None), "adamw_grad_norm_noalloc")


def adamw_step_table(d_table: int, n_tensors: int, mode: int, hp: adamw_hparams_t, step: int,
                     d_grad_norm: int = 0, d_nonfinite: int = 0, stream: int = 0) -> None:
    """One step over a tensor table held in device memory at address d_table
    (n_tensors adamw_tensor_t entries); plans are cached by table contents."""
    _check(load().adamw_step_table(d_table, n_tensors, mode, ctypes.byref(hp), step,
                                   d_grad_norm or None, d_nonfinite or None, stream or None),
           "adamw_step_table")


def adamw_step_table_cache_clear() -> int:
    return load().adamw_step_table_cache_clear()


def adamw_plan_destroy(plan: int) -> None:
    _check(load().adamw_plan_destroy(plan), "adamw_plan_destroy")


def adamw_lr_linear_warmup(base_lr: float, step: int, warmup: int, total: int) -> float:
    return float(load().adamw_lr_linear_warmup(base_lr, step, warmup, total))


def adamw_lr_linear_warmup_device(d_hp: int, d_step: int, base_lr: float, warmup: int,
                                  total: int, stream: int = 0) -> None:
    _check(load().adamw_lr_linear_warmup_device(d_hp, d_step, base_lr, warmup, total,
                                                stream or None), "adamw_lr_linear_warmup_device")


def adamw_plan_device_status(plan: int) -> int:
    """Reads and clears the plan's device status word (1: a bounded wait in
    one of its kernels ran out)."""
    out = ctypes.c_int32(0)
    _check(load().adamw_plan_device_status(plan, ctypes.byref(out)), "adamw_plan_device_status")
    return out.value


def adamw_build_flags() -> int:
    """BUILD_CHECK_BOUNDS / BUILD_BULK_STAGING bits of the loaded library."""
    return int(load().adamw_build_flags())


def adamw_plan_test_corrupt_chunk(plan: int, chunk: int, delta: int) -> None:
    """Bounds-checked builds only: lengthen update chunk ``chunk`` by ``delta``."""
    _check(load().adamw_plan_test_corrupt_chunk(plan, chunk, delta), "adamw_plan_test_corrupt_chunk")


def adamw_plan_test_skew_barrier(plan: int, delta: int) -> None:
    """Failure-path tests only: misalign the fused step's barrier counter."""
    _check(load().adamw_plan_test_skew_barrier(plan, delta), "adamw_plan_test_skew_barrier")


def adamw_plan_get_info(plan: int) -> adamw_plan_info_t:
    info = adamw_plan_info_t()
    _check(load().adamw_plan_get_info(plan, ctypes.byref(info)), "adamw_plan_get_info")
    return info


def adamw_plan_chunks(entries, mode: int, grid: int) -> list[adamw_chunk_t]:
    arr, n = _table(entries)
    count = ctypes.c_int64(0)
    rc = load().adamw_plan_chunks(arr, n, mode, grid, None, 0, ctypes.byref(count))
    if rc not in (ADAMW_OK, ADAMW_ERR_TOO_LARGE):
        _check(rc, "adamw_plan_chunks")
    out = (adamw_chunk_t * max(1, count.value))()
    _check(load().adamw_plan_chunks(arr, n, mode, grid, out, count.value, ctypes.byref(count)),
           "adamw_plan_chunks")
    return list(out[:count.value])


def adamw_step_scalars(hp: adamw_hparams_t, step: int) -> list[float]:
    out = (ctypes.c_float * 5)()
    _check(load().adamw_step_scalars(ctypes.byref(hp), step, out), "adamw_step_scalars")
    return list(out)


def adamw_copy_probe(dst: int, src: int, nbytes: int, stream: int = 0) -> None:
    _check(load().adamw_copy_probe(dst, src, nbytes, stream or None), "adamw_copy_probe")


def hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
            max_grad_norm=0.0) -> adamw_hparams_t:
    return adamw_hparams_t(lr, beta1, beta2, eps, weight_decay, max_grad_norm)


# --------------------------------------------------------- torch wrapper --

def buffer_dtypes(mode: int):
    """torch dtypes of param, grad, exp_avg, exp_avg_sq and aux in a storage
    mode (None: the mode does not use that buffer)."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    named = {MODE_BF16_KAHAN: (bf,) * 5,
             MODE_MIXED_FP32_MASTER: (f32, bf, f32, f32, bf),
             MODE_MIXED_BF16_REMAINDER: (bf, bf, f32, f32, torch.int16),
             MODE_BF16_PLAIN: (bf,) * 4 + (None,),
             MODE_BF16_KAHAN_FP32_VAR: (bf, bf, bf, f32, bf)}
    if mode in named:
        return named[mode]
    if mode not in ANYPREC_MODES:
        raise ValueError(f"unknown storage mode {mode}")
    f = mode & 15
    return (bf, bf, f32 if f & ANYPREC_M_FP32 else bf, f32 if f & ANYPREC_V_FP32 else bf,
            None if f & ANYPREC_NO_KAHAN else (f32 if f & ANYPREC_C_FP32 else bf))


class Plan:
    """A plan over lists of torch CUDA tensors (one list per buffer kind).

    bf16 Kahan mode: params, exp_avg, exp_avg_sq, aux (= compensation) bf16.
    Mixed mode: params (= fp32 master), exp_avg, exp_avg_sq fp32; aux = bf16
    param out.  Remainder mode: params bf16, exp_avg, exp_avg_sq fp32, aux =
    int16 remainder of the fp32 master.  Any-precision modes: as
    ``buffer_dtypes(mode)``.  grads are bf16 in all modes.  The tensors must stay alive and in
    place for the plan's lifetime (the plan holds references to them).
    """

    def __init__(self, params, grads, exp_avgs, exp_avg_sqs, auxs, mode: int,
                 norm: bool = False, fuse: bool = True):
        import torch
        if auxs is None:
            auxs = [None] * len(list(params))
        lists = [list(x) for x in (params, grads, exp_avgs, exp_avg_sqs, auxs)]
        n = len(lists[0])
        if any(len(x) != n for x in lists):
            raise ValueError("tensor lists differ in length")
        want = buffer_dtypes(mode)
        entries = []
        for k in range(n):
            ts = [x[k] for x in lists]
            numel = ts[0].numel()
            for j, (t, dt) in enumerate(zip(ts, want)):
                if dt is None:       # a buffer the mode does not use
                    continue
                # gradients may live in pinned host memory (read over the
                # CPU-GPU link); everything else on the device
                where_ok = t.is_cuda or (j == 1 and t.is_pinned())
                if not where_ok or t.dtype != dt or not t.is_contiguous() or t.numel() != numel:
                    raise TypeError(f"tensor {k}: want contiguous CUDA {dt} of {numel} elements"
                                    + (" (or pinned host memory)" if j == 1 else ""))
            entries.append(adamw_tensor_t(*(t.data_ptr() if t is not None else None for t in ts),
                                          numel))
        self._keep = lists
        self.mode = mode
        dev = lists[0][0].device if n else torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(dev):
            self.handle = adamw_plan_create(entries, mode, (PLAN_NORM if norm else 0)
                                            | (0 if fuse else PLAN_NO_FUSE))
        self.device = dev
        self.info = adamw_plan_get_info(self.handle)
        self.last_nonfinite = None

    def step(self, hp: adamw_hparams_t, step: int, grad_norm=None, nonfinite=None,
             stream=None) -> None:
        """One step at t = ``step``.  A clipped step (hp.max_grad_norm > 0)
        needs a non-finite flag; without ``nonfinite`` it goes to the plan's
        own int32 device tensor ``last_nonfinite`` (1: the step was skipped,
        so the caller must pass the same ``step`` again)."""
        import torch
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        if nonfinite is None and hp.max_grad_norm > 0:
            if self.last_nonfinite is None:
                self.last_nonfinite = torch.zeros(1, dtype=torch.int32, device=self.device)
            nonfinite = self.last_nonfinite
        adamw_step(self.handle, hp, step,
                   grad_norm.data_ptr() if grad_norm is not None else 0,
                   nonfinite.data_ptr() if nonfinite is not None else 0,
                   st.cuda_stream)

    def step_device(self, d_hp, d_step, flags: int = 0, grad_norm=None, nonfinite=None,
                    stream=None) -> None:
        """d_hp: CUDA uint8 tensor holding one adamw_hparams_t (see
        ``device_hparams``); d_step: CUDA int64 tensor, the applied-step count."""
        import torch
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        adamw_step_device(self.handle, d_hp.data_ptr(), d_step.data_ptr(), flags,
                          grad_norm.data_ptr() if grad_norm is not None else 0,
                          nonfinite.data_ptr() if nonfinite is not None else 0, st.cuda_stream)

    def grad_norm(self, grad_norm=None, nonfinite=None, stream=None) -> None:
        import torch
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        adamw_grad_norm(self.handle, grad_norm.data_ptr() if grad_norm is not None else 0,
                        nonfinite.data_ptr() if nonfinite is not None else 0, st.cuda_stream)

    def close(self) -> None:
        if getattr(self, "handle", None):
            adamw_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def device_hparams(hp: adamw_hparams_t, device="cuda"):
    """An adamw_hparams_t as a CUDA uint8 tensor, for adamw_step_device."""
    import torch
    raw = bytes(hp)
    return torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device)
