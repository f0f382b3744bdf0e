"""CPU oracle for the AdamW optimizer step (plain C, loaded with ctypes).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline leg are the only callers.  The CUDA library never imports, links or
runs anything here, and this package imports nothing from the CUDA library.

The arithmetic lives in ``adamw_ref.c`` (decoupled-weight-decay Adam with bias
correction, bf16 Kahan mode and fp32-master mixed mode, global-norm clipping);
this module only compiles it with ``gcc -ffp-contract=off`` and marshals numpy
arrays into it.  bf16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "adamw_ref.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle_adamw.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def compile_source(src_path: str, out_path: str) -> str:
    """Compile one oracle C source into a shared library at ``out_path``."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``adamw_ref.c`` when the library is missing or older."""
    if (force or not os.path.exists(LIB_PATH)
            or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE)):
        compile_source(SOURCE, LIB_PATH)
    return LIB_PATH


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float),
                ("max_grad_norm", ctypes.c_float)]


class TensorEntry(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("aux", ctypes.c_void_p), ("numel", ctypes.c_int64)]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(a: np.ndarray, dtype, n: int | None = None):
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"oracle wants contiguous {np.dtype(dtype)}, got {a.dtype}")
    if n is not None and a.size != n:
        raise ValueError(f"size {a.size} != {n}")


@dataclass
class Oracle:
    """Numpy-level wrappers around one loaded oracle library."""
    lib: ctypes.CDLL

    def __post_init__(self):
        L = self.lib
        vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
        hp = ctypes.POINTER(Hparams)
        L.oracle_f32_to_bf16.argtypes = [vp, vp, i64]
        L.oracle_bf16_to_f32.argtypes = [vp, vp, i64]
        L.oracle_step_scalars.argtypes = [hp, i64, vp]
        L.oracle_adamw_bf16_kahan.argtypes = [vp, vp, vp, vp, vp, i64, hp, i64, f32]
        L.oracle_adamw_bf16_plain.argtypes = [vp, vp, vp, vp, i64, hp, i64, f32]
        L.oracle_adamw_mixed.argtypes = [vp, vp, vp, vp, vp, i64, hp, i64, f32]
        L.oracle_adamw_remainder.argtypes = [vp, vp, vp, vp, vp, i64, hp, i64, f32]
        L.oracle_adamw_bf16_kahan_v32.argtypes = [vp, vp, vp, vp, vp, i64, hp, i64, f32]
        L.oracle_adamw_anyprec.argtypes = [vp, vp, vp, vp, vp, i64, ctypes.c_int32, hp, i64,
                                           f32]
        L.oracle_adamw_anyprec.restype = ctypes.c_int32
        L.oracle_lr_linear_warmup.argtypes = [f32, i64, i64, i64]
        L.oracle_lr_linear_warmup.restype = f32
        L.oracle_split_master.argtypes = [vp, vp, vp, i64]
        L.oracle_join_master.argtypes = [vp, vp, vp, i64]
        L.oracle_grad_sumsq.argtypes = [vp, i64, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_int32)]  # acc[2]
        L.oracle_clip_coef.argtypes = [ctypes.c_double, f32,
                                       ctypes.POINTER(ctypes.c_double)]
        L.oracle_clip_coef.restype = f32
        L.oracle_adamw_list_step.argtypes = [ctypes.POINTER(TensorEntry),
                                             ctypes.c_int32, ctypes.c_int32, hp,
                                             i64, ctypes.POINTER(ctypes.c_double)]
        L.oracle_adamw_list_step.restype = ctypes.c_int32

    # -- bf16 conversion -----------------------------------------------------
    def f32_to_bf16(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_bf16(_ptr(x), _ptr(out), x.size)
        return out

    def bf16_to_f32(self, h: np.ndarray) -> np.ndarray:
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float32)
        self.lib.oracle_bf16_to_f32(_ptr(h), _ptr(out), h.size)
        return out

    def step_scalars(self, hp: Hparams, t: int) -> np.ndarray:
        out = np.empty(5, dtype=np.float32)
        self.lib.oracle_step_scalars(ctypes.byref(hp), t, _ptr(out))
        return out

    # -- per-tensor steps (arrays updated in place) ----------------------------
    def bf16_kahan(self, p, g, m, v, c, hp: Hparams, t: int, coef: float = 1.0):
        n = p.size
        for a in (p, g, m, v, c):
            _check(a, np.uint16, n)
        self.lib.oracle_adamw_bf16_kahan(_ptr(p), _ptr(g), _ptr(m), _ptr(v),
                                         _ptr(c), n, ctypes.byref(hp), t, coef)

    def bf16_plain(self, p, g, m, v, hp: Hparams, t: int, coef: float = 1.0):
        n = p.size
        for a in (p, g, m, v):
            _check(a, np.uint16, n)
        self.lib.oracle_adamw_bf16_plain(_ptr(p), _ptr(g), _ptr(m), _ptr(v), n,
                                         ctypes.byref(hp), t, coef)

    def mixed(self, master, g, m, v, p_out, hp: Hparams, t: int, coef: float = 1.0):
        n = master.size
        for a, dt in ((master, np.float32), (g, np.uint16), (m, np.float32),
                      (v, np.float32), (p_out, np.uint16)):
            _check(a, dt, n)
        self.lib.oracle_adamw_mixed(_ptr(master), _ptr(g), _ptr(m), _ptr(v),
                                    _ptr(p_out), n, ctypes.byref(hp), t, coef)

    def remainder(self, p16, g, m, v, r16, hp: Hparams, t: int, coef: float = 1.0):
        n = p16.size
        for a, dt in ((p16, np.uint16), (g, np.uint16), (m, np.float32), (v, np.float32),
                      (r16, np.int16)):
            _check(a, dt, n)
        self.lib.oracle_adamw_remainder(_ptr(p16), _ptr(g), _ptr(m), _ptr(v), _ptr(r16), n,
                                        ctypes.byref(hp), t, coef)

    def bf16_kahan_v32(self, p, g, m, v, c, hp: Hparams, t: int, coef: float = 1.0):
        n = p.size
        for a, dt in ((p, np.uint16), (g, np.uint16), (m, np.uint16), (v, np.float32),
                      (c, np.uint16)):
            _check(a, dt, n)
        self.lib.oracle_adamw_bf16_kahan_v32(_ptr(p), _ptr(g), _ptr(m), _ptr(v), _ptr(c), n,
                                             ctypes.byref(hp), t, coef)

    def anyprec(self, p, g, m, v, c, flags: int, hp: Hparams, t: int, coef: float = 1.0):
        """AnyPrecisionAdamW step; ``flags`` as oracle_adamw_anyprec (1: fp32
        exp_avg, 2: fp32 exp_avg_sq, 4: fp32 compensation, 8: no Kahan, c is
        then None)."""
        n = p.size
        dm, dv, dc = anyprec_dtypes(flags)
        for a, dt in ((p, np.uint16), (g, np.uint16), (m, dm), (v, dv)):
            _check(a, dt, n)
        if dc is not None:
            _check(c, dc, n)
        rc = self.lib.oracle_adamw_anyprec(_ptr(p), _ptr(g), _ptr(m), _ptr(v),
                                           _ptr(c) if dc is not None else None, n, flags,
                                           ctypes.byref(hp), t, coef)
        if rc != 0:
            raise ValueError(f"invalid any-precision flags {flags}")

    def lr_linear_warmup(self, base_lr: float, t: int, warmup: int, total: int) -> float:
        return float(np.float32(self.lib.oracle_lr_linear_warmup(base_lr, t, warmup, total)))

    def split_master(self, x: np.ndarray):
        x = np.ascontiguousarray(x, dtype=np.float32)
        p16 = np.empty(x.shape, np.uint16)
        r16 = np.empty(x.shape, np.int16)
        self.lib.oracle_split_master(_ptr(x), _ptr(p16), _ptr(r16), x.size)
        return p16, r16

    def join_master(self, p16: np.ndarray, r16: np.ndarray) -> np.ndarray:
        p16 = np.ascontiguousarray(p16, dtype=np.uint16)
        r16 = np.ascontiguousarray(r16, dtype=np.int16)
        out = np.empty(p16.shape, np.float32)
        self.lib.oracle_join_master(_ptr(p16), _ptr(r16), _ptr(out), p16.size)
        return out

    # -- norm ------------------------------------------------------------------
    def grad_sumsq(self, grads) -> tuple[float, bool]:
        """Sum of squares over the tensors in order (compensated fp64) and
        whether any element is non-finite."""
        acc = (ctypes.c_double * 2)(0.0, 0.0)
        bad = ctypes.c_int32(0)
        for g in grads:
            _check(g, np.uint16)
            self.lib.oracle_grad_sumsq(_ptr(g), g.size, acc, ctypes.byref(bad))
        return acc[0] + acc[1], bool(bad.value)

    def clip_coef(self, sumsq: float, max_norm: float) -> tuple[float, float]:
        norm = ctypes.c_double(0.0)
        coef = self.lib.oracle_clip_coef(sumsq, max_norm, ctypes.byref(norm))
        return float(np.float32(coef)), norm.value

    # -- whole list -------------------------------------------------------------
    def list_step(self, tensors, mode: int, hp: Hparams, t: int):
        """``tensors``: list of (param, grad, exp_avg, exp_avg_sq, aux) numpy
        arrays.  Returns (skipped: bool, norm: float)."""
        arr = (TensorEntry * max(1, len(tensors)))()
        u16, f32, i16 = np.uint16, np.float32, np.int16
        if mode >= ANYPREC:
            want = (u16, *anyprec_dtypes(mode - ANYPREC))
        else:
            want = {0: (u16, u16, u16, u16), 1: (f32, f32, f32, u16), 2: (u16, f32, f32, i16),
                    3: (u16, u16, u16, None), 4: (u16, u16, f32, u16)}[mode]
        for k, (p, g, m, v, a) in enumerate(tensors):
            n = g.size
            _check(p, want[0], n); _check(g, np.uint16, n); _check(m, want[1], n)
            _check(v, want[2], n)
            if want[3] is not None:
                _check(a, want[3], n)
            arr[k] = TensorEntry(p.ctypes.data, g.ctypes.data, m.ctypes.data,
                                 v.ctypes.data, a.ctypes.data if a is not None else None, n)
        norm = ctypes.c_double(0.0)
        rc = self.lib.oracle_adamw_list_step(arr, len(tensors), mode,
                                             ctypes.byref(hp), t,
                                             ctypes.byref(norm))
        if rc < 0:
            raise ValueError(f"unknown mode {mode}")
        return bool(rc), norm.value


# Mode numbers of the any-precision step: ANYPREC + flags.
ANYPREC = 16


def anyprec_dtypes(flags: int):
    """Storage types of exp_avg, exp_avg_sq and the compensation (None without
    Kahan summation) for any-precision flags."""
    if flags & ~15 or (flags & 12) == 12:
        raise ValueError(f"invalid any-precision flags {flags}")
    f32, u16 = np.float32, np.uint16
    return (f32 if flags & 1 else u16, f32 if flags & 2 else u16,
            None if flags & 8 else (f32 if flags & 4 else u16))


def load(path: str | None = None) -> Oracle:
    """Load the oracle (building it first when ``path`` is None)."""
    global _lib
    if path is not None:
        return Oracle(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = Oracle(ctypes.CDLL(build()))
        return _lib


def hparams(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
            max_grad_norm=0.0) -> Hparams:
    return Hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm)
