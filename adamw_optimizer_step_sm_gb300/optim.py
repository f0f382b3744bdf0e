"""``AnyPrecisionAdamW`` and ``MasterWeightAdamW``: ``torch.optim``
optimizers whose step is one call into the adamw_sm library
(``adamw_step_device``) per parameter group.  ``MasterWeightAdamW`` is the
fp32-master update (see its docstring); the rest of this note is about
``AnyPrecisionAdamW`` and holds for both where it concerns the layout and
the step.

It takes the options the pure-bf16 recipe passes to its optimizer ("[pure
bf16 training] w/ AnyPrecisionAdamW and Kahan summation", "Train from
scratch": ``--optim adamw_anyprecision --optim_args 'use_kahan_summation=true,
momentum_dtype=bfloat16, variance_dtype=bfloat16,
compensation_buffer_dtype=bfloat16'`` with ``--learning_rate 0.0002
--adam_beta1 0.9 --adam_beta2 0.95 --weight_decay 0.1``); those values are the
defaults here.  Parameters are bf16 CUDA tensors; each of the three optimizer
buffers may be bf16 or fp32, and Kahan summation on or off (the library's
``ADAMW_MODE_ANYPREC`` storage modes).  ``max_grad_norm > 0`` clips by the
global norm of the group's gradients inside the step and skips a step whose
gradients hold inf or NaN (no state written, counter not advanced);
``track_grad_norm`` reports the norm without clipping (one more read of the
gradients).

Layout: the optimizer owns one flat buffer per kind (gradient, exp_avg,
exp_avg_sq, compensation) for each group, every tensor at a 2048-element
boundary, and points each ``p.grad`` at its slice of the gradient buffer;
``zero_grad`` zeroes that buffer in place (it never sets gradients to None),
so backward passes accumulate straight into it and a step copies nothing.
A gradient found elsewhere at step time (the first step, or a ``p.grad``
assigned by the caller) is copied in once and re-pointed; so use this
optimizer's ``zero_grad`` (``Module.zero_grad`` sets the gradients to None,
and each step would then copy them in).  The step counter
and the hyperparameters live in device memory, so ``step`` never waits for
the GPU; ``last_grad_norm`` and ``last_nonfinite`` are device tensors.

Every parameter of a group is stepped on every call: a parameter whose
``p.grad`` is None is an error (a zero gradient still decays the moments and
the weight, which is not what skipping a parameter means).
"""
from __future__ import annotations

import torch

from . import adamw_sm as A

# Each tensor of a group starts at a multiple of this many elements in the
# group's flat buffers (4 KB of a bf16 stream), the boundaries the library's
# partition cuts tiles on.
_ALIGN = 2048

_DTYPES = {torch.bfloat16: False, torch.float32: True}


def storage_mode(use_kahan_summation: bool, momentum_dtype: torch.dtype,
                 variance_dtype: torch.dtype, compensation_buffer_dtype: torch.dtype) -> int:
    """The library's storage mode for AnyPrecisionAdamW's options."""
    for name, dt in (("momentum_dtype", momentum_dtype), ("variance_dtype", variance_dtype),
                     ("compensation_buffer_dtype", compensation_buffer_dtype)):
        if dt not in _DTYPES:
            raise ValueError(f"{name} must be torch.bfloat16 or torch.float32, not {dt}")
    flags = (A.ANYPREC_M_FP32 if _DTYPES[momentum_dtype] else 0) \
        | (A.ANYPREC_V_FP32 if _DTYPES[variance_dtype] else 0)
    if use_kahan_summation:
        flags |= A.ANYPREC_C_FP32 if _DTYPES[compensation_buffer_dtype] else 0
    else:
        flags |= A.ANYPREC_NO_KAHAN
    return A.MODE_ANYPREC | flags


class _GroupBuffers:
    """A group's flat buffers, views, plan and device-side step state.

    The plan's param and aux streams depend on the mode: the model's bf16
    parameters and the compensation (any precision); an fp32 master the
    optimizer owns and the model's bf16 parameters as output (fp32 master);
    the model's bf16 parameters and an int16 remainder (bf16 + remainder)."""

    def __init__(self, params, mode: int):
        dts = A.buffer_dtypes(mode)
        dev = params[0].device
        numels = [p.numel() for p in params]
        offs, n = [], 0
        for k in numels:
            offs.append(n)
            n += -(-k // _ALIGN) * _ALIGN
        n = max(n, 1)
        flat = lambda dt: None if dt is None else torch.zeros(n, dtype=dt, device=dev)
        view = lambda buf, p, o: None if buf is None else buf[o:o + p.numel()].view(p.shape)
        self.grad, self.exp_avg, self.exp_avg_sq = flat(torch.bfloat16), flat(dts[2]), flat(dts[3])
        self.grads = [view(self.grad, p, o) for p, o in zip(params, offs)]
        self.exp_avgs = [view(self.exp_avg, p, o) for p, o in zip(params, offs)]
        self.exp_avg_sqs = [view(self.exp_avg_sq, p, o) for p, o in zip(params, offs)]
        self.master, self.masters = None, [None] * len(params)
        self.comp, self.comps = None, [None] * len(params)
        if mode == A.MODE_MIXED_FP32_MASTER:
            # the fp32 master starts as the model's bf16 values, exactly
            self.master = flat(torch.float32)
            self.masters = [view(self.master, p, o) for p, o in zip(params, offs)]
            for m, p in zip(self.masters, params):
                m.copy_(p.detach())
            plan_p, plan_aux = self.masters, list(params)
        elif mode == A.MODE_MIXED_BF16_REMAINDER:
            # remainder 0: the master equals the model's bf16 values
            self.comp = flat(torch.int16)
            self.comps = [view(self.comp, p, o) for p, o in zip(params, offs)]
            plan_p, plan_aux = list(params), self.comps
        else:
            self.comp = flat(dts[4])
            self.comps = [view(self.comp, p, o) for p, o in zip(params, offs)]
            plan_p, plan_aux = list(params), (self.comps if self.comp is not None else None)
        self.plan = A.Plan(plan_p, self.grads, self.exp_avgs, self.exp_avg_sqs, plan_aux, mode,
                           norm=True)
        # the version counter of each model parameter when its master was
        # last made to agree with it (the library's own writes to the
        # parameter do not move the counter; a load or an in-place op does)
        self.versions = [p._version for p in params]
        self.step = torch.zeros(1, dtype=torch.int64, device=dev)
        self.grad_norm = torch.zeros(1, dtype=torch.float64, device=dev)
        self.nonfinite = torch.zeros(1, dtype=torch.int32, device=dev)
        self.d_hp = torch.zeros(len(bytes(A.hparams())), dtype=torch.uint8, device=dev)
        self.hp_key = None


class _FlatAdamW(torch.optim.Optimizer):
    """The shared machinery: flat buffers per group, one device-resident
    library step per group, checkpoints into the optimizer's own buffers."""
    _aux_name = "compensation"

    def __init__(self, params, mode: int, lr: float, betas, eps: float, weight_decay: float,
                 max_grad_norm: float, track_grad_norm: bool):
        if not lr >= 0.0 or not eps > 0.0 or not weight_decay >= 0.0:
            raise ValueError("want lr >= 0, eps > 0 and weight_decay >= 0")
        if not (0.0 <= betas[0] < 1.0 and 0.0 <= betas[1] < 1.0):
            raise ValueError("want betas in [0, 1)")
        self.mode = mode
        self.track_grad_norm = track_grad_norm
        defaults = dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                        max_grad_norm=max_grad_norm)
        self._buffers: dict[int, _GroupBuffers] = {}
        super().__init__(params, defaults)
        for group in self.param_groups:
            self._buffers_of(group)

    # -- set-up -------------------------------------------------------------
    def _buffers_of(self, group) -> _GroupBuffers:
        key = id(group)
        b = self._buffers.get(key)
        if b is None:
            params = group["params"]
            if not params:
                raise ValueError("empty parameter group")
            dev = params[0].device
            for p in params:
                if not p.is_cuda or p.dtype != torch.bfloat16 or not p.is_contiguous() \
                        or p.device != dev:
                    raise TypeError(f"{type(self).__name__} steps contiguous bf16 CUDA "
                                    "parameters of one device")
            with torch.cuda.device(dev):
                b = _GroupBuffers(params, self.mode)
            for k, (p, g) in enumerate(zip(params, b.grads)):
                if p.grad is not None:
                    g.copy_(p.grad)
                p.grad = g
                st = self.state[p]
                st["exp_avg"] = b.exp_avgs[k]
                st["exp_avg_sq"] = b.exp_avg_sqs[k]
                if b.master is not None:
                    st["master"] = b.masters[k]
                if b.comp is not None:
                    st[self._aux_name] = b.comps[k]
                st["step"] = b.step
            self._buffers[key] = b
        return b

    def add_param_group(self, param_group):
        super().add_param_group(param_group)
        if hasattr(self, "_buffers"):
            self._buffers_of(self.param_groups[-1])

    # -- the master copy (MasterWeightAdamW) ----------------------------------
    def _sync_master(self, b: _GroupBuffers, k: int, p, force: bool) -> None:
        """Makes parameter k's master agree with the model parameter p again.
        fp32 master: kept when p is its round-to-nearest-even bf16 value
        (the parameter was reloaded with what this optimizer wrote), else
        replaced by p's value.  Remainder: set to zero (the master is p)."""
        if b.master is not None:
            m = b.masters[k]
            if force or not torch.equal(m.to(torch.bfloat16), p.detach()):
                m.copy_(p.detach())
        elif self.mode == A.MODE_MIXED_BF16_REMAINDER:
            b.comps[k].zero_()
        b.versions[k] = p._version

    def _check_masters(self, group, b: _GroupBuffers) -> None:
        if self.mode not in (A.MODE_MIXED_FP32_MASTER, A.MODE_MIXED_BF16_REMAINDER):
            return
        for k, p in enumerate(group["params"]):
            if p._version != b.versions[k]:
                self._sync_master(b, k, p, force=False)

    @torch.no_grad()
    def sync_master(self) -> None:
        """Re-derives every master copy from the model's current bf16
        parameters (fp32 master = the parameter's value; remainder = 0).
        ``step`` does this by itself for a parameter changed in place (a
        model ``load_state_dict``, ``p.copy_``); call it after changing a
        parameter through ``p.data``, which ``step`` cannot see."""
        for group in self.param_groups:
            b = self._buffers_of(group)
            for k, p in enumerate(group["params"]):
                self._sync_master(b, k, p, force=True)

    # -- the step -----------------------------------------------------------
    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for group in self.param_groups:
            b = self._buffers_of(group)
            self._check_masters(group, b)
            for k, (p, g) in enumerate(zip(group["params"], b.grads)):
                if p.grad is None:
                    raise RuntimeError(f"parameter {k} of a group has no gradient; "
                                       f"{type(self).__name__} steps every parameter")
                if p.grad.data_ptr() != g.data_ptr():
                    g.copy_(p.grad)
                    p.grad = g
            beta1, beta2 = group["betas"]
            # plain floats (a scheduler may keep lr as a tensor)
            key = tuple(float(x) for x in (group["lr"], beta1, beta2, group["eps"],
                                           group["weight_decay"], group["max_grad_norm"]))
            if key != b.hp_key:
                hp = A.hparams(lr=key[0], beta1=key[1], beta2=key[2], eps=key[3],
                               weight_decay=key[4], max_grad_norm=key[5])
                # refuse out-of-range values here: on the device they would
                # only make the step skip
                A.adamw_step_scalars(hp, 1)
                host = torch.frombuffer(bytearray(bytes(hp)), dtype=torch.uint8)
                b.d_hp.copy_(host.pin_memory(), non_blocking=True)
                b.hp_key = key
            clip = group["max_grad_norm"] > 0
            norm = clip or self.track_grad_norm
            b.plan.step_device(b.d_hp, b.step, A.STEP_CLIP if clip else 0,
                               grad_norm=b.grad_norm if norm else None, nonfinite=b.nonfinite)
        return loss

    def zero_grad(self, set_to_none: bool = True):
        """Zeroes the gradient buffers in place; ``set_to_none`` is ignored
        (the gradients stay views of the optimizer's buffer)."""
        for group in self.param_groups:
            b = self._buffers_of(group)
            b.grad.zero_()
            for p, g in zip(group["params"], b.grads):
                p.grad = g

    # -- observation and checkpoints ----------------------------------------
    @property
    def last_grad_norm(self) -> list[torch.Tensor]:
        """Per group, the global gradient norm of the last step (fp64, device;
        computed when clipping or with ``track_grad_norm``)."""
        return [self._buffers_of(g).grad_norm for g in self.param_groups]

    @property
    def last_nonfinite(self) -> list[torch.Tensor]:
        """Per group, 1 when the last step's gradients held inf or NaN, else 0
        (int32, device).  With clipping on such a step wrote nothing and the
        step counter stayed; without clipping the values went through."""
        return [self._buffers_of(g).nonfinite for g in self.param_groups]

    def load_state_dict(self, state_dict):
        """Loads hyperparameters and state into this optimizer's own buffers
        (values are copied, each in its buffer's type)."""
        groups = state_dict["param_groups"]
        if len(groups) != len(self.param_groups):
            raise ValueError("loaded state has a different number of parameter groups")
        saved = state_dict["state"]
        for group, sg in zip(self.param_groups, groups):
            if len(sg["params"]) != len(group["params"]):
                raise ValueError("loaded state has a different group size")
            for name in ("lr", "betas", "eps", "weight_decay", "max_grad_norm"):
                if name in sg:
                    group[name] = tuple(sg[name]) if name == "betas" else sg[name]
            b = self._buffers_of(group)
            master_key = {A.MODE_MIXED_FP32_MASTER: "master",
                          A.MODE_MIXED_BF16_REMAINDER: "remainder"}.get(self.mode)
            for k, (idx, p) in enumerate(zip(sg["params"], group["params"])):
                s = saved.get(idx) or {}
                for name in ("exp_avg", "exp_avg_sq", "compensation", "master", "remainder"):
                    if name in s and name in self.state[p]:
                        self.state[p][name].copy_(s[name])
                if "step" in s:
                    b.step.copy_(torch.as_tensor(s["step"]).reshape(1))
                if master_key is not None:
                    if master_key in s:
                        # the loaded master is authoritative for the model's
                        # parameter as it stands now
                        b.versions[k] = p._version
                    else:
                        # a state saved without this optimizer's master (by
                        # another optimizer, or another master layout)
                        with torch.no_grad():
                            self._sync_master(b, k, p, force=True)
            b.hp_key = None


class AnyPrecisionAdamW(_FlatAdamW):
    """Pure-bf16 AdamW with the recipe's options: bf16 parameters, each of
    momentum, variance and Kahan compensation bf16 or fp32, Kahan summation
    on or off (the recipe's values are the defaults).  State per parameter:
    exp_avg, exp_avg_sq, compensation (with Kahan summation), step."""

    def __init__(self, params, lr: float = 2e-4, betas=(0.9, 0.95), eps: float = 1e-8,
                 weight_decay: float = 0.1, use_kahan_summation: bool = True,
                 momentum_dtype: torch.dtype = torch.bfloat16,
                 variance_dtype: torch.dtype = torch.bfloat16,
                 compensation_buffer_dtype: torch.dtype = torch.bfloat16,
                 max_grad_norm: float = 0.0, track_grad_norm: bool = False):
        mode = storage_mode(use_kahan_summation, momentum_dtype, variance_dtype,
                            compensation_buffer_dtype)
        super().__init__(params, mode, lr, betas, eps, weight_decay, max_grad_norm,
                         track_grad_norm)


class MasterWeightAdamW(_FlatAdamW):
    """AdamW on bf16 model parameters with an fp32 master: the update the
    distributed Adam of "Distributed optimizer support for BERT" (NeMo PR
    #5305, "Usage": distributed_fused_adam) applies to each data-parallel
    shard, here over one process's parameters.  fp32 m and v; every step
    updates the master and writes the bf16 parameters from it (round to
    nearest even).

    The master starts as the model's values when the optimizer is built.  A
    parameter changed in place afterwards (``model.load_state_dict``,
    ``p.copy_``) is seen at the next ``step`` by its version counter: the
    fp32 master is kept if the parameter is still its bf16 rounding (the
    same checkpoint loaded into both), else re-taken from the parameter; the
    remainder is reset to zero.  ``load_state_dict`` takes the saved master
    when the state has one and re-derives it from the parameter when not.
    A change made through ``p.data`` bypasses the counter: call
    ``sync_master()`` after it.

    ``master="fp32"``: the optimizer keeps an fp32 master copy (state
    ``master``), 12 B/param of optimizer state.  ``master="remainder"``: the
    master is the model's bf16 parameter plus an int16 remainder of its bit
    pattern (state ``remainder``; the "16-bit master param" of the page's
    memory estimate), 10 B/param, the same trajectory bit for bit (the bf16
    parameter is then the master rounded to nearest with ties away from
    zero).  Defaults are torch.optim.AdamW's; the pages give none for this
    update."""

    def __init__(self, params, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-8,
                 weight_decay: float = 0.01, master: str = "fp32", max_grad_norm: float = 0.0,
                 track_grad_norm: bool = False):
        modes = {"fp32": A.MODE_MIXED_FP32_MASTER, "remainder": A.MODE_MIXED_BF16_REMAINDER}
        if master not in modes:
            raise ValueError('master must be "fp32" or "remainder"')
        self._aux_name = "remainder"
        super().__init__(params, modes[master], lr, betas, eps, weight_decay, max_grad_norm,
                         track_grad_norm)
