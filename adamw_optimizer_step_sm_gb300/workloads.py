"""Seeded synthetic workloads for the AdamW step: tensor-list shapes and the
random parameter / gradient recipe.

This module holds no optimizer arithmetic.  It only draws numbers and lays out
tensors, so the CUDA path and the CPU oracle can be fed identical bytes.

Shapes
  * OPT-125m / OPT-1.3b tensor lists, the two models trained in
    "[pure bf16 training] w/ AnyPrecisionAdamW and Kahan summation"
    (transformers PR #21312), sections "opt-125m / bf16-pure training from
    scratch" and "opt-1.3b / bf16-pure training from scratch".  Their weights
    are not available; only the public model shapes are used (hidden 768 / 2048,
    12 / 24 layers, FFN 3072 / 8192, vocab 50272, 2050 learned positions).
  * One 13,850,000-element shard = a quarter of the 55.4M-parameter BERT of
    "Distributed optimizer support for BERT" (NeMo PR #5305), memory-savings
    estimate under the 4xA40 table, at data-parallel size 4.

Values
  * params ~ N(0, 0.02), LayerNorm weights 1 and biases 0;
  * grads ~ N(0, sigma), fresh for every step from (seed, step); optionally
    1 % of entries multiplied by 100 (a heavy tail);
  * exp_avg = exp_avg_sq = compensation = 0 at step 0.
Random draws use torch generators on the device the tensors live on; parity
tests copy the drawn bytes to the host for the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED = 42   # the run recipes on the pages pass --seed 42

MODE_BF16_KAHAN = 0
MODE_MIXED = 1
MODE_REMAINDER = 2
MODE_BF16_PLAIN = 3
MODE_BF16_KAHAN_V32 = 4

# torch dtypes of (param, exp_avg, exp_avg_sq, aux) per mode (None: unused)
MODE_DTYPES = {
    MODE_BF16_KAHAN: (torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.bfloat16),
    MODE_MIXED: (torch.float32, torch.float32, torch.float32, torch.bfloat16),
    MODE_REMAINDER: (torch.bfloat16, torch.float32, torch.float32, torch.int16),
    MODE_BF16_PLAIN: (torch.bfloat16, torch.bfloat16, torch.bfloat16, None),
    MODE_BF16_KAHAN_V32: (torch.bfloat16, torch.bfloat16, torch.float32, torch.bfloat16),
}

# AnyPrecisionAdamW storage modes: MODE_ANYPREC + flags (1: fp32 exp_avg,
# 2: fp32 exp_avg_sq, 4: fp32 compensation, 8: no compensation).
MODE_ANYPREC = 16
ANYPREC_MODES = tuple(MODE_ANYPREC | f for f in range(16) if (f & 12) != 12)
for _m in ANYPREC_MODES:
    _f = _m & 15
    MODE_DTYPES[_m] = (torch.bfloat16,
                       torch.float32 if _f & 1 else torch.bfloat16,
                       torch.float32 if _f & 2 else torch.bfloat16,
                       None if _f & 8 else (torch.float32 if _f & 4 else torch.bfloat16))
del _m, _f


@dataclass(frozen=True)
class TensorSpec:
    name: str
    numel: int
    kind: str = "weight"   # "weight" | "bias" | "ln_weight" | "ln_bias"


def opt_tensor_list(hidden: int, layers: int, ffn: int, vocab: int = 50272,
                    positions: int = 2050) -> list[TensorSpec]:
    """The parameter tensors of an OPT decoder, in a fixed order:
    token embedding, position embedding, per layer (q, k, v, out_proj weights
    and biases, attention LayerNorm, fc1, fc2, final LayerNorm), and the
    decoder's final LayerNorm."""
    h = hidden
    out = [TensorSpec("embed_tokens", vocab * h), TensorSpec("embed_positions", positions * h)]
    for i in range(layers):
        pre = f"layers.{i}."
        for proj in ("q_proj", "k_proj", "v_proj", "out_proj"):
            out.append(TensorSpec(pre + proj + ".weight", h * h))
            out.append(TensorSpec(pre + proj + ".bias", h, "bias"))
        out.append(TensorSpec(pre + "self_attn_layer_norm.weight", h, "ln_weight"))
        out.append(TensorSpec(pre + "self_attn_layer_norm.bias", h, "ln_bias"))
        out.append(TensorSpec(pre + "fc1.weight", h * ffn))
        out.append(TensorSpec(pre + "fc1.bias", ffn, "bias"))
        out.append(TensorSpec(pre + "fc2.weight", ffn * h))
        out.append(TensorSpec(pre + "fc2.bias", h, "bias"))
        out.append(TensorSpec(pre + "final_layer_norm.weight", h, "ln_weight"))
        out.append(TensorSpec(pre + "final_layer_norm.bias", h, "ln_bias"))
    out.append(TensorSpec("final_layer_norm.weight", h, "ln_weight"))
    out.append(TensorSpec("final_layer_norm.bias", h, "ln_bias"))
    return out


@dataclass(frozen=True)
class Workload:
    name: str
    mode: int
    tensors: tuple[TensorSpec, ...]
    steps: int
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    max_grad_norm: float = 0.0
    p_std: float = 0.02
    g_std: float = 1e-2
    heavy_tail: bool = False
    # (step, tensor index, element index) that receives +inf, or None
    inf_at: tuple[int, int, int] | None = None
    seed: int = SEED
    description: str = ""

    @property
    def numels(self) -> list[int]:
        return [t.numel for t in self.tensors]

    @property
    def total(self) -> int:
        return sum(self.numels)

    @property
    def n_tensors(self) -> int:
        return len(self.tensors)

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, max_grad_norm=self.max_grad_norm)


OPT_125M = tuple(opt_tensor_list(768, 12, 3072))
OPT_1_3B = tuple(opt_tensor_list(2048, 24, 8192))

WORKLOADS: dict[str, Workload] = {
    "flat1m_bf16_kahan": Workload(
        "flat1m_bf16_kahan", MODE_BF16_KAHAN, (TensorSpec("flat", 1 << 20),), 10,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        description="one flat tensor of 1,048,576 elements, pure-bf16 Kahan"),
    "bert55m_shard_mixed": Workload(
        "bert55m_shard_mixed", MODE_MIXED, (TensorSpec("shard", 13_850_000),), 20,
        lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, g_std=1e-3,
        description="one 13,850,000-element shard (55.4M / 4), fp32 master"),
    "opt125m_bf16_kahan": Workload(
        "opt125m_bf16_kahan", MODE_BF16_KAHAN, OPT_125M, 10,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        heavy_tail=True, description="OPT-125m tensor list, pure-bf16 Kahan"),
    "opt1.3b_bf16_kahan": Workload(
        "opt1.3b_bf16_kahan", MODE_BF16_KAHAN, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        heavy_tail=True, description="OPT-1.3b tensor list, pure-bf16 Kahan"),
    "opt1.3b_mixed_clip": Workload(
        "opt1.3b_mixed_clip", MODE_MIXED, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
        max_grad_norm=1.0, g_std=1e-2, inf_at=(3, 200, 12345),
        description="OPT-1.3b tensor list, fp32 master + global-norm clip 1.0, "
                    "+inf injected at step 3"),
    "bert55m_shard_mixed_clip": Workload(
        "bert55m_shard_mixed_clip", MODE_MIXED, (TensorSpec("shard", 13_850_000),), 20,
        lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, g_std=1e-3,
        max_grad_norm=1.0, inf_at=(7, 0, 4242),
        description="one 13,850,000-element shard, fp32 master, global-norm clip 1.0 "
                    "(one fused launch per step), +inf injected at step 7"),
    "bert55m_shard_remainder": Workload(
        "bert55m_shard_remainder", MODE_REMAINDER, (TensorSpec("shard", 13_850_000),), 20,
        lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, g_std=1e-3,
        description="one 13,850,000-element shard, fp32 master held as bf16 param + "
                    "16-bit remainder"),
    "opt1.3b_remainder_clip": Workload(
        "opt1.3b_remainder_clip", MODE_REMAINDER, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
        max_grad_norm=1.0, g_std=1e-2, inf_at=(3, 200, 12345),
        description="OPT-1.3b tensor list, bf16 param + 16-bit remainder master, "
                    "global-norm clip 1.0, +inf injected at step 3"),
    "opt1.3b_bf16_plain": Workload(
        "opt1.3b_bf16_plain", MODE_BF16_PLAIN, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        heavy_tail=True, description="OPT-1.3b tensor list, pure bf16 without Kahan "
                                     "compensation"),
    "opt1.3b_bf16_kahan_v32": Workload(
        "opt1.3b_bf16_kahan_v32", MODE_BF16_KAHAN_V32, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        heavy_tail=True, description="OPT-1.3b tensor list, bf16 Kahan with fp32 variance"),
    "opt1.3b_anyprec_fp32_state": Workload(
        "opt1.3b_anyprec_fp32_state", MODE_ANYPREC | 7, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        heavy_tail=True, description="OPT-1.3b tensor list, bf16 param with fp32 momentum, "
                                     "variance and Kahan compensation"),
    "opt1.3b_anyprec_m32": Workload(
        "opt1.3b_anyprec_m32", MODE_ANYPREC | 1, OPT_1_3B, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, g_std=1e-2,
        heavy_tail=True, description="OPT-1.3b tensor list, bf16 Kahan with fp32 momentum"),
    # profiling-size case of the clipped mixed step (2 GB of state, > L2)
    "opt125m_mixed_clip": Workload(
        "opt125m_mixed_clip", MODE_MIXED, OPT_125M, 5,
        lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
        max_grad_norm=1.0, g_std=1e-2, heavy_tail=True,
        description="OPT-125m tensor list, fp32 master + global-norm clip 1.0"),
}


# ------------------------------------------------------------------ drawing --

def _gen(device, *key: int) -> torch.Generator:
    """A generator on ``device`` seeded from an integer key tuple."""
    s = 0
    for k in key:
        s = (s * 1_000_003 + int(k) + 1) % (1 << 62)
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def _draw_normal(n: int, std: float, gen: torch.Generator, device,
                 chunk: int = 1 << 28) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e].normal_(0.0, std, generator=gen)
    return out


def tensor_offsets(numels, align_elems: int = 8) -> tuple[list[int], int]:
    """Offsets of the tensors inside one flat buffer, each rounded up to
    ``align_elems`` elements (16 bytes for bf16 at 8), and the buffer length."""
    offs, o = [], 0
    for n in numels:
        o = (o + align_elems - 1) // align_elems * align_elems
        offs.append(o)
        o += n
    return offs, o


@dataclass
class State:
    """Flat device buffers of one workload plus per-tensor views."""
    workload: Workload
    param: torch.Tensor        # bf16 (mode 0) or fp32 master (mode 1)
    exp_avg: torch.Tensor
    exp_avg_sq: torch.Tensor
    aux: torch.Tensor | None   # bf16 compensation / bf16 param out / int16 remainder
    offsets: list[int] = field(default_factory=list)

    def views(self, flat: torch.Tensor | None) -> list:
        if flat is None:
            return [None] * len(self.offsets)
        return [flat[o:o + n] for o, n in zip(self.offsets, self.workload.numels)]


def make_state(w: Workload, device="cpu", align_elems: int = 8, skew: int = 0,
               tail_pad: int = 0) -> State:
    """Initial optimizer state: params drawn, moments and aux zero.  Tensors sit
    in one flat buffer per kind at offsets rounded to ``align_elems`` elements,
    the first one ``skew`` elements in (ragged layouts use 1 and a skew), with
    ``tail_pad`` spare elements after the last one."""
    offs, length = tensor_offsets(w.numels, align_elems)
    offs = [o + skew for o in offs]
    length += skew + tail_pad
    p32 = torch.zeros(length, dtype=torch.float32, device=device)
    gen = _gen(device, w.seed, 1)
    for spec, o in zip(w.tensors, offs):
        dst = p32[o:o + spec.numel]
        if spec.kind == "ln_weight":
            dst.fill_(1.0)
        elif spec.kind == "ln_bias":
            dst.zero_()
        else:
            dst.copy_(_draw_normal(spec.numel, w.p_std, gen, device))
    pdt, mdt, vdt, adt = MODE_DTYPES[w.mode]
    # remainder mode starts from bf16-exact masters: the remainder is zero
    param = p32.to(pdt) if pdt != torch.float32 else p32
    del p32
    z = lambda dt: torch.zeros(length, dtype=dt, device=device) if dt is not None else None
    return State(w, param, z(mdt), z(vdt), z(adt), offs)


def make_grad(w: Workload, step: int, device="cpu", offsets: list[int] | None = None,
              length: int | None = None) -> torch.Tensor:
    """The flat bf16 gradient of ``step`` (1-based), drawn from (seed, step),
    laid out like ``make_state`` (default layout, or the given offsets)."""
    if offsets is None:
        offsets, length = tensor_offsets(w.numels)
    elif length is None:
        length = max((o + n for o, n in zip(offsets, w.numels)), default=0)
    gen = _gen(device, w.seed, 2, step)
    g = _draw_normal(length, w.g_std, gen, device)
    if w.heavy_tail:
        chunk = 1 << 28
        for s in range(0, length, chunk):
            e = min(length, s + chunk)
            u = torch.rand(e - s, generator=gen, device=device)
            g[s:e] = torch.where(u < 0.01, g[s:e] * 100.0, g[s:e])
            del u
    gb = g.to(torch.bfloat16)
    del g
    # zero what lies between tensors so it is never "data"
    mask = torch.ones(length, dtype=torch.bool, device=device)
    for o, n in zip(offsets, w.numels):
        mask[o:o + n] = False
    gb[mask] = 0
    if w.inf_at is not None and w.inf_at[0] == step:
        _, k, e = w.inf_at
        gb[offsets[k] + e] = float("inf")
    return gb


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's bit patterns as a numpy uint16 array (host copy)."""
    import numpy as np
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_array(t: torch.Tensor):
    return t.detach().contiguous().cpu().numpy()


def truncated(w: Workload, n_elems: int) -> Workload:
    """The first ``n_elems`` elements of a workload's tensor list (the last
    tensor cut short), same recipe: a bounded sample of the same workload."""
    out, left = [], n_elems
    for t in w.tensors:
        if left <= 0:
            break
        out.append(TensorSpec(t.name, min(t.numel, left), t.kind))
        left -= out[-1].numel
    from dataclasses import replace
    return replace(w, name=f"{w.name}[:{n_elems}]", tensors=tuple(out), inf_at=None)
