"""Constants the pages print, checked against the workloads and the storage
layout of the two modes.  See tests/golden/page_constants.json for citations."""
import json
import os

import torch

from adamw_optimizer_step_sm_gb300 import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


def test_recipe_hyperparameters_used_by_bf16_workloads():
    r = GOLD["run_recipe"]
    for name in ("flat1m_bf16_kahan", "opt125m_bf16_kahan", "opt1.3b_bf16_kahan"):
        w = W.WORKLOADS[name]
        assert (w.lr, w.beta1, w.beta2, w.weight_decay) == (
            r["learning_rate"], r["adam_beta1"], r["adam_beta2"], r["weight_decay"])
        assert w.seed == r["seed"] and w.mode == W.MODE_BF16_KAHAN


def _bytes_per_param(mode):
    w = W.Workload("t", mode, (W.TensorSpec("x", 64),), 1, 1e-3, 0.9, 0.95, 1e-8, 0.0)
    st = W.make_state(w)
    g = W.make_grad(w, 1)
    el = lambda t: t.element_size()
    optim = el(st.exp_avg) + el(st.exp_avg_sq) + (el(st.aux) if mode == W.MODE_BF16_KAHAN else 0)
    weights = el(st.param) + (el(st.aux) if mode == W.MODE_MIXED else 0)
    return optim, el(g), weights


def test_storage_matches_page_breakdown():
    mb = GOLD["memory_breakdown_bytes_per_param"]
    o, g, w = _bytes_per_param(W.MODE_BF16_KAHAN)
    assert (o, g, w) == (mb["bf16_pure"]["optim"], mb["bf16_pure"]["grad"], mb["bf16_pure"]["weights"])
    o, g, w = _bytes_per_param(W.MODE_MIXED)
    assert (o, g, w) == (mb["bf16_mixed"]["optim"], mb["bf16_mixed"]["grad"], mb["bf16_mixed"]["weights"])
    n13 = W.WORKLOADS["opt1.3b_bf16_kahan"].total
    assert abs(n13 * 10 / 1e9 - mb["bf16_pure"]["total_gb_at_1.3b"]) < 0.2
    assert abs(n13 * 16 / 1e9 - mb["bf16_mixed"]["total_gb_at_1.3b"]) < 0.3


def test_bert_shard_is_a_quarter_of_55_4m():
    z = GOLD["zero_saving_estimate"]
    assert W.WORKLOADS["bert55m_shard_mixed"].total * z["data_parallel_size"] == z["params"]
    saving = z["params"] * z["bytes_per_param_sharded"] * (1 - 1 / z["data_parallel_size"]) / 1e6
    assert round(saving) == z["saving_mb"] or abs(saving - z["saving_mb"]) < 1


def test_opt_shapes():
    assert W.WORKLOADS["opt125m_bf16_kahan"].total == 125_239_296
    assert W.WORKLOADS["opt125m_bf16_kahan"].n_tensors == 196
    assert W.WORKLOADS["opt1.3b_bf16_kahan"].total == 1_315_758_080
    assert W.WORKLOADS["opt1.3b_bf16_kahan"].n_tensors == 388


def test_inputs_are_seeded_and_fresh_per_step():
    w = W.WORKLOADS["flat1m_bf16_kahan"]
    a, b = W.make_grad(w, 1), W.make_grad(w, 1)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), W.make_grad(w, 2).view(torch.int16))
    s = W.make_state(w)
    assert s.param.dtype == torch.bfloat16 and float(s.param.float().std()) > 0.015
    assert float(s.exp_avg.float().abs().max()) == 0.0
