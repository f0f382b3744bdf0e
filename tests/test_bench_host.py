"""Host-side pieces of bench.py: byte accounting, the max-over-ranks timing
reduction on two gloo ranks (the N > 1 replica path), clock-log parsing and
the reference (CPU oracle) arm on a tiny sample."""
import json
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from adamw_optimizer_step_sm_gb300 import workloads as W


def test_bytes_per_param():
    assert bench.bytes_per_param(W.WORKLOADS["opt1.3b_bf16_kahan"]) == 18
    assert bench.bytes_per_param(W.WORKLOADS["bert55m_shard_mixed"]) == 28
    assert bench.bytes_per_param(W.WORKLOADS["opt1.3b_mixed_clip"]) == 30


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, _ = bench.dist_env()
    bench.barrier(w)
    t = bench.reduce_max(1.5 + rank, w, torch.device("cpu"))
    out[rank] = (w, r, t)
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert out[0] == (2, 0, 2.5) and out[1] == (2, 1, 2.5)


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max(3.25, 1, torch.device("cpu")) == 3.25


def test_clock_log_parsing():
    c = bench.ClockSampler(0)
    c.proc = None
    assert c.stop() is None

    class FakeProc:
        def terminate(self): pass
        def wait(self, timeout=None): return 0
        def kill(self): pass

    class FakeThread:
        def join(self, timeout=None): pass

    c.proc, c._t = FakeProc(), FakeThread()
    c.lines = ["0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1980, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 345, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    r = c.stop()
    assert r["sm_max_mhz"] == 2070 and r["sm_mhz"] == 1972.5 and r["reasons"] == ["sw_power_cap"]


def test_traffic_is_dropped_when_kernel_sources_change(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    os.makedirs(tmp_path / "adamw_optimizer_step_sm_gb300" / "csrc")
    for f in bench.KERNEL_SOURCES:
        (tmp_path / "adamw_optimizer_step_sm_gb300" / "csrc" / f).write_text("a")
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(
        {"x": {"kernel_source_hash": h, "dram_bytes_per_launch": 123}}))
    assert bench.recorded_traffic("x") == 123
    # a comment or a blank line is not a change of the code
    (tmp_path / "adamw_optimizer_step_sm_gb300" / "csrc" / bench.KERNEL_SOURCES[0]).write_text(
        "a // note\n/* block\n comment */\n")
    assert bench.recorded_traffic("x") == 123
    (tmp_path / "adamw_optimizer_step_sm_gb300" / "csrc" / bench.KERNEL_SOURCES[0]).write_text("b")
    assert bench.recorded_traffic("x") is None


def test_code_only_drops_comments_and_layout_but_keeps_literals():
    src = 'int a = 1; // one\n/* two\n lines */ const char* s = "x // y /* z */";\n  char c = \'/\';'
    assert bench._code_only(src) == 'int a = 1; const char* s = "x // y /* z */"; char c = \'/\';'
    assert bench._code_only("a+b") != bench._code_only("a-b")


def test_reference_arm_prints_one_json_line(capsys):
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1",
                "--workload", "opt125m_bf16_kahan", "--ref-sample", str(1 << 16)])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert capsys.readouterr().out.strip() == ""


def test_every_storage_mode_has_a_name_and_a_byte_count():
    for mode in list(range(5)) + list(W.ANYPREC_MODES):
        name, storage = bench.mode_name(mode)
        assert name and storage
        w = W.Workload("x", mode, (W.TensorSpec("a", 8),), 1, lr=1e-3, beta1=0.9, beta2=0.95,
                       eps=1e-8, weight_decay=0.0)
        assert 14 <= bench.bytes_per_param(w) <= 30
    assert bench.bytes_per_param(W.WORKLOADS["opt1.3b_anyprec_fp32_state"]) == 30
    assert bench.mode_name(W.MODE_ANYPREC | 9)[1] == "bf16 p/g, fp32 m, bf16 v, no compensation"


def test_mode_override_keeps_the_list_and_renames_the_workload():
    import argparse
    a = argparse.Namespace(workload="opt1.3b_bf16_kahan", mode=W.MODE_ANYPREC | 7)
    w = bench.workload_of(a)
    base = W.WORKLOADS["opt1.3b_bf16_kahan"]
    assert w.name == "opt1.3b_mode23" and w.mode == 23 and w.tensors == base.tensors
    assert w.hparams() == base.hparams() and bench.bytes_per_param(w) == 30
    assert bench.workload_of(argparse.Namespace(workload="opt1.3b_bf16_kahan", mode=None)) is base
