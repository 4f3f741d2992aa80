"""Host logic of bench.py that needs no GPU: the over-ranks aggregation of a
multi-process run (two gloo ranks on CPU) and the ncu-traffic lookup that is
only trusted while the kernel's sources match the capture."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, units, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, rate = bench.job_rate(ms_by_rank[rank], units, world, dist, torch.device("cpu"))
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_job_rate_single_process():
    ms, rate = bench.job_rate(2.0, 1000, 1)
    assert ms == 2.0 and rate == pytest.approx(1000 / 2e-3)


def test_job_rate_two_gloo_ranks_takes_the_slowest_rank():
    world, units = 2, 4096
    ms_by_rank = [1.5, 2.5]
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, ms_by_rank, units, out), nprocs=world, join=True)
        got = dict(out)
    for r in range(world):
        ms, rate = got[r]
        assert ms == pytest.approx(2.5)                       # max over ranks
        assert rate == pytest.approx(world * units / 2.5e-3)  # all ranks' units / slowest time


def _fake_root(tmp_path, record_sha):
    csrc = tmp_path / "linear_token_mixer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in set(n for v in bench.KERNEL_SOURCES.values() for n in v):
        (csrc / name).write_text("// source of %s\n" % name)
    (tmp_path / "profiles").mkdir()
    rec = {"chunked prefill/falcon1_bf16": {"sources_sha256": record_sha,
                                            "dram_bytes_per_launch": 123456}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    return tmp_path


def test_stored_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    root = _fake_root(tmp_path, "0" * 64)
    monkeypatch.setattr(bench, "ROOT", str(root))
    # sources changed since the capture: no traffic figure
    assert bench.stored_traffic("chunked prefill", "falcon1_bf16") is None
    rec = json.loads((root / "profiles" / "traffic.json").read_text())
    rec["chunked prefill/falcon1_bf16"]["sources_sha256"] = bench.sources_sha256("chunked prefill")
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.stored_traffic("chunked prefill", "falcon1_bf16") == 123456
    # another workload has no record
    assert bench.stored_traffic("chunked prefill", "linattn_bf16") is None
    # editing a kernel source invalidates the record
    (root / "linear_token_mixer_gb300" / "csrc" / "fw_sm100.cuh").write_text("// edited\n")
    assert bench.stored_traffic("chunked prefill", "falcon1_bf16") is None


def test_alu_roofline_flop_counts_per_head_token():
    # multiply-adds per head-token by the write's definition: residual reads
    # S^T x_j (one per pair; none for the inner-product forms), the rank-W write,
    # the decay of S and the read S^T q
    from linear_token_mixer_gb300 import inputs as I
    d = 128
    per = lambda name, **kw: bench.window_flops(I.WORKLOADS[name].with_shape(B=1, H=1, T=1, **kw)) / (2 * d * d)
    assert per("falcon3_bf16") == 4 + 4 + 2
    assert per("falcon3a_bf16") == 4 + 2
    assert per("falcon2_bf16") == 1 + 1 + 2     # a step per value column: W = 1
    assert per("falcon2_bf16", mode="falcon2a") == 1 + 2


def test_reference_arm_line(capsys, monkeypatch):
    # the reference arm times the oracle on the host and prints one line with the
    # GPU arm's metric, unit and config, an e2e object without host copies, and
    # a cpu_baseline describing the run; ranks other than 0 print nothing
    import argparse
    args = argparse.Namespace(workload=bench.HEADLINE, gpus=1, steps=1, warmup=0)
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    from linear_token_mixer_gb300 import inputs as I
    w = I.WORKLOADS[bench.HEADLINE]
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["config"] == bench.headline_config(w, 1)
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("name", ["falcon1_bf16", "falcon1a_bf16", "falcon2_bf16", "linattn_bf16"])
def test_reference_arm_runs_the_oracle_of_the_workload_mode(capsys, monkeypatch, name):
    # --impl reference with any headline workload times the oracle entry of that
    # workload's own mode (not another mode's), and says which one ran
    import argparse
    import oracle
    from linear_token_mixer_gb300 import inputs as I
    calls = []
    for fn in ("falcon1", "falcon2", "falcon3", "linattn"):
        real = getattr(oracle, fn)
        monkeypatch.setattr(oracle, fn, (lambda f, r: lambda *a, **k: (calls.append((f, k.get("inner", False))), r(*a, **k))[1])(fn, real))
    w = I.WORKLOADS[name]
    monkeypatch.setattr(I, "WORKLOADS", dict(I.WORKLOADS, **{name: w.with_shape(T=64)}))
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(argparse.Namespace(workload=name, gpus=1, steps=1, warmup=0))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["cpu_baseline"]["oracle"] == w.mode
    fam = {"falcon1": "falcon1", "falcon1a": "falcon1", "falcon2": "falcon2",
           "falcon2a": "falcon2", "linattn": "linattn"}[w.mode]
    assert calls and all(c == (fam, w.mode.endswith("a")) for c in calls), calls
    assert line["config"]["mode"] == w.mode


def test_headline_kernel_labels_follow_the_dispatch():
    from linear_token_mixer_gb300 import inputs as I
    W = I.WORKLOADS
    assert bench.prefill_kernel(W["falcon1_bf16"]) == "chunked prefill"
    assert bench.prefill_kernel(W["linattn_bf16"]) == "chunked prefill"
    assert bench.prefill_kernel(W["falcon1_fp32"]) == "recurrent (SIMT)"
    # few long chains: two segments at once (32 chains, T = 32768, 152 SMs)
    assert bench.prefill_kernel(W["falcon1_long"]) == "chunked prefill (two segments)"
    assert bench.prefill_kernel(W["falcon1_long"], sms=64) == "chunked prefill"
    assert bench.prefill_kernel(W["falcon1_bf16"].with_shape(phi="elu1")) == "recurrent (SIMT)"
    f2 = W["falcon2_bf16"]
    assert bench.prefill_kernel(f2) == "chunked prefill (per channel)"
    assert bench.prefill_kernel(f2.with_shape(phi="elu1")) == "window prefill (SIMT)"
    assert bench.prefill_kernel(f2.with_shape(dtype=torch.float32)) == "window prefill (SIMT)"
    # the per-channel kernel's tcgen05 products: Gram, X S0, Q S0, state update
    ht = f2.B * f2.H * f2.T
    assert bench.matmul_flops_prefill(f2) == ht * (4 * 64 * 128 + 6 * 128 * 128)
    assert bench.matmul_flops_prefill(f2.with_shape(mode="falcon2a")) == ht * (4 * 64 * 128 + 4 * 128 * 128)
    # no tensor-core FLOPs are claimed for a launch that runs no tensor-core kernel
    assert bench.matmul_flops_prefill(f2.with_shape(phi="elu1")) is None
    assert bench.matmul_flops_prefill(W["falcon1_fp32"]) is None
    assert bench.matmul_flops_prefill(W["falcon1_bf16"]) > 0
    assert "falcon3_bf16" not in bench.PREFILL_WORKLOADS
