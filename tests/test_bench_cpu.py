"""Host-side logic of bench.py without a GPU: the per-step byte/flop model, the max-over-ranks
reduction across two gloo ranks, and the reference (oracle) arm on the tiny workload."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_algorithmic_model_config2():
    wl = workloads.make(2)
    a = bench.algorithmic(wl)
    H, T = 4096, 256
    # base GEMM: one grouped launch for q/k/v (x read once) and one for o, per step
    assert bench.gemm_launch_groups(wl) == [[0, 1, 2], [3]]
    assert a["gemm_bytes"] == (4 * H * H * 2 + 2 * T * H * 2 + 4 * T * H * 2) // 2
    assert a["gemm_flops"] == 4 * 2 * T * H * H // 2
    w_bytes = 4 * H * H * 2
    # resident adapters used by the batch, A and B once per slot
    used = np.unique(wl.token_adapter)
    assert a["lora_page_bytes"] == 2 * int(wl.ranks[used].sum()) * 4 * H * 2
    assert a["step_bytes"] == w_bytes + 2 * T * H * 2 + 4 * T * H * 2 + a["lora_page_bytes"]
    assert 60e6 < a["lora_page_bytes"] < 140e6            # ~101 MB expected for this draw family
    # decode shape is HBM-bound: arithmetic intensity below the measured ridge
    pk = bench.load_peaks()
    assert a["step_flops"] / a["step_bytes"] < pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"]


def test_algorithmic_prefill_is_tensor_bound():
    wl = workloads.make(3)
    a = bench.algorithmic(wl)
    assert bench.gemm_launch_groups(wl) == [[0, 1, 2], [3]]          # one persistent launch for q/k/v
    pk = bench.load_peaks()
    assert a["step_flops"] / a["step_bytes"] > pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
v = bench.max_over_ranks(1.5 + r, dist)
bench.barrier(dist)
print(json.dumps({{"rank": r, "max": v}}))
dist.destroy_process_group()
"""


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(_WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    vals = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    assert sorted(v["rank"] for v in vals) == [0, 1]
    assert all(v["max"] == 2.5 for v in vals)


def test_reference_arm_tiny_workload(capsys):
    bench.main(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["higher_is_better"] is True


def test_reference_arm_nonzero_rank_is_silent(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--config", "1", "--steps", "1", "--gpus", "2"])
    assert capsys.readouterr().out.strip() == ""


def test_gpus_flag_relaunches_or_checks_the_world(monkeypatch):
    """--gpus N outside torchrun starts N ranks; inside torchrun it must match WORLD_SIZE."""
    calls = []
    monkeypatch.setattr(bench, "relaunch_under_torchrun", lambda n, argv: calls.append((n, list(argv))) or 0)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.check_world(1, ["--gpus", "1"]) is None and calls == []
    assert bench.check_world(4, ["--gpus", "4", "--steps", "3"]) == 0
    assert calls == [(4, ["--gpus", "4", "--steps", "3"])]
    monkeypatch.setenv("WORLD_SIZE", "4")
    assert bench.check_world(4, []) is None
    with pytest.raises(SystemExit):
        bench.check_world(2, [])
    with pytest.raises(SystemExit):
        bench.check_world(0, [])


def test_gemm_kernel_names_restate_the_tile_choice():
    """The layer stack's q/k/v group (2,496 tokens, H = 5120) runs 256-feature tiles and its o
    projection 128-feature ones (200 tiles of 256 features would leave the second wave nearly
    empty); a decode batch of one slot takes the split-K kernel."""
    import bench
    assert bench.gemm_kernel_name(5120, 2496, 152, 3) == ["gemm_lora_persistent<2>"]
    assert bench.gemm_kernel_name(5120, 2496, 152, 1) == ["gemm_lora_persistent<1>"]
    assert bench.gemm_kernel_name(4096, 256, 152, 1) == ["gemm_lora_kernel"]
    assert bench.gemm_kernel_name(4096, 9553, 152, 1) == ["gemm_lora_persistent<2>"]
