"""Host-side logic of bench.py that needs no GPU: how --gpus N starts its ranks, the check
that --gpus matches the ranks it runs under, and the workload description both arms share."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402  (imports nothing beyond the standard library at module level)


def test_gpus_without_torchrun_starts_one_rank_per_gpu(monkeypatch):
    seen = {}

    def fake_call(cmd):
        seen["cmd"] = cmd
        return 0

    monkeypatch.setattr(bench.subprocess, "call", fake_call)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "7", "--warmup", "3"])

    class A:
        gpus = 4
        master_port = 29555

    assert bench.spawn_ranks(A) == 0
    cmd = seen["cmd"]
    assert cmd[:3] == [sys.executable, "-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29555"
    assert cmd[-6:] == ["--gpus", "4", "--steps", "7", "--warmup", "3"]
    assert os.path.basename(cmd[-7]) == "bench.py"


@pytest.mark.parametrize("world,gpus", [("1", "2"), ("2", "1"), ("4", "2")])
def test_gpus_must_match_the_ranks(world, gpus):
    env = dict(os.environ, WORLD_SIZE=world, RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", gpus, "--impl", "reference"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "WORLD_SIZE" in r.stderr


def test_both_arms_describe_the_same_workload():
    from denoising_sampler_step_gb300 import inputs
    wl = inputs.WORKLOADS[bench.WORKLOAD]
    c = bench.config_of(wl)
    assert c == bench.config_of(wl)
    assert set(c) == {"workload", "rows", "V", "d", "budget_nats", "l2"}
    assert c["rows"] == 256 and c["V"] == 262144 and c["d"] == 2816


def test_default_bench_times_the_tensor_bound_workloads():
    from denoising_sampler_step_gb300 import inputs
    names = bench.DEFAULT_ALSO.split(",")
    assert names == ["batch8", "late_batch32"]
    assert [inputs.WORKLOADS[n].R for n in names] == [2048, 8192]


def test_stored_traffic_is_taken_on_the_current_kernel_source():
    """The DRAM traffic the bench line reports comes from profiles/soft_embed_traffic.json only
    while its kernel-source hash is the current one: the committed file matches the committed
    kernel, and the traffic per call is what the profile states (1.02x the algorithmic bytes)."""
    tj = bench.stored_traffic()
    assert tj, "profiles/soft_embed_traffic.json was taken on another kernel source"
    assert tj["kernel_source_sha"] == bench.source_sha()
    from denoising_sampler_step_gb300 import cost
    sc = cost.StepCost(rows=256, V=262144, d=2816, vocab=262144)
    assert 1.0 <= tj["traffic_bytes_per_launch"] / sc.gemm_bytes <= 1.03
    assert 1.0 <= tj["e4m3_traffic_bytes_per_launch"] / sc.e4m3_gemm_bytes <= 1.05


def test_kernel_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """Comments and blank space do not change the hash; code does."""
    src = os.path.join(ROOT, "denoising_sampler_step_gb300", "csrc")
    dst = tmp_path / "denoising_sampler_step_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in ("soft_embed.cu", "dg_common.cuh"):
        (dst / f).write_text(open(os.path.join(src, f)).read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_sha()
    p = dst / "soft_embed.cu"
    p.write_text(p.read_text() + "\n// a comment\n/* and another */\n\n")
    assert bench.source_sha() == h0
    p.write_text(p.read_text() + "\nstatic int an_extra_line = 0;\n")
    assert bench.source_sha() != h0
