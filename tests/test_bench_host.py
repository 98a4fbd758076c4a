"""Host-side logic of bench.py: workload naming, aggregation over ranks
(including a two-rank gloo run on CPU) and the reference arm's contract."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_workload_names():
    w, causal = bench.workload_by_name("d128_n4096_causal")
    assert (w.B, w.H, w.N, w.d, causal) == (4, 32, 4096, 128, True)
    w, causal = bench.workload_by_name("d128_n4096_noncausal")
    assert causal is False
    w, causal = bench.workload_by_name("custom_2_16_4096_128_causal")
    assert (w.B, w.H, w.N, w.d, causal) == (2, 16, 4096, 128, True)
    with pytest.raises(SystemExit):
        bench.workload_by_name("gpt2_small_n1024_d64_noncausal")  # only causal in that workload
    with pytest.raises(SystemExit):
        bench.workload_by_name("nope")


def test_decode_and_fp8_workload_names():
    assert bench.decode_spec("decode_8_32_1_16384_128_causal") == dict(B=8, H=32, Nq=1, Nk=16384, d=128, causal=True)
    assert bench.fp8_spec("fp8_4_32_4096_causal") == dict(B=4, H=32, N=4096, d=128, causal=True)
    assert bench.fp8_spec("fp8_1_16_16384_noncausal")["causal"] is False
    assert bench.fp8_spec("d128_n4096_causal") is None and bench.decode_spec("fp8_4_32_4096_causal") is None


def test_code_sha_ignores_comments_only(tmp_path, monkeypatch):
    """The traffic figures stay valid across comment edits of a kernel source and not across code edits."""
    csrc = tmp_path / "exact_io_aware_32_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("// head\nint f(int x) {  // note\n  return x + 1; /* a\n b */\n}\n")
    a = bench.code_sha("k.cu")
    (csrc / "k.cu").write_text("/* other words */\nint f(int x) {\n\n  return x + 1;\n}  // tail\n")
    assert bench.code_sha("k.cu") == a
    (csrc / "k.cu").write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_sha("k.cu") != a


def test_aggregate_uses_slowest_rank():
    v, t = bench.aggregate([1.0, 2.0, 1.5], [10.0, 10.0, 10.0])
    assert t == 2.0 and v == 15.0


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.reduce_max_over_ranks([1.0 + rank, 5.0 - rank], dist, "cpu")
    out[rank] = vals
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_two_ranks_gloo():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == [2.0, 5.0]


def test_reduce_max_without_group():
    assert bench.reduce_max_over_ranks([3.0, 1.0], None, "cpu") == [3.0, 1.0]


def test_reference_arm_contract():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--workload", "custom_1_1_256_64_causal", "--reference-budget", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["value"] > 0 and j["e2e"]["h2d_bytes_per_step"] == 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--impl", "reference"])
