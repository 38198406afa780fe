"""bench.py's N > 1 host logic on CPU: two gloo ranks launched like the bench
(torch.distributed.run, 127.0.0.1); the replicas' time is the slowest rank's,
and the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "tests", "rank_worker.py")]
    env = dict(os.environ, OMP_NUM_THREADS="1", RANK_OUT_DIR=str(tmp_path))
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2)]
    assert [x["rank"] for x in lines] == [0, 1]
    for x in lines:
        assert x["world"] == 2 and x["slowest"] == 7.5


def test_max_over_ranks_alone_is_the_value_itself():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, None) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.main()
    assert capsys.readouterr().out == ""
