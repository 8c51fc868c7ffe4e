"""The multi-rank host path of bench.py, on host cores: two ranks over gloo, launched the way a
multi-GPU run is (torch.distributed.run, one process per rank, rendezvous on 127.0.0.1).

The operation has no exchange step, so N ranks run N independent replicas.  What the ranks
share is the timing: every time is the slowest rank's, and the whole-job rate is the work of
all replicas over that time.  The reference arm runs on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, tmp_path, timeout=240):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port())] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_times_are_the_slowest_ranks_and_the_rate_counts_every_replica(tmp_path):
    out = tmp_path / "ranks"
    out.mkdir()
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import json, os, sys
        sys.path.insert(0, {ROOT!r})
        import bench
        dist, rank, world = bench.init_dist()
        assert dist is not None and dist.get_backend() == "gloo"
        # rank 0 is slower on the first time, rank 1 on the second
        mine = [10.0 + 5.0 * (rank == 0), 7.0 + 3.0 * (rank == 1)]
        worst = bench.max_over_ranks(dist, mine)
        rate = bench.job_tflops(world, 3.0e12, worst[0])
        with open(os.path.join({str(out)!r}, f"{{rank}}.json"), "w") as f:
            json.dump({{"rank": rank, "world": world, "worst": worst, "rate": rate}}, f)
        dist.destroy_process_group()
    """))
    r = torchrun([str(script)], tmp_path)
    assert r.returncode == 0, r.stderr[-3000:]
    got = sorted((json.loads((out / f"{i}.json").read_text()) for i in range(2)), key=lambda d: d["rank"])
    assert [d["rank"] for d in got] == [0, 1]
    for d in got:
        assert d["world"] == 2
        assert d["worst"] == [15.0, 10.0]
        # 2 replicas x 3 TFLOP each in 15 ms
        assert abs(d["rate"] - 2 * 3.0e12 / 15e-3 / 1e12) < 1e-9


def test_one_process_keeps_its_own_times():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [1.5, 2]) == [1.5, 2.0]
    assert bench.job_tflops(1, 1e12, 1000.0) == 1.0  # 1 TFLOP in one second


def test_reference_arm_prints_one_line_from_rank_zero(tmp_path):
    r = torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--config", "0", "--steps", "1",
                  "--warmup", "1", "--ref-seconds", "0.5"], tmp_path)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
