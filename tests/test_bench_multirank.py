"""The benchmark's multi-rank plumbing on the CPU: two ranks over gloo,
launched the way a multi-GPU run is launched (torch.distributed.run,
127.0.0.1).  Every run of the layer is a replica, so the only collectives are
the timing barrier and the max over ranks; the reference arm runs on rank 0
alone and the other ranks exit 0 without output."""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, timeout=300):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port())] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_barrier_and_max_over_ranks_with_two_gloo_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import bench
        rank, world, local = bench.dist_setup(None)
        bench.barrier(world)
        m = bench.max_over_ranks(1.5 + rank, world)
        open({str(tmp_path)!r} + "/rank%d.txt" % rank, "w").write("%d %d %r" % (rank, world, m))
        import torch.distributed as dist
        dist.destroy_process_group()
    """))
    r = torchrun([str(script)])
    assert r.returncode == 0, r.stderr[-2000:]
    got = [(tmp_path / f"rank{i}.txt").read_text().split() for i in range(2)]
    assert [(g[0], g[1], float(g[2])) for g in got] == [("0", "2", 2.5), ("1", "2", 2.5)]


def test_reference_arm_prints_one_line_from_rank_zero_only():
    r = torchrun(["bench.py", "--impl", "reference", "--config", "tiny", "--gpus", "2",
                  "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
