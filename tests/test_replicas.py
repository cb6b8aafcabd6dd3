"""The multi-process side of the bench on CPU (gloo, world size 2): the layer
does not shard, so N GPUs run N independent replicas and the ranks share
only the host-side control plane -- a barrier around the timed region and
the maximum of the ranks' times.  Also: under a multi-rank launch the
reference arm runs on rank 0 alone and the other ranks leave without work."""
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _env(rank, world, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    return env


def test_control_barrier_and_max_over_two_gloo_ranks():
    port = _free_port()
    code = textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {ROOT!r})
        import bench
        rank, world, _ = bench.dist_env()
        ctl = bench.Control(world)
        ctl.barrier()
        got = ctl.max(10.0 + 5.0 * rank)      # a slower rank 1
        ctl.barrier()
        print("MAX", rank, got, flush=True)
        ctl.close()
    """)
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    for r, out in enumerate(outs):
        assert f"MAX {r} 15.0" in out, out


def test_single_rank_control_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ctl = bench.Control(1)
    ctl.barrier()
    assert ctl.max(3.5) == 3.5
    ctl.close()


def test_reference_arm_leaves_other_ranks_without_work():
    port = _free_port()
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=_env(1, 2, port), cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
