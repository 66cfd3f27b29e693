"""The bench's multi-rank path on CPU: two gloo ranks run replicas with
different step times; the whole-job figure uses the slowest rank's time and
all ranks' bytes.  The reference arm prints from rank 0 only.  --gpus N
without a torchrun environment spawns the N ranks itself."""
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_ms = [2.0, 5.0][rank]
    q.put((rank, bench.combine_ranks(step_ms, 1_000_000, world, torch.device("cpu"))))
    dist.barrier()
    dist.destroy_process_group()


def test_combine_ranks_takes_the_slowest_rank_and_all_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        ms, gbs = out[rank]
        assert ms == 5.0
        assert abs(gbs - 2 * 1_000_000 / 5e-3 / 1e9) < 1e-12


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    ms, gbs = bench.combine_ranks(4.0, 8_000_000, 1, torch.device("cpu"))
    assert ms == 4.0 and abs(gbs - 2.0) < 1e-12


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def _rank_job(argv):
    """A replica as bench.launch_replicas starts it: joins the gloo group from
    the environment it was given and reports its rank's view."""
    import torch.distributed as dist

    out_dir = argv[0]
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    ms, gbs = __import__("bench").combine_ranks([3.0, 7.0][rank], 1_000_000, world,
                                                torch.device("cpu"))
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{os.environ['RANK']} {os.environ['LOCAL_RANK']} {os.environ['WORLD_SIZE']} "
                f"{os.environ['MASTER_ADDR']} {ms} {gbs}")
    dist.destroy_process_group()


def test_launch_replicas_spawns_ranks_with_torchrun_environment(tmp_path):
    sys.path.insert(0, ROOT)
    import bench

    bench.launch_replicas(2, _rank_job, [str(tmp_path)])
    for r in (0, 1):
        rank, local, world, addr, ms, gbs = open(tmp_path / f"rank{r}.txt").read().split()
        assert (rank, local, world, addr) == (str(r), str(r), "2", "127.0.0.1")
        assert float(ms) == 7.0
        assert abs(float(gbs) - 2 * 1_000_000 / 7e-3 / 1e9) < 1e-9
