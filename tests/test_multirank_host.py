"""The N-rank path of bench.py on CPU: world_size-2 gloo ranks run the same
barrier and max-over-ranks timing as the GPU replicas (one process per GPU,
no data-path collective), and the reference arm's non-zero ranks exit
without work."""

import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench._dist_init()
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench._barrier(w)
    m = bench._max_over_ranks(10.0 + 7.5 * rank, w)   # each rank's own step time
    bench._barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out, f"r{rank}"), "w") as f:
        f.write(repr(m))


def test_two_gloo_ranks_share_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    got = [float(open(tmp_path / f"r{r}").read()) for r in range(world)]
    assert got == [17.5, 17.5]


def test_reference_arm_nonzero_rank_exits_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_bench_kernel_work_table():
    """The roofline's algorithmic work per kernel class: every entry a
    (bound, amount) pair, the FLOP counts of the step, and the merge bytes of
    the bench workload's planner figures (16384 merged rows, 32768 partial
    rows per batch entry: 1.35 GB)."""
    import bench
    w = bench.kernel_work(partial_rows=32768, merge_rows=16384)
    assert set(w) == {"tile_fwd", "tile_bwd", "merge", "permute", "delta", "convert"}
    for bound, amount in w.values():
        assert bound in ("tensor", "hbm") and amount > 0
    assert w["tile_fwd"] == ("tensor", bench.FLOP_FWD) and w["tile_bwd"] == ("tensor", bench.FLOP_BWD)
    assert abs(w["merge"][1] - 1.3548e9) < 1e6
    assert set(bench._TRAFFIC) <= set(w)


def test_bench_traffic_table_shape():
    """Each recorded DRAM figure: bytes per step, the kernel sources it was
    captured from (files of the library) and a 16-hex-digit digest of them."""
    import os
    import re
    import bench
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tile_attention_lse_gb300", "csrc")
    for name, (nbytes, files, digest) in bench._TRAFFIC.items():
        assert isinstance(nbytes, float) and 1e8 < nbytes < 1e12, name
        assert files and all(os.path.exists(os.path.join(csrc, f)) for f in files), name
        assert re.fullmatch(r"[0-9a-f]{16}", digest), name
