"""The multi-rank host logic of bench.py on CPU: two gloo ranks, one batch each
(different seeds, different inputs, no data-path collective), the timed region
closed by a barrier, and the slowest rank's time taken for the whole job."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from speculative_decoding_copy_gb300 import workloads as WL
        wl = WL.WORKLOADS["tiny"]
        inp = WL.make_inputs(wl, bench.rank_seed(rank))
        digest = float(np.asarray(inp["ctx"], dtype=np.float64).sum() + np.asarray(inp["tgt"], dtype=np.float64).sum())
        ms_local = 10.0 + 5.0 * rank                   # rank 1 is the slower one
        dist.barrier()
        ms = bench.max_over_ranks(ms_local, "cpu")
        q.put((rank, bench.rank_seed(rank), digest, ms, bench.whole_job_value(world, 100, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    res = sorted(q.get(timeout=5) for _ in range(2))
    (r0, s0, d0, ms0, v0), (r1, s1, d1, ms1, v1) = res
    assert (r0, r1) == (0, 1)
    assert s0 != s1 and d0 != d1                      # independent batches
    assert ms0 == ms1 == 15.0                          # every rank reports the slowest time
    assert v0 == v1 == pytest.approx(2 * 100 / 0.015)  # steps of both ranks per second


def test_gpus_flag_starts_its_own_ranks():
    """`bench.py --gpus 2` outside torchrun starts two ranks itself (torch.distributed.run,
    rendezvous on 127.0.0.1); with the reference arm only rank 0 works and prints, and the
    other rank exits 0 without work. Runs on the CPU (the reference arm is the oracle)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR",
                                                           "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
