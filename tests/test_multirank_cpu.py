"""The bench's multi-rank host logic on CPU: two gloo ranks, as torchrun would
start them.  Each rank draws its own seeded batch, the job time is the
slowest rank's, throughput counts every rank's tokens, and the reference arm
runs on rank 0 alone."""
import json
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.timeout(300) if hasattr(pytest.mark, "timeout") else []


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    from mixture_experts_layer_mok_gb300 import inputs as gen

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    r, w, loc = bench.dist_env()
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w, "cpu")     # rank 1 is the slow one
    inp = gen.make_workload("tiny", seed=r)
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as fh:
        json.dump({"rank": r, "world": w, "local": loc, "slowest": slowest,
                   "x0": inp.x[0, :4].float().tolist(), "te0": inp.top_experts[0].tolist()}, fh)


def test_two_gloo_ranks_time_and_seed(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1] and all(x["world"] == 2 for x in res)
    assert all(x["slowest"] == 15.0 for x in res)              # max over ranks, on every rank
    assert res[0]["x0"] != res[1]["x0"]                        # each rank its own batch (seed = rank)


def test_job_throughput_counts_every_rank():
    import bench

    # two ranks, 4096 tokens each, 10 steps, slowest rank 20 ms in total
    assert bench.job_tokens_per_s(4096, 2, 10, 20.0) == pytest.approx(4096 * 2 * 10 / 0.020)
    assert bench.job_tokens_per_s(4096, 1, 10, 20.0) == pytest.approx(4096 * 10 / 0.020)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def _ref_main(rank, world, port, outdir):
    import contextlib
    import io

    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import sys

    import bench

    sys.argv = ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"]
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main()
    with open(os.path.join(outdir, f"ref{rank}.txt"), "w") as fh:
        fh.write(buf.getvalue())


def test_reference_arm_prints_on_rank0_only(tmp_path):
    port = _free_port()
    mp.start_processes(_ref_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text().strip()
    assert out1 == ""
    assert len(out0) == 1
    line = json.loads(out0[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["n_gpus"] == 2                       # the job's N, though only host cores work
