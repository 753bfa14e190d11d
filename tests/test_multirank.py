"""The replicated (N > 1) path of bench.py on CPU: two gloo ranks.

Multi-GPU here is replicas only: every rank runs its own seeded batch on its
own GPU, with no collective on the data path; the bench then takes the
whole-job figures over the process group (work units summed, times the
slowest rank's).  These tests run that host logic with the gloo backend."""
import importlib.util
import multiprocessing as mproc
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _load_bench()
        r, w, local = bench.dist_env()
        # per-rank work and times, different on purpose
        units, step_s, e2e_s = 100.0 * (rank + 1), 1e-3 * (rank + 1), 3e-3 - 1e-3 * rank
        job = bench.whole_job(units, step_s, e2e_s, w, torch.device("cpu"))
        case = bench.make_workload("tiny_gqa_decode", 7 + r)  # the bench seeds rank r with seed + r
        ref_ran = None
        if rank != 0:  # the reference arm: rank 0 alone runs the oracle, the others do no work
            import argparse
            import contextlib
            import io
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                bench.run_reference(argparse.Namespace(workload="tiny_gqa_decode", seed=7,
                                                       block_size=16, steps=1, warmup=1, gpus=2))
            ref_ran = buf.getvalue()
        out[rank] = (r, w, local, job, [int(x) for x in case.context_lens], case.num_seqs, ref_ran)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_whole_job_figures():
    world = 2
    ctx = mproc.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for pr in procs:
            pr.start()
        for pr in procs:
            pr.join(timeout=240)
        codes = [pr.exitcode for pr in procs]
        for pr in procs:
            if pr.is_alive():
                pr.kill()
        assert codes == [0, 0], codes
        res = dict(out)
    for rank in range(world):
        r, w, local, job, ctx_lens, nseq, _ = res[rank]
        assert (r, w, local) == (rank, world, rank)
        units, step_s, e2e_s = job
        assert units == pytest.approx(300.0)        # summed over ranks
        assert step_s == pytest.approx(2e-3)        # the slower rank's step
        assert e2e_s == pytest.approx(3e-3)         # the slower rank's end-to-end step
    # each rank has its own batch of the same shape
    assert res[0][5] == res[1][5]
    assert res[0][4] != res[1][4]
    assert res[1][6] == ""  # a non-zero rank prints nothing for the reference arm


def test_single_rank_passthrough():
    bench = _load_bench()
    assert bench.whole_job(5.0, 1e-3, 2e-3, 1, None) == (5.0, 1e-3, 2e-3)


def test_reference_arm_line_keeps_the_contract(capsys):
    # rank 0 of the reference arm: the oracle timed on the host cores, one
    # JSON line with the bench's keys, its own cpu_baseline and an e2e with
    # no device copies
    import argparse
    import json
    bench = _load_bench()
    bench.run_reference(argparse.Namespace(workload="tiny_gqa_decode", seed=3, block_size=16,
                                           steps=1, warmup=1, gpus=1))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["gpu_launches"] == 0
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny_gqa_decode"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
