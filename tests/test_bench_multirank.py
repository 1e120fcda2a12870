"""Host logic of bench.py for N > 1 ranks (one replica of the workload per GPU, no
data-path collective): the barrier, the max over ranks of the step time and the
whole-job rate, run as two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      CUDA_VISIBLE_DEVICES="")  # host logic only: gloo on the CPU
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    ms = 1.0 + rank  # rank 1 is the slower one
    slowest = bench.max_over_ranks(ms, w)
    rate = bench.whole_job_rate(1000, slowest, w)
    # a graph capture that failed on rank 0 only voids the job's graph timing
    g_fail = bench.graph_ms_over_ranks(-1.0 if rank == 0 else 0.5, w)
    g_ok = bench.graph_ms_over_ranks(0.5 + rank, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, slowest, rate, g_fail, g_ok))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for _, w, slowest, rate, g_fail, g_ok in out:
        assert w == 2 and slowest == 2.0
        assert rate == pytest.approx(2 * 1000 / 2e-3)
        assert g_fail == (None, True) and g_ok == (1.5, False)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(10, 2.0, 1) == pytest.approx(5000.0)


def test_oracle_sample_of_the_varlen_headline():
    """The CPU baseline's bounded sample keeps the leading tokens of every sequence
    with that sequence's own initial state, on the first heads only."""
    sys.path.insert(0, ROOT)
    import bench
    import kda_inputs as ki
    import torch
    lens = [5, 3000, 2048, 100] + [64] * 12
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 8, 64, 64, "bf16", seed=3, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    x, text = bench.oracle_sample(4, d, threads=20)   # 20 threads over 16 sequences: 2 heads
    keep = [min(n, bench.ORACLE_SEQ_TOKENS) for n in lens]
    assert x["cu_seqlens"].tolist() == ki.cu_seqlens_from_lengths(keep).tolist()
    assert x["q"].shape == (1, sum(keep), 2, 64) and x["initial_state"].shape == (16, 2, 64, 64)
    a, b = int(cu[1]), int(cu[1]) + bench.ORACLE_SEQ_TOKENS
    assert torch.equal(x["k"][:, 5:5 + bench.ORACLE_SEQ_TOKENS], d["k"][:, a:b, :2])
    assert torch.equal(x["initial_state"], d["initial_state"][:, :2])
    assert "16 sequences" in text and "2 of 8 heads" in text
