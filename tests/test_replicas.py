"""The N>1 replicas path on CPU: world-size-2 gloo ranks (no GPU).

Each rank decodes its own sequence of the toy workload through the oracle
and the ranks exchange nothing but the measurement's barrier and max over
ranks, as the GPU replicas do.  Checks: the rank -> sequence assignment,
that a replica's results equal a single-process run of its sequence, the
max-over-ranks reduction and the whole-job rate, and that the reference
arm does its work on rank 0 only.
"""

import io
import multiprocessing as mp
import os
import pickle
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

from speculative_decoding_draft_stream_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOY = "toy_v4096_h256"
STEPS = 4


def _decode(seq: int):
    """Per step: I_t and the top-k ids and values of one sequence (oracle)."""
    import oracle
    from synth import Workload, get_config

    cfg = get_config(TOY)
    wl = Workload(cfg)
    W = wl.w_head()
    st = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
    st.init(wl.prompt(seq), wl.prefill_logits(seq))
    trees = wl.trees(seq)
    out = []
    for t in range(STEPS):
        st.append(trees[t], wl.verify_logits(seq, t), wl.verify_row(seq, t))
        I = st.active()
        _, _, ids, vals = oracle.sub_head_step(wl.hiddens(seq, t), W, I, cfg.k)
        out.append((I, ids, vals))
    return out


def _rank_main(rank: int, world: int, port: int, path: str):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        (seq,) = replicas.rank_sequences(rank, world)
        dist.barrier()
        res = _decode(seq)
        dist.barrier()
        # a stand-in for each rank's timed region: rank r "took" 0.25 * (r + 1) s
        slowest = replicas.max_over_ranks(0.25 * (rank + 1), dist)
        rate = replicas.whole_job_rate(STEPS, world, slowest)
        got = [None] * world
        dist.all_gather_object(got, {"rank": rank, "seq": seq, "res": res, "slowest": slowest, "rate": rate})
        if rank == 0:
            with open(path, "wb") as f:
                pickle.dump(got, f)
    finally:
        dist.destroy_process_group()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_rank_sequences_disjoint_and_weak():
    for world in (1, 2, 4, 8):
        for per in (1, 3):
            seqs = [replicas.rank_sequences(r, world, per) for r in range(world)]
            flat = [s for x in seqs for s in x]
            assert sorted(flat) == list(range(world * per))
            assert all(len(x) == per for x in seqs)
    assert replicas.rank_sequences(1, 2) == [1]
    with pytest.raises(ValueError):
        replicas.rank_sequences(2, 2)


def test_single_process_reduction_and_rate():
    assert replicas.max_over_ranks(1.5) == 1.5
    assert replicas.whole_job_rate(512, 1, 0.01) == pytest.approx(51200.0)
    assert replicas.whole_job_rate(512, 4, 0.02) == pytest.approx(102400.0)
    with pytest.raises(ValueError):
        replicas.whole_job_rate(1, 1, 0.0)


def test_two_gloo_replicas_match_single_process(tmp_path):
    pytest.importorskip("torch.distributed")
    world, port, path = 2, _free_port(), str(tmp_path / "gathered.pkl")
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, path)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert [p.exitcode for p in procs] == [0, 0]
    with open(path, "rb") as f:
        got = pickle.load(f)

    assert [g["rank"] for g in got] == [0, 1]
    assert [g["seq"] for g in got] == [0, 1]
    for g in got:
        assert g["slowest"] == pytest.approx(0.5)  # max over ranks, seen by every rank
        assert g["rate"] == pytest.approx(world * STEPS / 0.5)
    # each replica equals the same sequence decoded alone
    for g in got:
        alone = _decode(g["seq"])
        for (I, ids, vals), (I2, ids2, vals2) in zip(g["res"], alone):
            assert np.array_equal(I, I2) and np.array_equal(ids, ids2) and np.array_equal(vals, vals2)
    # and the two ranks really decoded different sequences
    assert not all(np.array_equal(a[0], b[0]) for a, b in zip(got[0]["res"], got[1]["res"]))


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2",
                                      "--warmup", "0"])
    args = bench.parse_args()
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    assert buf.getvalue() == ""
