"""Host logic of the benchmark's multi-process path (replicas), on CPU with
gloo and world size 2: the whole-job time is the slowest rank's, tokens add up,
and the reference arm does no work on ranks other than 0."""

import os
import socket
import sys

import pytest
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r = bench.reduce_over_ranks(10.0 + rank, 100 + 7 * rank, 1.0 + 0.5 * rank, 50 + rank,
                                torch.device("cpu"))
    q.put((rank, r))
    dist.destroy_process_group()


def test_replicas_reduce_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(2):
        assert out[rank] == (11.0, 207.0, 1.5, 101.0)


def test_reference_arm_idle_on_other_ranks():
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    args = argparse.Namespace(steps=3, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_traffic_figure_only_for_the_kernel_it_was_taken_on(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "traffic.md"
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(prof))
    assert bench.captured_traffic() is None          # no summary
    prof.write_text(f"- kernel sources sha256: `{bench.kernel_source_hash()}`\n"
                    "- traffic per launch (bytes): 5278000000\n")
    assert bench.captured_traffic() == 5278000000
    prof.write_text("- kernel sources sha256: `0000`\n- traffic per launch (bytes): 5278000000\n")
    assert bench.captured_traffic() is None          # taken on other kernel sources


def test_expected_accept_matches_enumeration():
    """E[a] of the draft recipe (each draft copies the target's argmax with
    probability 0.7) against an enumeration of all 2^gamma hit patterns pushed
    through the oracle's greedy accept rule."""
    import itertools

    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    import oracle
    for gamma in range(0, 8):
        target = np.arange(100, 101 + gamma, dtype=np.int32)
        e = 0.0
        for hits in itertools.product((0, 1), repeat=gamma):
            d = np.array([target[i] if h else -1 - i for i, h in enumerate(hits)], dtype=np.int32)
            a, _ = oracle.spec_verify(target, d)
            e += a * np.prod([0.7 if h else 0.3 for h in hits])
        assert abs(e - bench.expected_accept(gamma)) < 1e-12, (gamma, e)
    assert abs(bench.expected_accept(4) - 1.7731) < 1e-12
