"""Host logic of bench.py: byte/element accounting, row selection, the
max-over-ranks timing and barrier of the multi-process path (world size 2 on
the gloo backend, CPU only)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import workloads as W


def test_algorithmic_bytes():
    wl = W.SCAN_TINY
    assert bench.pass_bytes(wl, "fwd") == 12 * wl.N + 4 * wl.C
    assert bench.pass_bytes(wl, "bwd") == 20 * wl.N + 8 * wl.C
    assert bench.pass_bytes(W.SCAN_BF16, "fwd") == 6 * W.SCAN_BF16.N + 2 * W.SCAN_BF16.C
    assert bench.pass_bytes(W.SRU, "bwd") == 40 * W.SRU.N + 8 * W.SRU.C + 16 * W.SRU.D
    d = W.DEER
    assert bench.pass_bytes(d, "solve", 1) == 8 * d.N + 4 * d.D
    assert bench.pass_bytes(d, "solve", 3) == (8 + 12 + 12) * d.N + 12 * d.D
    assert bench.pass_elems(d, "solve", 6) == 6 * d.N


def test_step_rate_is_harmonic_mix():
    rates = {n: 1e9 for n, _, _ in bench.ROWS}
    assert bench.step_rate_from_rows(rates, 6) == pytest.approx(1e9)


def test_select_rows(monkeypatch):
    monkeypatch.setattr(bench, "ROWS", list(bench.ROWS))
    bench.select_rows(["scan_large.bwd", "deer"], 1024)
    assert [(n, p) for n, _, p in bench.ROWS] == [("scan_large", ("bwd",)), ("deer", ("solve",))]
    assert all(wl.T == 1024 for _, wl, _ in bench.ROWS)


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo")
    bench.barrier(2)
    out[rank] = bench.max_over_ranks(10.0 + rank, 2)
    dist.destroy_process_group()


def test_two_rank_max_timing():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
    assert dict(out) == {0: 11.0, 1: 11.0}
