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


def test_code_hash_ignores_comments_and_blank_lines():
    src = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    same = "// a header comment\nint f(int x) {\n\n    return x + 1;   \n}\n"
    other = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench.code_hash([src]) == bench.code_hash([same])
    assert bench.code_hash([src]) != bench.code_hash([other])
    assert bench.code_hash([src, other]) != bench.code_hash([other, src])


def test_recorded_traffic_needs_the_captured_sources(monkeypatch):
    rec = bench.NCU_TRAFFIC["deer.solve"]
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {
        "ok": dict(rec, src=bench.src_hash(rec["file"])),
        "stale": dict(rec, src="0" * 16)})
    assert bench.recorded_traffic("ok") == rec["bytes"]
    assert bench.recorded_traffic("stale") is None
    assert bench.recorded_traffic("absent") is None


def test_clock_summary():
    c = bench.Clocks(0)
    na = "Not Active"
    c.lines = [
        f"0, 2070, 2070, 812.3, 0x0000000000000000, {na}, {na}, {na}, {na}\n",
        f"0, 1965, 2070, 1390.0, 0x0000000000000004, {na}, {na}, {na}, Active\n",
        f"0, 2070, 2070, 900.1, 0x0000000000000000, {na}, {na}, {na}, {na}\n",
        "garbage line\n",
        "0, [N/A], 2070, 1.0, 0x0, x, x, x, x\n",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = []
    assert bench.Clocks(0).summary()["samples"] == 0


def test_measured_peak_parsing():
    assert bench.hbm_peak_from({"hbm_gbs": 7012.5}) == 7012.5
    assert bench.hbm_peak_from({"hbm_gbs": {"value": 7100, "clock_mhz": 2070}}) == 7100.0
    assert bench.hbm_peak_from({"hbm": {"burst": "7200"}}) == 7200.0
    assert bench.hbm_peak_from({"bf16_tflops": 1900}) is None
    assert bench.hbm_peak_from({"hbm_gbs": None}) is None
    assert bench.hbm_peak_from({"hbm_gbs": {"burst": 7300, "sustained": 7000}}) == 7300.0
    assert bench.hbm_peak_from({"hbm_gbs": {"sustained": 7000}}) == 7000.0
    assert bench.hbm_peak_from(["hbm_gbs"]) is None
    assert bench.hbm_peak_from({"hbm_gbs": 0}) is None
