#!/usr/bin/env python3
"""Benchmark of the chunked linear-recurrence hot path on one GB300 (or N
independent replicas under torchrun).

One step = one pass of every hot-path operation over its full-size synthetic
workload, in this order ([T, B, D] layout, seed 0):
  sru         fp32 32x2048x1024    fused SRU forward + backward
  scan_long   fp32 1x1048576x128   forward scan (million-step carry)
  scan_large  bf16 16x8192x4096    forward + backward scan
  scan_tiny   fp32 4x1024x256      forward + backward scan
  deer        fp32 4x65536x256     DEER Newton solve to max|dy| < 1e-5 (K iterations)

Metric: scan elements per second (each element of each pass counts once; a
DEER solve counts N*K) and the algorithmic HBM bytes per second.  Inputs are
resident in HBM before the timed region; every input except scan_tiny's
(12.6 MB) is larger than the 129 MB L2, and each step streams ~18 GB, so no
step starts with its inputs cached.  The scan_tiny passes are launch-bound
(a few microseconds of device work each): the step calls them after
scan_large, so that the host enqueues them while the GPU is still busy.

`value` and `ms_per_step` come from exactly --steps timed steps.  The
per-operation figures (`ops`) are medians over those steps and further steps
run until --ops-seconds have passed (clocks are sampled over both).

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import threading
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "scan elements/s and achieved HBM GB/s (fraction of GB300 peak), fwd+bwd"
UNIT = "elements/s"
FALLBACK_HBM_GBS = 6800.0
EPS, KMAX = 1e-5, 20

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture, keyed by operation; valid only while the kernel's sources (the
# shared device headers and its own kernel file) hash to `src`.  Filled from
# the committed ncu summaries under profiles/.  deer.solve: the DRAM bytes read
# and written by a K = 6 solve -- the reduce-only pass, iteration 1 and five
# later iterations, captured at full size (profiles/dram_traffic.md) -- over
# its K iteration launches.
NCU_TRAFFIC = {"deer.solve": {"bytes": 767176085, "src": "26d378f98ef291e6",
                              "file": "deer_kernels.cu"}}


def code_hash(texts) -> str:
    """Hash of source texts (an iterable of strings, in a fixed order) with
    line comments, trailing blanks and blank lines left out."""
    h = hashlib.sha256()
    for text in texts:
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def src_hash(kernel_file: str = "deer_kernels.cu") -> str:
    """Hash of the code one operation's kernels are compiled from: the shared
    device headers, the launch configuration and that operation's kernel
    file (the host-only C-ABI files and the other operations' kernel files do
    not change its kernel)."""
    cdir = os.path.join(ROOT, "linear_recurrence_scan_chunked_gb300", "csrc")
    names = [n for n in sorted(os.listdir(cdir)) if n.endswith(".cuh") or n in ("lr_launch.h", kernel_file)]
    return code_hash(open(os.path.join(cdir, n)).read() for n in names)


def recorded_traffic(op: str):
    """NCU_TRAFFIC's DRAM bytes per launch for `op`, or None when there is no
    record or the kernel's sources changed since it was captured."""
    tr = NCU_TRAFFIC.get(op)
    return tr["bytes"] if tr and tr.get("src") == src_hash(tr["file"]) else None


def hbm_peak_from(d):
    """The measured HBM copy bandwidth (GB/s) in a parsed peaks file, or None:
    a number under hbm_gbs / hbm_GBs / hbm, or that key's value, burst or
    (failing both) sustained entry -- the kernels are timed on their own, so
    the burst figure is the one that applies."""
    if not isinstance(d, dict):
        return None
    for k in ("hbm_gbs", "hbm_GBs", "hbm"):
        if k in d:
            v = d[k]
            if isinstance(v, dict):
                v = v.get("value", v.get("burst", v.get("sustained")))
            try:
                v = float(v)
            except (TypeError, ValueError):
                return None
            return v if v > 0 else None
    return None


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            v = hbm_peak_from(json.load(open(p)))
            if v is not None:
                return v, "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------- workloads

def esize(wl):
    return 2 if wl.dtype == "bf16" else 4


# (name, workload, passes); bytes per element per pass (algorithmic).  The
# launch-bound scan_tiny row runs after scan_large, while the GPU is still busy
# with it, so that its launches are enqueued ahead as in a training loop
# (the DEER solve at the end of a step waits for its residuals on the host:
# whatever comes first in the next step starts on an idle GPU).
ROWS = [("sru", W.SRU, ("fwd", "bwd")),
        ("scan_long", W.SCAN_LONG, ("fwd",)),
        ("scan_large", W.SCAN_BF16, ("fwd", "bwd")),
        ("scan_tiny", W.SCAN_TINY, ("fwd", "bwd")),
        ("deer", W.DEER, ("solve",))]


def select_rows(only, T):
    """Restrict the step to the named operations (name or name.pass)."""
    global ROWS
    if not only:
        return
    keep = []
    for name, wl, passes in ROWS:
        ps = tuple(p for p in passes if name in only or f"{name}.{p}" in only)
        if ps:
            keep.append((name, W.like(wl, T=T, name=wl.name) if T else wl, ps))
    if not keep:
        raise SystemExit(f"--only {only}: no such operation")
    ROWS = keep


def pass_bytes(wl, p, k=1):
    """Algorithmic HBM bytes of one pass (state/parameter vectors included)."""
    es, N, C, D = esize(wl), wl.N, wl.C, wl.D
    if wl.kind == "scan":
        return (3 * es * N + es * C) if p == "fwd" else (5 * es * N + 2 * es * C)
    if wl.kind == "sru":
        return (6 * es * N + es * C + 8 * D) if p == "fwd" else (10 * es * N + 2 * es * C + 16 * D)
    # DEER: iteration 1 reads u and writes y; later iterations also read y_old
    return es * N * (2 + 3 * (k - 1)) + 4 * D * k


def pass_elems(wl, p, k=1):
    return wl.N * (k if p == "solve" else 1)


# Rows replayed as CUDA graphs inside the step (none: the tiny scan's passes,
# called directly behind scan_large, measured 8.7-9.7 / 8.9 us per pass against
# 10.0 / 11.0 us as one-kernel graph replays).
GRAPH_ROWS = ()


class Bench:
    def __init__(self, dev):
        import torch
        import linear_recurrence_scan_chunked_gb300 as lrs
        self.torch, self.lrs, self.dev = torch, lrs, dev
        lrs.load()
        self.host = {}
        self.d = {}
        for name, wl, _ in ROWS:
            inp = W.make_inputs(wl, 0)
            self.host[name] = inp
            self.d[name] = {k: self._to_dev(v, wl, k) for k, v in inp.items()}
            o = self.d[name]
            e = lambda: torch.empty((wl.T, wl.B, wl.D), dtype=self._tdt(wl), device=dev)
            if wl.kind == "scan":
                o["h"] = e()
                if wl.backward:
                    o["da"], o["db"] = e(), e()
                    o["dh0"] = torch.empty((wl.B, wl.D), dtype=self._tdt(wl), device=dev)
            elif wl.kind == "sru":
                o["h"], o["c"] = e(), e()
                o["grad"] = {k: e() for k in ("dxt", "duf", "dur", "dx")}
                o["grad"]["dbf"] = torch.empty(wl.D, device=dev)
                o["grad"]["dbr"] = torch.empty(wl.D, device=dev)
                o["grad"]["dc0"] = torch.empty((wl.B, wl.D), dtype=self._tdt(wl), device=dev)
            else:
                o["y"] = e()
        self.k_last = 0
        self.graphs = {}
        torch.cuda.synchronize()

    def _tdt(self, wl):
        return self.torch.bfloat16 if wl.dtype == "bf16" else self.torch.float32

    def _to_dev(self, v, wl, key):
        t = self.torch
        if key in ("w", "bf", "br") or wl.dtype == "f32":
            return t.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(self.dev)
        return t.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(t.bfloat16).to(self.dev)

    # one row; returns (elements, bytes, launches)
    def run_row(self, name, wl, passes, ev=None):
        elems = byts = launches = 0
        for p in passes:
            if ev is not None:
                ev[(name, p)][0].record()
            g = self.graphs.get((name, p))
            if g is not None:
                g.replay()
                launches += 1
            else:
                launches += self.run_pass(name, wl, p)
            if ev is not None:
                ev[(name, p)][1].record()
            k = self.k_last if p == "solve" else 1
            elems += pass_elems(wl, p, k)
            byts += pass_bytes(wl, p, k)
        return elems, byts, launches

    def run_pass(self, name, wl, p):
        """One pass through the public binding; returns the kernel launches."""
        L, o = self.lrs, self.d[name]
        launches = 0
        if True:
            if wl.kind == "scan" and p == "fwd":
                L.lr_scan_fwd(o["a"], o["b"], o["h0"], o["h"])
                launches += 1
            elif wl.kind == "scan":
                L.lr_scan_bwd(o["a"], o["h"], o["g"], o["h0"], o["da"], o["db"], o["dh0"])
                launches += 1
            elif wl.kind == "sru" and p == "fwd":
                L.sru_fwd(o["xt"], o["uf"], o["ur"], o["x"], o["bf"], o["br"], o["c0"], o["h"], o["c"])
                launches += 1
            elif wl.kind == "sru":
                L.sru_bwd(o["xt"], o["uf"], o["ur"], o["x"], o["bf"], o["br"], o["c"], o["dh"],
                          o["c0"], out=o["grad"])
                launches += 3  # fused backward + two bias-reduction stages
            else:
                r = L.deer_diag_solve_ex(o["w"], o["u"], o["h0"], o["y"], eps=EPS, kmax=KMAX)
                if r["status"] != L.LR_OK:
                    raise RuntimeError(f"DEER did not converge (status {r['status']})")
                self.k_last = r["iters"]
                self.hist_last = r["hist"]
                # iterations are enqueued in batches; those after the stopping
                # test return at once but are still launches
                launches += r["launches"]
        return launches

    def capture_graphs(self):
        """After the warm-up (every row has sized the library's workspace):
        capture each pass of the launch-bound rows as a CUDA graph."""
        t = self.torch
        for name, wl, passes in ROWS:
            if name not in GRAPH_ROWS:
                continue
            for p in passes:
                g = t.cuda.CUDAGraph()
                with t.cuda.graph(g):
                    self.run_pass(name, wl, p)
                self.graphs[(name, p)] = g
        t.cuda.synchronize()

    def back_to_back_us(self, name, reps=64, rounds=15):
        """Device time per launch of each pass of a launch-bound row, from a
        graph of `reps` launches in a row (each starts when the previous one
        ends): the kernel's own time, no host in between.  Median of
        `rounds` replays."""
        t = self.torch
        wl = next(w for n, w, _ in ROWS if n == name)
        passes = next(ps for n, _, ps in ROWS if n == name)
        out = {}
        for p in passes:
            g = t.cuda.CUDAGraph()
            with t.cuda.graph(g):
                for _ in range(reps):
                    self.run_pass(name, wl, p)
            g.replay()
            ts = []
            for _ in range(rounds):
                e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
                t.cuda.synchronize()
                e0.record()
                g.replay()
                e1.record()
                t.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3 / reps)
            us = statistics.median(ts)
            byt = pass_bytes(wl, p)
            out[p] = {"us_per_launch": round(us, 3), "GBps": round(byt / (us / 1e6) / 1e9, 1),
                      "launches_per_graph": reps}
            del g
        return out

    def step(self, ev=None):
        tot = [0, 0, 0]
        for name, wl, passes in ROWS:
            r = self.run_row(name, wl, passes, ev)
            tot = [a + b for a, b in zip(tot, r)]
        return tot

    def time_deer_bwd(self, peak, reps=10):
        """deer_diag_bwd on the DEER workload: mean event time over `reps`
        launches after 3 warm-up launches (inputs larger than L2)."""
        t, L, o = self.torch, self.lrs, self.d["deer"]
        wl = W.DEER
        if "dy" not in o:
            o["dy"] = t.from_numpy(W.normal(0, 90, (wl.T, wl.B, wl.D))).to(self.dev)
            o["du"] = t.empty_like(o["dy"])
            o["dw"] = t.empty(wl.D, device=self.dev)
        run = lambda: L.deer_diag_bwd(o["w"], o["y"], o["dy"], o["h0"], o["du"], o["dw"],
                                      want_dh0=False)
        for _ in range(3):
            run()
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        t.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            run()
        e1.record()
        t.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        byt = 12 * wl.N + 8 * wl.D  # read y, dy; write du; w, dw
        return {"ms": round(ms, 4), "launches": 3, "GBps": round(byt / (ms / 1e3) / 1e9, 1),
                "frac": round(byt / (ms / 1e3) / 1e9 / peak, 3),
                "workload": f"deer fp32 T={wl.T} B={wl.B} D={wl.D}, gradient through the solution"}

    def time_deer_variants(self, peak, reps=5):
        """At the DEER workload's size: the ODE form (steps dt ~ U(0.1, 1)), a
        warm-started solve (the guess is the solution for u + 1e-3 sin, a
        nearby problem, as the previous training step's would be), the
        per-sequence stopping test and bf16 storage: mean solve time, K,
        algorithmic GB/s."""
        t, L, wl = self.torch, self.lrs, W.DEER
        o = self.d["deer"]
        N, D = wl.N, wl.D
        out = {}
        dt = t.from_numpy(W.uniform(0, 44, (wl.T,), 0.1, 1.0)).to(self.dev)
        y = t.empty_like(o["u"])
        res = {}

        def ode():
            res["k"] = L.deer_ode_solve(o["w"], o["u"], dt, o["h0"], y, eps=EPS, kmax=KMAX)[1]

        ms = self._mean_ms(ode, reps)
        k = res["k"]
        byt = (8 + 12 * (k - 1)) * N + 4 * D * k + 4 * wl.T * k
        out["deer_ode.solve"] = {"ms": round(ms, 4), "iters": k, "GBps": round(byt / (ms / 1e3) / 1e9, 1),
                                 "frac": round(byt / (ms / 1e3) / 1e9 / peak, 3),
                                 "workload": f"deer ODE form fp32 T={wl.T} B={wl.B} D={wl.D}, dt ~ U(0.1, 1)"}
        u2 = o["u"] + 1e-3 * t.sin(t.arange(N, device=self.dev, dtype=t.float32)).view_as(o["u"])
        guess = t.empty_like(o["u"])
        L.deer_diag_solve(o["w"], u2, o["h0"], guess, eps=EPS, kmax=KMAX)

        def warm():
            res["k"] = L.deer_diag_solve_ex(o["w"], o["u"], o["h0"], y, y_init=guess, eps=EPS,
                                           kmax=KMAX)["iters"]

        ms = self._mean_ms(warm, reps)
        k = res["k"]
        byt = 12 * N * k + 4 * D * k
        out["deer.warm"] = {"ms": round(ms, 4), "iters": k, "GBps": round(byt / (ms / 1e3) / 1e9, 1),
                            "frac": round(byt / (ms / 1e3) / 1e9 / peak, 3),
                            "workload": f"deer fp32 T={wl.T} B={wl.B} D={wl.D} from a nearby problem's solution"}

        def per_seq():
            r = L.deer_diag_solve_ex(o["w"], o["u"], o["h0"], y, eps=EPS, kmax=KMAX, per_sequence=True)
            res["k"], res["ks"] = r["iters"], r["seq_iters"]

        ms = self._mean_ms(per_seq, reps)
        k = res["k"]
        byt = (8 + 12 * (k - 1)) * N + 4 * D * k
        out["deer.per_sequence"] = {"ms": round(ms, 4), "iters": k, "seq_iters": res["ks"],
                                    "GBps": round(byt / (ms / 1e3) / 1e9, 1),
                                    "frac": round(byt / (ms / 1e3) / 1e9 / peak, 3),
                                    "workload": f"deer fp32 T={wl.T} B={wl.B} D={wl.D}, "
                                                "one stopping test per sequence"}
        # bf16 storage: the same workload's u rounded to bf16; the iterates
        # are stored in bf16, so the stopping test is taken at 1e-2 (bf16
        # rounding of the iterate puts a floor of ~1e-3 under the residual)
        ub = o["u"].to(t.bfloat16)
        yb = t.empty_like(ub)

        def bf16():
            r = L.deer_diag_solve_ex(o["w"], ub, None, yb, eps=1e-2, kmax=KMAX)
            res["k"], res["st"] = r["iters"], r["status"]

        ms = self._mean_ms(bf16, reps)
        k = res["k"]
        byt = (4 + 6 * (k - 1)) * N + 4 * D * k
        out["deer_bf16.solve"] = {"ms": round(ms, 4), "iters": k, "status": res["st"],
                                  "GBps": round(byt / (ms / 1e3) / 1e9, 1),
                                  "frac": round(byt / (ms / 1e3) / 1e9 / peak, 3),
                                  "workload": f"deer bf16 storage T={wl.T} B={wl.B} D={wl.D}, eps 1e-2"}
        del dt, y, u2, guess, ub, yb
        return out

    def _mean_ms(self, run, reps):
        t = self.torch
        for _ in range(3):
            run()
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        t.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            run()
        e1.record()
        t.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def time_lstm(self, peak, reps=10):
        """lstm_cell_fwd and lstm_cell_bwd on the LSTM cell workload (the SRU
        layer's size): mean event time over `reps` launches after 3 warm-up
        launches (every array larger than L2).  Device buffers are freed
        afterwards."""
        t, L, wl = self.torch, self.lrs, W.LSTM
        inp = W.make_inputs(wl, 0)
        d = {k: t.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(self.dev)
             for k, v in inp.items()}
        z = [d[k] for k in ("zf", "zi", "zc", "zo", "bf", "bi", "bc", "bo")]
        h, c = t.empty_like(d["zf"]), t.empty_like(d["zf"])
        grad = {k: t.empty_like(d["zf"]) for k in ("dzf", "dzi", "dzc", "dzo")}
        grad.update({k: t.empty(wl.D, device=self.dev) for k in ("dbf", "dbi", "dbc", "dbo")})
        grad["dc0"] = t.empty((wl.B, wl.D), device=self.dev)
        N, C, D = wl.N, wl.C, wl.D
        out = {}
        for p, run, byt, launches in (
                ("fwd", lambda: L.lstm_cell_fwd(*z, d["c0"], h, c),
                 24 * N + 4 * C + 16 * D, 1),  # read 4 gates, write h, c; c0; 4 biases
                ("bwd", lambda: L.lstm_cell_bwd(*z, c, d["dh"], d["c0"], out=grad),
                 40 * N + 8 * C + 32 * D, 3)):  # read 4 gates, c, dh, write 4; c0, dc0; biases
            ms = self._mean_ms(run, reps)
            gbs = byt / (ms / 1e3) / 1e9
            out[f"lstm.{p}"] = {"ms": round(ms, 4), "launches": launches, "GBps": round(gbs, 1),
                                "frac": round(gbs / peak, 3),
                                "workload": f"lstm cell fp32 T={wl.T} B={wl.B} D={wl.D}, {p}"}
        del d, z, h, c, grad
        t.cuda.empty_cache()
        return out

    # ---- end to end: host buffers, copies inside the timed region
    def setup_e2e(self):
        t = self.torch
        self.pin_in, self.pin_out = {}, {}
        self.h2d = self.d2h = 0
        for name, wl, passes in ROWS:
            o = self.d[name]
            ins = [k for k in self.host[name] if k not in ("w", "bf", "br")]
            self.pin_in[name] = {k: o[k].cpu().pin_memory() for k in ins}
            outs = {}
            if wl.kind == "scan":
                outs = {k: o[k] for k in (("h", "da", "db", "dh0") if wl.backward else ("h",))}
            elif wl.kind == "sru":
                outs = {"h": o["h"], "c": o["c"], **o["grad"]}
            else:
                outs = {"y": o["y"]}
            self.pin_out[name] = {k: (v, t.empty(v.shape, dtype=v.dtype, pin_memory=True))
                                  for k, v in outs.items()}
            self.h2d += sum(v.numel() * v.element_size() for v in self.pin_in[name].values())
            self.d2h += sum(v.numel() * v.element_size() for v, _ in self.pin_out[name].values())
        self.s_in, self.s_out = t.cuda.Stream(), t.cuda.Stream()

    def link_ceiling(self, nbytes=1 << 30, reps=3):
        """Pinned host <-> device copy bandwidth on this machine, GB/s: H2D alone,
        D2H alone, and both at once on two streams (as the e2e step runs
        them).  Best of `reps`."""
        t = self.torch
        n = nbytes // 4
        hin = t.empty(n, dtype=t.float32, pin_memory=True)
        hout = t.empty(n, dtype=t.float32, pin_memory=True)
        d1 = t.empty(n, dtype=t.float32, device=self.dev)
        d2 = t.empty(n, dtype=t.float32, device=self.dev)
        s1, s2 = t.cuda.Stream(), t.cuda.Stream()

        def one(src, dst, st):
            with t.cuda.stream(st):
                dst.copy_(src, non_blocking=True)

        res = {}
        for key, fn, byt in (("h2d", lambda: one(hin, d1, s1), nbytes),
                             ("d2h", lambda: one(d2, hout, s2), nbytes),
                             ("both", lambda: (one(hin, d1, s1), one(d2, hout, s2)), 2 * nbytes)):
            ts = []
            for _ in range(reps):
                t.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                t.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
            res[key + "_GBps"] = round(byt / min(ts) / 1e9, 1)
        del hin, hout, d1, d2
        return res

    def e2e_step(self):
        """One step from pinned host buffers: every row's inputs stream in on
        one copy stream, a row's kernels run on the current stream once its
        own inputs have landed, and its outputs stream out on a second copy
        stream, so the host link carries both directions at once, overlapped
        with the kernels.  Returns after every copy has completed."""
        t = self.torch
        comp = t.cuda.current_stream()
        ready = {}
        with t.cuda.stream(self.s_in):
            for name, wl, passes in ROWS:
                o = self.d[name]
                for k, hv in self.pin_in[name].items():
                    o[k].copy_(hv, non_blocking=True)
                ready[name] = t.cuda.Event()
                ready[name].record(self.s_in)
        elems = 0
        for name, wl, passes in ROWS:
            comp.wait_event(ready[name])
            e, _, _ = self.run_row(name, wl, passes)
            elems += e
            done = t.cuda.Event()
            done.record(comp)
            self.s_out.wait_event(done)
            with t.cuda.stream(self.s_out):
                for k, (dv, hv) in self.pin_out[name].items():
                    hv.copy_(dv, non_blocking=True)
        self.s_in.synchronize()
        comp.synchronize()
        self.s_out.synchronize()
        return elems


# ------------------------------------------------------------ clocks

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.p, self.lines = index, None, []

    def __enter__(self):
        # sample every 20 ms; the timed region starts once the first sample is
        # in (nvidia-smi takes a while to start)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
            return self
        self.first = threading.Event()

        def reader():
            for line in self.p.stdout:
                if line.strip():
                    self.lines.append(line)
                    self.first.set()
            self.first.set()

        self.t = threading.Thread(target=reader, daemon=True)
        self.t.start()
        self.first.wait(timeout=10)
        self.lines.clear()  # keep samples from the timed region only
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
            self.t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------- CPU (oracle) side

class OracleSampler:
    """Times the fp64 oracle, as it stands, on a bounded sample of every row's
    workload: the first T' time steps of C' channels (a time prefix of a
    channel subset is an exact sub-problem).  A short calibration run sizes the
    sample so each row takes about budget_s / rows seconds; the sampled inputs
    are generated once and reused by every timed run."""

    def __init__(self, budget_s: float):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.nth = oracle.num_threads()
        per = budget_s / len(ROWS)
        self.subs = {}
        for name, wl, passes in ROWS:
            Cs = min(wl.C, max(128, 8 * self.nth))
            Tc = min(wl.T, 256)
            inp = self._inputs(wl, Tc, Cs)
            el, dt, _ = self._run(wl, passes, inp)
            target = el / max(dt, 1e-4) * per  # elements that take about `per` seconds
            Ts = int(min(wl.T, max(Tc, target / (el / Tc))))
            if Ts == wl.T:  # the whole time axis fits: widen the channel sample instead
                Cs = int(min(wl.C, max(Cs, (target / (el / (Tc * Cs)) / wl.T) // 128 * 128)))
            self.subs[name] = self._inputs(wl, Ts, Cs)

    @staticmethod
    def _inputs(wl, T, Cs):
        if wl.kind == "sru":
            sub = W.like(wl, T=T, B=max(1, Cs // min(wl.D, 128)), D=min(wl.D, 128))
        else:
            sub = W.like(wl, T=T, B=1, D=Cs)
        inp = {k: (np.asarray(v, np.float64) if k in ("w", "bf", "br") else W.to_f64(v, wl.dtype))
               for k, v in W.make_inputs(sub, 0).items()}
        return sub, inp

    def _run(self, wl, passes, sub_inp):
        o, (sub, inp) = self.oracle, sub_inp
        t0 = time.perf_counter()
        el, k = 0, 1
        if wl.kind == "scan":
            h = o.scan_fwd(inp["a"], inp["b"], inp["h0"])
            el += sub.N
            if "bwd" in passes:
                o.scan_bwd(inp["a"], h, inp["g"], inp["h0"])
                el += sub.N
        elif wl.kind == "sru":
            h, c = o.sru_fwd(inp["xt"], inp["uf"], inp["ur"], inp["x"], inp["bf"], inp["br"], inp["c0"])
            o.sru_bwd(inp["xt"], inp["uf"], inp["ur"], inp["x"], inp["bf"], inp["br"], c, inp["dh"], inp["c0"])
            el += 2 * sub.N
        else:
            _, k, _, _ = o.deer(inp["w"], inp["u"], inp["h0"], eps=EPS, kmax=KMAX)
            el += sub.N * k
        return el, time.perf_counter() - t0, k

    def run_single_thread(self):
        """The same rows on one thread, each sample cut to 1/threads of its
        channels (about the same wall time): elements/s per row."""
        rates = {}
        n0 = self.oracle.num_threads()
        self.oracle.set_num_threads(1)
        try:
            for name, wl, passes in ROWS:
                sub, inp = self.subs[name]
                if wl.kind == "sru":
                    nb = max(1, sub.B // self.nth)
                    cut = W.like(sub, B=nb)
                    ci = {k: (v if np.ndim(v) == 1 else v[:, :nb] if np.ndim(v) == 3 else v[:nb])
                          for k, v in inp.items()}
                else:
                    nd = max(1, sub.D // self.nth)
                    cut = W.like(sub, D=nd)
                    ci = {k: (v[:nd] if k == "w" else v[..., :nd]) for k, v in inp.items()}
                el, dt, _ = self._run(wl, passes, (cut, ci))
                rates[name] = el / dt
        finally:
            self.oracle.set_num_threads(n0)
        return rates

    def run(self):
        """One pass over the samples: (elements/s per row, description, DEER K)."""
        rates, desc, kd = {}, [], 1
        for name, wl, passes in ROWS:
            el, dt, k = self._run(wl, passes, self.subs[name])
            if wl.kind == "deer":
                kd = k
            rates[name] = el / dt
            sub = self.subs[name][0]
            desc.append(f"{name}: first {sub.T} of T={wl.T} steps x {sub.C} of C={wl.C} channels, "
                        f"{dt:.2f} s ({el / dt / 1e6:.1f} M el/s)")
        return rates, "; ".join(desc), kd


def step_rate_from_rows(rates: dict, k_deer: int) -> float:
    """Elements/s of one full step when each row runs at its measured rate."""
    tot_el = tot_t = 0.0
    for name, wl, passes in ROWS:
        for p in passes:
            e = pass_elems(wl, p, k_deer)
            tot_el += e
            tot_t += e / rates[name]
    return tot_el / tot_t


# ------------------------------------------------------------------- main

def dist_init(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_dict():
    return {"workload": "; ".join(f"{n} {wl.dtype} T={wl.T} B={wl.B} D={wl.D} "
                                  f"{'+'.join(p)}" for n, wl, p in ROWS),
            "layout": "[T,B,D], D contiguous", "seed": 0,
            "storage": "as each workload names it (f32 or bf16); arithmetic in f32",
            "l2": "inputs larger than the 129 MB L2 except scan_tiny (12.6 MB); each step streams ~18 GB",
            "deer": {"eps": EPS, "kmax": KMAX},
            "distributions": "see workloads/__init__.py (N(0,0.01) read as std 0.01)"}


def run_reference(args, ws, rank):
    """The oracle on the host cores, same metric and step structure; each step
    is a bounded sample of the workload (the whole run stays within minutes)."""
    if rank != 0:
        return
    budget = max(4.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    smp = OracleSampler(budget)
    for _ in range(args.warmup):
        smp.run()
    vals, ks = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r, desc, kd = smp.run()
        ks.append(kd)
        vals.append(step_rate_from_rows(r, kd))
    wall = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": smp.nth, "kind": "oracle",
                             "sample": desc + f"; rates combined in the step's element mix, "
                                              f"DEER counted as N*K with the sample's K={ks[-1]}"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# Small programs of the bench's kernels for ncu captures: one short launch per
# kernel of interest, inputs still larger than the 129 MB L2, the public
# binding on the seeded inputs of `workloads`.  Launch order per case:
#   deer   DEER fp32 4x65536x256 (full size), three Newton iterations (eps = 0):
#          k_seg reduce-only (iteration 1's segment aggregates), then k_seg1 three
#          times (consume only), then the one-thread epoch retire
#   large  scan_large bf16 16x2048x4096 (T reduced from 8192): fwd, bwd
#   long   scan_long fp32 1x262144x128 (T reduced from 2^20): fwd
#   sru    SRU fp32 32x512x1024 (T reduced from 2048): fwd, bwd, 2 bias kernels
#   lstm   LSTM cell fp32 32x512x1024 (T reduced from 2048): fwd, bwd, 2 bias kernels
#   deerbwd  DEER backward fp32 4x65536x256 (full size) from a 3-iteration solve
#          (as `deer`), then k_seg (backward) and 2 dw kernels
#   tiny   scan_tiny fp32 4x1024x256 (full size; 12.6 MB, L2-resident after the
#          first launch): fwd, bwd, fwd, bwd
PROFILE_CASES = ("deer", "large", "long", "longfull", "sru", "lstm", "deerbwd", "tiny")


def profile_case(name):
    import dataclasses
    import torch
    import linear_recurrence_scan_chunked_gb300 as L
    L.load()

    def dev(inp, k):
        v = inp[k]
        if v.dtype == np.uint16:
            return torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()

    if name == "deer":
        inp = W.make_inputs(W.DEER, 0)
        L.deer_diag_solve(dev(inp, "w"), dev(inp, "u"), None, None, eps=0.0, kmax=3)
    elif name == "deerbwd":
        inp = W.make_inputs(W.DEER, 0)
        w, u = dev(inp, "w"), dev(inp, "u")
        y = L.deer_diag_solve(w, u, None, None, eps=0.0, kmax=3)[0]
        dy = torch.from_numpy(W.normal(0, 90, u.shape)).cuda()
        L.deer_diag_bwd(w, y, dy, None)
    elif name == "large":
        inp = W.make_inputs(dataclasses.replace(W.SCAN_BF16, T=2048), 0)
        a, b, g = dev(inp, "a"), dev(inp, "b"), dev(inp, "g")
        L.lr_scan_bwd(a, L.lr_scan_fwd(a, b, None), g, None)
    elif name == "tiny":
        inp = W.make_inputs(W.SCAN_TINY, 0)
        a, b, g = dev(inp, "a"), dev(inp, "b"), dev(inp, "g")
        for _ in range(2):
            L.lr_scan_bwd(a, L.lr_scan_fwd(a, b, None), g, None)
    elif name in ("long", "longfull"):
        wl = W.SCAN_LONG if name == "longfull" else dataclasses.replace(W.SCAN_LONG, T=1 << 18)
        inp = W.make_inputs(wl, 0)
        L.lr_scan_fwd(dev(inp, "a"), dev(inp, "b"), dev(inp, "h0"))
    elif name == "sru":
        inp = W.make_inputs(dataclasses.replace(W.SRU, T=512), 0)
        d = {k: dev(inp, k) for k in inp}
        h, c = L.sru_fwd(d["xt"], d["uf"], d["ur"], d["x"], d["bf"], d["br"], d["c0"])
        L.sru_bwd(d["xt"], d["uf"], d["ur"], d["x"], d["bf"], d["br"], c, d["dh"], d["c0"])
    elif name == "lstm":
        inp = W.make_inputs(dataclasses.replace(W.LSTM, T=512), 0)
        d = {k: dev(inp, k) for k in inp}
        z = [d[k] for k in ("zf", "zi", "zc", "zo", "bf", "bi", "bc", "bo")]
        h, c = L.lstm_cell_fwd(*z, d["c0"])
        L.lstm_cell_bwd(*z, c, d["dh"], d["c0"])
    torch.cuda.synchronize()
    if L.last_error() != L.LR_OK:
        raise RuntimeError("device error in the profiling case")
    print(f"profile case {name}: ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ops-seconds", type=float, default=2.5,
                    help="per-operation medians: steps after the timed ones until this much "
                         "time has passed since the timed region began")
    ap.add_argument("--no-next", action="store_true", help="skip the next rows (next_ops)")
    ap.add_argument("--only", action="append", default=[],
                    help="run only these operations (e.g. scan_large.bwd); for profiling cases")
    ap.add_argument("--T", type=int, default=0, help="override T of the selected rows (profiling cases)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="run one small program of the bench's kernels (for ncu) and exit")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    select_rows(args.only, args.T)
    ws, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
        barrier(ws)
        return

    import torch
    import linear_recurrence_scan_chunked_gb300 as lrs
    if args.warmup < 3:
        print("note: fewer than 3 warm-up steps requested; using 3", file=sys.stderr)
        args.warmup = 3
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    b = Bench(dev)
    for i in range(args.warmup):
        if i == args.warmup - 1:  # every shape has sized the workspace by now
            b.capture_graphs()
        b.step()
    torch.cuda.synchronize()
    if lrs.last_error() != lrs.LR_OK:
        raise RuntimeError("device error during warm-up")

    ev = {(n, p): (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for n, _, ps in ROWS for p in ps}
    per = {key: [] for key in ev}
    ks = []
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    elems = byts = launches = 0
    n_ops_steps = 0
    with Clocks(local) as clk:
        t_begin = time.perf_counter()
        start.record()
        for _ in range(args.steps):
            e, by, la = b.step(ev)
            elems, byts, launches = elems + e, byts + by, launches + la
            ks.append(b.k_last)
            torch.cuda.synchronize()  # per-row events are read per step
            for key, (e0, e1) in ev.items():
                per[key].append(e0.elapsed_time(e1))
        end.record()
        torch.cuda.synchronize()
        # more steps, for the per-operation medians only (not in `value`)
        while time.perf_counter() - t_begin < args.ops_seconds:
            b.step(ev)
            torch.cuda.synchronize()
            n_ops_steps += 1
            for key, (e0, e1) in ev.items():
                per[key].append(e0.elapsed_time(e1))
        ops_wall = time.perf_counter() - t_begin
    barrier(ws)
    ms = start.elapsed_time(end)
    ms = max_over_ranks(ms, ws)
    if lrs.last_error() != lrs.LR_OK:
        raise RuntimeError("device error during the timed region")
    ms_step = ms / args.steps
    value = elems * ws / (ms / 1e3)
    gbs = byts * ws / (ms / 1e3) / 1e9

    # per-operation breakdown and the dominant kernel's roofline
    peak, peak_kind = peak_hbm()
    k_med = int(statistics.median(ks))
    ops = {}
    for (n, p), ts in per.items():
        wl = next(w for nn, w, _ in ROWS if nn == n)
        k = k_med if p == "solve" else 1
        t_ms = statistics.median(ts)
        launches_op = k if p == "solve" else 1
        byt = pass_bytes(wl, p, k)
        ops[f"{n}.{p}"] = {"ms": round(t_ms, 4), "launches": launches_op,
                           "GBps": round(byt / (t_ms / 1e3) / 1e9, 1),
                           "frac": round(byt / (t_ms / 1e3) / 1e9 / peak, 3)}
    dom = max(ops, key=lambda k: ops[k]["ms"])
    dn, dp = dom.split(".")
    dwl = next(w for nn, w, _ in ROWS if nn == dn)
    k = k_med if dp == "solve" else 1
    launch_ms = ops[dom]["ms"] / ops[dom]["launches"]
    bytes_per_launch = pass_bytes(dwl, dp, k) / ops[dom]["launches"]
    achieved = bytes_per_launch / (launch_ms / 1e3) / 1e9
    traffic = recorded_traffic(dom)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": dom,
            "peak_source": f"{peak_kind} HBM copy bandwidth",
            "bytes_per_launch": bytes_per_launch}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config_dict(),
            "hbm_GBps": round(gbs, 1), "hbm_frac": round(gbs / peak, 4), "deer_iters": k_med,
            "deer_resid_history": [float(f"{r:.3e}") for r in getattr(b, "hist_last", [])],
            "gpu_launches": launches, "clocks": clk.summary(), "roofline": roof, "ops": ops,
            "ops_timing": {"stat": "median", "steps": args.steps + n_ops_steps,
                           "seconds": round(ops_wall, 2),
                           "graph_rows": list(GRAPH_ROWS)}}
    if "scan_tiny" in b.d:
        # the tiny scan's kernels back to back (graph of 64 launches): their
        # own device time, to which the step's per-pass figure adds a launch
        # and the events around it
        bb = b.back_to_back_us("scan_tiny")
        for p_, r in bb.items():
            r["frac"] = round(r["GBps"] / peak, 3)
        line["scan_tiny_back_to_back"] = bb

    # the next rows on the same scan, outside the step: the gradient through
    # the DEER solution at the DEER workload's size (from the step's own
    # solution), DEER's ODE form and a warm-started solve there, and the LSTM
    # cell forward and backward
    if not args.no_next:
        nxt = {}
        if "deer" in b.d:
            nxt["deer.bwd"] = b.time_deer_bwd(peak)
            nxt.update(b.time_deer_variants(peak))
        nxt.update(b.time_lstm(peak))
        line["next_ops"] = nxt

    if not args.no_e2e:
        b.setup_e2e()
        b.e2e_step()  # warm
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(ws)
        e0.record()
        el = 0
        for _ in range(args.e2e_steps):
            el += b.e2e_step()
        e1.record()
        torch.cuda.synchronize()
        t = max_over_ranks(e0.elapsed_time(e1), ws)
        line["e2e"] = {"value": el * ws / (t / 1e3), "unit": UNIT, "h2d_bytes_per_step": b.h2d,
                       "d2h_bytes_per_step": b.d2h, "ms_per_step": t / args.e2e_steps}
        # the host link's ceiling on this machine: the e2e step moves h2d + d2h
        # bytes per step, both directions at once
        lk = b.link_ceiling()
        moved = (b.h2d + b.d2h) / (t / args.e2e_steps / 1e3) / 1e9
        line["e2e"]["link"] = {**lk, "achieved_GBps": round(moved, 1),
                               "frac_of_both": round(moved / lk["both_GBps"], 3),
                               "how": "pinned 1 GiB copies, best of 3: H2D, D2H, both at once "
                                      "on two streams"}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        smp = OracleSampler(args.cpu_budget)
        rates, desc, _ = smp.run()
        r1 = smp.run_single_thread()
        line["cpu_baseline"] = {"value": step_rate_from_rows(rates, k_med), "unit": UNIT,
                                "cores": smp.nth, "kind": "oracle",
                                "sample": desc + f"; extrapolated to the step mix with K={k_med}",
                                "single_thread": {"value": step_rate_from_rows(r1, k_med),
                                                  "unit": UNIT, "cores": 1,
                                                  "sample": "the same samples cut to 1/"
                                                            f"{smp.nth} of their channels"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(ws)


if __name__ == "__main__":
    main()
