"""Benchmark of the GDN speculative tree-verify step on one GB300 (or N replicas).

One step = gdn_conv_tree_step + gdn_tree_verify + gdn_commit over one round of
the throughput sweep: 64 sequences in a 128-slot pool, d = 128, 16-node random
draft trees (grouped heads H_k = 16, H_v = 32; the headline) plus the other
three sub-workloads (non-grouped 32/32, 64-token chains).  100 seeded rounds
are generated on the device before timing; steps cycle through them and the
pools persist across steps, as in a real decode loop.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is nodes/s over all ranks (each rank a
replica with its own pools: weak scaling).  L2 is flushed before every timed
step: a 256 MB write, then a 256 MB read of another buffer, so the flush's
dirty lines are written back before the step starts (--l2-dirty skips the
read and leaves them to the step).  Each step is timed with CUDA events on the
launching stream around the whole step (`value`, `ms_per_step`), and in a
second pass of the same K steps with events between the kernels as well (the
per-kernel split and roofline; those events stop the kernels' launches from
overlapping each other's tails).  `e2e` repeats the measurement through the same C
ABI from pinned host buffers, with the step's inputs copied in and its output
copied out inside the timed region.  `cpu_baseline` times the oracle on the
host cores on a bounded sample of the same workload.  `--impl reference` times
the oracle alone (the only reference implementation of this method here).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gdn_workloads as W  # noqa: E402

METRIC = "GDN tree-verify+commit nodes/s and achieved HBM GB/s (% of GB300 peak)"
HEADLINE = "grouped_tree16"
N_ROUNDS = 100
L2_FLUSH_BYTES = 256 << 20
L2_DIRTY = False  # --l2-dirty: flush by the write alone


class L2Flush:
    """Evicts the step's data from L2 between timed steps: a write of a buffer
    larger than L2, then (unless L2_DIRTY) a read of a second one, so that the
    write's dirty lines drain to DRAM outside the timed region."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = None if L2_DIRTY else torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.zeros((), dtype=torch.float32, device=device)

    def __call__(self, i):
        self.w.fill_(float(i))
        if self.r is not None:
            self.sink.add_(self.r.sum())

    @staticmethod
    def describe_static():
        if L2_DIRTY:
            return "flushed before every timed step (256 MB write; its dirty lines drain during the step)"
        return ("flushed before every timed step (256 MB write, then a 256 MB read of another buffer so "
                "the write's dirty lines drain before the step)")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------ algorithmic bytes
def algo_bytes(sp: W.Spec, parents: np.ndarray, node_off: np.ndarray, accepted: np.ndarray,
               compact: bool = False):
    """Bytes the method must move per launch (conv weights once per layer).
    compact: windows travel as three int32 references per node, and the commit
    gathers the accepted window (3 C floats) from x and the history."""
    sh = sp.shape
    S, Hv, d = sh.n_seqs, sh.h_v, sh.d
    C = sh.conv_channels
    N = int(node_off[-1])
    conv = N * C * 4 + S * 3 * C * 4 + 16 * C + N * C * 4 + (N * 3 * 4 if compact else N * 3 * C * 4)
    verify = S * Hv * d * d * 4 + N * C * 4 + N * 2 * Hv * 4 + N * Hv * d * 4 + N * Hv * (2 * d + 1) * 4
    commit = 0
    for s in range(S):
        a = int(accepted[s])
        if a < 0:
            continue
        n0 = int(node_off[s])
        m = 0
        while a >= 0:
            m += 1
            a = int(parents[n0 + a])
        commit += 2 * Hv * d * d * 4 + m * Hv * (2 * d + 1) * 4 + 2 * 3 * C * 4 + (3 * 4 if compact else 0)
    return {"conv": conv, "verify": verify, "commit": commit}


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- workload
class DeviceWorkload:
    """Pools, weights and N_ROUNDS rounds of inputs resident on the device.

    Tree structure, accepted nodes, gate projections and conv weights come from
    the SplitMix64 generator of gdn_workloads; the bulk tensors (tokens x and
    the two pools) are drawn on the device with torch's Philox generator keyed
    by the same stream keys, with the same distributions."""

    def __init__(self, sp: W.Spec, rounds: int, device, seed_offset: int = 0, layer: int = 0,
                 compact: bool = False):
        import torch
        self.sp, self.device = sp, device
        sh = sp.shape
        self.C = sh.conv_channels
        self.rs = (2 * sh.d + 1 + 3) // 4 * 4           # smallest replay row stride
        lp = W.layer_params(sp, layer, with_pools=False)
        g = torch.Generator(device=device)
        g.manual_seed(W.stream_key(sp.seed, seed_offset, layer, W.TID_STATE) & ((1 << 63) - 1))
        self.ssm = torch.randn((sh.n_slots, sh.h_v, sh.d, sh.d), generator=g, device=device) * 0.1
        g.manual_seed(W.stream_key(sp.seed, seed_offset, layer, W.TID_HIST) & ((1 << 63) - 1))
        self.hist = torch.randn((sh.n_slots, 3, self.C), generator=g, device=device)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.w, self.dt, self.A = t(lp.conv_w), t(lp.dt_bias), t(lp.A)
        self.slot_map = t(W.slot_map(sp))
        self.rounds = []
        self.host_rounds = []
        for r in range(rounds):
            ri = W.round_inputs(sp, layer, r, with_x=False)
            g.manual_seed(W.stream_key(sp.seed, seed_offset, layer, W.TID_X, r) & ((1 << 63) - 1))
            x = torch.randn((int(ri.node_off[-1]), self.C), generator=g, device=device)
            self.rounds.append(dict(x=x, ba=t(ri.ba), parents=t(ri.parents), node_off=t(ri.node_off),
                                    accepted=t(ri.accepted)))
            self.host_rounds.append(ri)
        N = int(self.host_rounds[0].node_off[-1])
        self.N = N
        self.xc = torch.empty((N, self.C), device=device)
        self.compact = compact
        self.win = torch.empty((1 if compact else N, 3, self.C), device=device)
        self.wref = torch.empty((N, 3), dtype=torch.int32, device=device)
        self.o = torch.empty((N, sh.h_v, sh.d), device=device)
        self.replay = torch.empty((N, sh.h_v, self.rs), device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        import gated_deltanet_speculative_gdn_gb300 as G
        self.G = G
        self.dims = G.GdnDims.make(sh.n_seqs, N, sh.n_slots, sh.h_k, sh.h_v, sh.d, sp.max_seq_nodes)
        # chains longer than one 16-node chunk go through the chain entry point
        # (chunked form, d = 128); shorter ones are single tensor-core items
        self.chain = sp.tree_kind == "chain" and sh.d == 128 and sp.max_seq_nodes > 16
        self.verify = G.gdn_chain_verify if self.chain else G.gdn_tree_verify

    def step(self, r, events=None, inputs=None):
        """conv -> verify -> commit on round r; events[i] recorded before call i."""
        G, sh = self.G, self.sp.shape
        R = inputs if inputs is not None else self.rounds[r]
        if events:
            events[0].record()
        if self.compact:
            G.gdn_conv_tree_step_compact(self.dims, R["x"], self.C, self.w, self.hist, R["parents"],
                                         R["node_off"], self.slot_map, self.xc, self.wref, self.status)
        else:
            G.gdn_conv_tree_step(self.dims, R["x"], self.C, self.w, self.hist, R["parents"], R["node_off"],
                                 self.slot_map, self.xc, self.win, self.status)
        if events:
            events[1].record()
        self.verify(self.dims, self.xc, R["ba"], 2 * sh.h_v, self.dt, self.A, self.ssm, 1.0,
                    R["parents"], R["node_off"], self.slot_map, self.o, self.replay, self.rs, self.status)
        if events:
            events[2].record()
        if self.compact:
            G.gdn_commit_compact(self.dims, R["accepted"], R["parents"], R["node_off"], self.slot_map,
                                 self.replay, self.rs, R["x"], self.C, self.wref, self.ssm, self.hist, self.status)
        else:
            G.gdn_commit(self.dims, R["accepted"], R["parents"], R["node_off"], self.slot_map, self.replay,
                         self.rs, self.win, self.ssm, self.hist, self.status)
        if events:
            events[3].record()


def source_sha(name: str) -> str:
    p = os.path.join(ROOT, "gated_deltanet_speculative_gdn_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


KERNEL_SRC = {"conv": "gdn_conv.cu", "verify": "gdn_verify.cu", "commit": "gdn_commit.cu"}


def ncu_traffic(kernel: str, variant: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None
    when absent or when the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        e = t[variant][kernel]
        if e.get("src_sha") != source_sha(KERNEL_SRC[kernel]):
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


class Ranks:
    """The host side of a multi-process run: one process per GPU, each an
    independent replica of the workload (no data-path exchange).  `barrier`
    lines the ranks up around a timed region, `max` takes a per-rank figure's
    maximum over the ranks, and only rank 0 reports.  With one process every
    method is local.  The process group is NCCL on GPUs; the tests use gloo."""

    def __init__(self, dist=None, device=None):
        self.dist = dist
        self.device = device
        self.rank = dist.get_rank() if dist is not None else 0
        self.world = dist.get_world_size() if dist is not None else 1

    @property
    def main(self) -> bool:
        return self.rank == 0

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, values):
        if self.dist is None:
            return [float(v) for v in values]
        import torch
        t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return [float(v) for v in t.tolist()]


def time_variant(variant: str, steps: int, warmup: int, device, seed_offset: int = 0,
                 e2e: bool = False, clocks: bool = False, ranks: Ranks = None):
    import torch
    ranks = ranks or Ranks()
    compact = variant.endswith("_compact")
    sp = W.sweep_spec(variant[: -len("_compact")] if compact else variant, rounds=N_ROUNDS)
    wl = DeviceWorkload(sp, min(N_ROUNDS, max(steps + warmup, 1)), device, seed_offset, compact=compact)
    flush = L2Flush(device)
    nr = len(wl.rounds)
    for i in range(warmup):
        flush(i)
        wl.step(i % nr)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    if sampler:
        sampler.__enter__()
        time.sleep(0.3)
    torch.cuda.synchronize()
    ranks.barrier()                                  # every rank's timed region starts together
    for i in range(steps):
        flush(i)                                     # L2 flush, outside the step's events
        wl.step((warmup + i) % nr, ev[i])
        ends[i].record()
    torch.cuda.synchronize()
    ranks.barrier()
    # The same K steps again with events only around each whole step: events
    # between the kernels would stop a kernel's launch from overlapping the
    # previous one's tail (programmatic dependent launch), so the step time
    # comes from this pass and the per-kernel split from the one above.
    whole = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    ranks.barrier()
    for i in range(steps):
        flush(i)
        whole[i][0].record()
        wl.step((warmup + i) % nr)
        whole[i][1].record()
    torch.cuda.synchronize()
    ranks.barrier()
    if sampler:
        sampler.__exit__()
    assert int(wl.status.item()) == 0, wl.G.gdn_status_str(int(wl.status.item()))
    per = {"conv": [], "verify": [], "commit": []}
    step_ms = [a.elapsed_time(b) for a, b in whole]
    step_ms_kernel_events = []
    for i in range(steps):
        e = ev[i] + [ends[i]]
        per["conv"].append(e[0].elapsed_time(e[1]))
        per["verify"].append(e[1].elapsed_time(e[2]))
        per["commit"].append(e[2].elapsed_time(e[3]))
        step_ms_kernel_events.append(e[0].elapsed_time(e[3]))
    bytes_ = [algo_bytes(sp, wl.host_rounds[(warmup + i) % nr].parents, wl.host_rounds[(warmup + i) % nr].node_off,
                         wl.host_rounds[(warmup + i) % nr].accepted, compact) for i in range(steps)]
    out = {"sp": sp, "wl": wl, "step_ms": step_ms, "step_ms_kernel_events": step_ms_kernel_events, "per": per,
           "bytes": bytes_,
           "clocks": sampler.summary() if sampler else None}
    if e2e:
        out["e2e"] = time_e2e(wl, steps, warmup)
        out["e2e_overlapped"] = time_e2e_overlapped(wl, steps, warmup)
    return out


def time_e2e(wl: DeviceWorkload, steps: int, warmup: int, host_rounds: int = 8):
    """Same step through the C ABI from pinned host buffers: H2D of the step's
    inputs and D2H of its attention output inside the timed region."""
    import torch
    nr = min(host_rounds, len(wl.rounds))
    host = []
    for r in range(nr):
        host.append({k: v.cpu().pin_memory() for k, v in wl.rounds[r].items()})
    dev_in = {k: torch.empty_like(v) for k, v in wl.rounds[0].items()}
    o_host = torch.empty(wl.o.shape, dtype=wl.o.dtype).pin_memory()
    st_host = torch.empty(1, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h = wl.o.numel() * wl.o.element_size() + 4
    flush = L2Flush(wl.device)

    def one(r):
        for k, v in host[r].items():
            dev_in[k].copy_(v, non_blocking=True)
        wl.step(r, None, dev_in)
        o_host.copy_(wl.o, non_blocking=True)
        st_host.copy_(wl.status, non_blocking=True)

    for i in range(warmup):
        one(i % nr)
    torch.cuda.synchronize()
    times = []
    for i in range(steps):
        flush(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        one((warmup + i) % nr)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.mean(times)
    return {"ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def time_e2e_overlapped(wl: DeviceWorkload, steps: int, warmup: int, host_rounds: int = 8):
    """The same steps through the C ABI from pinned host buffers with the copies
    on their own streams: step i's inputs go up (one copy stream) while step
    i - 1 computes and step i - 2's output comes back (a second copy stream),
    with double-buffered device inputs and outputs and events between the
    streams.  Every step's copies are inside the timed region; the figure is
    whole-run throughput (no L2 flush between steps: the three streams run
    concurrently)."""
    import torch
    nr = min(host_rounds, len(wl.rounds))
    host = [{k: v.cpu().pin_memory() for k, v in wl.rounds[r].items()} for r in range(nr)]
    dev_in = [{k: torch.empty_like(v) for k, v in wl.rounds[0].items()} for _ in range(2)]
    o_dev = [wl.o, torch.empty_like(wl.o)]
    o_host = [torch.empty(wl.o.shape, dtype=wl.o.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h = wl.o.numel() * wl.o.element_size()
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev() for _ in range(2)]
    in_free = [ev() for _ in range(2)]
    done = [ev() for _ in range(2)]
    out_free = [ev() for _ in range(2)]
    for e in in_free + out_free:
        e.record(comp)

    def run(i0, n):
        for i in range(i0, i0 + n):
            b, r = i % 2, i % nr
            with torch.cuda.stream(up):
                up.wait_event(in_free[b])
                for k, v in host[r].items():
                    dev_in[b][k].copy_(v, non_blocking=True)
                in_ready[b].record(up)
            comp.wait_event(in_ready[b])
            comp.wait_event(out_free[b])
            wl.o = o_dev[b]
            wl.step(r, None, dev_in[b])
            in_free[b].record(comp)
            done[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                o_host[b].copy_(o_dev[b], non_blocking=True)
                out_free[b].record(down)

    run(0, warmup)
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    run(warmup, steps)
    comp.wait_stream(down)
    z.record(comp)
    torch.cuda.synchronize()
    wl.o = o_dev[0]
    return {"ms_per_step": a.elapsed_time(z) / steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def time_config(index: int, steps: int, warmup: int, device):
    """The smaller workloads as whole steps: config 1 (a chain of 8), config 2
    (four 16-node trees) and config 3 (the 48-layer stack: conv -> verify ->
    commit per layer, each layer with its own weights and pools, timed as one
    step over all layers).  Each is timed twice: launched from the host call
    by call, and as one CUDA graph per round (the same launches captured once
    and replayed), which removes the host's per-launch cost from the step."""
    import torch
    sp = W.spec(index)
    nr = min(sp.rounds, 4)
    wls = [DeviceWorkload(sp, nr, device, layer=l) for l in range(sp.layers)]
    flush = L2Flush(device)

    def step(r):
        for wl in wls:
            wl.step(r % nr)

    def timed(run):
        times = []
        for i in range(steps):
            flush(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run(warmup + i)
            b.record()
            times.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in times)

    for i in range(warmup):
        flush(i)
        step(i)
    torch.cuda.synchronize()
    ms = timed(step)
    graphs = []
    for r in range(nr):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(r)
        graphs.append(g)
    for i in range(warmup):
        flush(i)
        graphs[i % nr].replay()
    torch.cuda.synchronize()
    ms_graph = timed(lambda r: graphs[r % nr].replay())
    st = int(sum(int(wl.status.item()) != 0 for wl in wls))
    assert st == 0, "device status set"
    hr = [wls[0].host_rounds[(warmup + i) % nr] for i in range(steps)]
    byts = statistics.mean(sum(algo_bytes(sp, r.parents, r.node_off, r.accepted).values()) for r in hr) * sp.layers
    nodes = wls[0].N * sp.layers
    best = min(ms, ms_graph)
    return {"workload": sp.name, "layers": sp.layers, "nodes_per_step": nodes, "ms_per_step": round(best, 5),
            "nodes_per_s": round(nodes / (best * 1e-3), 1), "step_algo_gbs": round(byts / (best * 1e-3) / 1e9, 1),
            "ms_per_step_host_launches": round(ms, 5), "ms_per_step_cuda_graph": round(ms_graph, 5),
            "gpu_launches_per_step": 4 * sp.layers}


def time_decode(steps: int, warmup: int, device):
    """The plain decode step at the headline shape (64 sequences, one token
    each, 128-slot pool, 16/32 heads, d = 128), state and history in place."""
    import torch
    import gated_deltanet_speculative_gdn_gb300 as G
    sp = W.Spec("decode64", W.Shape(64, 128, 16, 32, 128), "chain", [1] * 64, 5)
    sh = sp.shape
    S, C = sh.n_seqs, sh.conv_channels
    g = torch.Generator(device=device)
    g.manual_seed(W.stream_key(sp.seed, 0, W.TID_STATE) & ((1 << 63) - 1))
    ssm = torch.randn((sh.n_slots, sh.h_v, sh.d, sh.d), generator=g, device=device) * 0.1
    hist = torch.randn((sh.n_slots, 3, C), generator=g, device=device)
    lp = W.layer_params(sp, 0, with_pools=False)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    w, dt, A, sm = t(lp.conv_w), t(lp.dt_bias), t(lp.A), t(W.slot_map(sp))
    nr = 8
    xs = [torch.randn((S, C), generator=g, device=device) for _ in range(nr)]
    bas = [t(W.round_inputs(sp, 0, r, with_x=False).ba) for r in range(nr)]
    xc = torch.empty((S, C), device=device)
    o = torch.empty((S, sh.h_v, sh.d), device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    dm = G.GdnDims.make(S, S, sh.n_slots, sh.h_k, sh.h_v, sh.d, 16)
    flush = L2Flush(device)

    def step(i):
        G.gdn_decode_step(dm, xs[i % nr], C, w, hist, bas[i % nr], 2 * sh.h_v, dt, A, ssm, 1.0, sm, xc, o, status)

    for i in range(warmup):
        flush(i)
        step(i)
    torch.cuda.synchronize()
    ev = []
    for i in range(steps):
        flush(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step(warmup + i)
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    byts = (S * C * 4 + 2 * S * 3 * C * 4 + 16 * C + S * C * 4 + 2 * S * sh.h_v * sh.d * sh.d * 4 +
            S * 2 * sh.h_v * 4 + S * sh.h_v * sh.d * 4)
    return {"workload": "64 sequences x 1 token, 128-slot pool, H_k=16, H_v=32, d=128", "ms_per_step": round(ms, 5),
            "tokens_per_s": round(S / (ms * 1e-3), 1), "algo_bytes": byts,
            "algo_gbs": round(byts / (ms * 1e-3) / 1e9, 1), "launches_per_step": 3}


def time_gated_norm(wl: "DeviceWorkload", steps: int, warmup: int):
    """The gated RMS norm (sigmoid gate) over the headline verify output."""
    import torch
    sh = wl.sp.shape
    g = torch.Generator(device=wl.device)
    g.manual_seed(W.stream_key(wl.sp.seed, 0, W.TID_Z) & ((1 << 63) - 1))
    z = torch.randn((wl.N, sh.h_v * sh.d), generator=g, device=wl.device)
    nw = torch.ones(sh.d, device=wl.device) + 0.1 * torch.randn(sh.d, generator=g, device=wl.device)
    y = torch.empty_like(wl.o)
    flush = L2Flush(wl.device)
    for i in range(warmup):
        wl.G.gdn_gated_rmsnorm(wl.dims, wl.o, z, sh.h_v * sh.d, nw, 1e-6, 1, y)
    torch.cuda.synchronize()
    ev = []
    for i in range(steps):
        flush(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        wl.G.gdn_gated_rmsnorm(wl.dims, wl.o, z, sh.h_v * sh.d, nw, 1e-6, 1, y)
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(x.elapsed_time(b) for x, b in ev)
    byts = 3 * wl.N * sh.h_v * sh.d * 4 + sh.d * 4
    return {"ms": round(ms, 5), "algo_bytes": byts, "algo_gbs": round(byts / (ms * 1e-3) / 1e9, 1)}


# -------------------------------------------------------------- CPU baseline
def oracle_sample(variant: str, budget_s: float = 12.0, seqs_per_step=None, first_seq: int = 0, stride: int = 1):
    """Times the oracle (single-threaded C) on whole sequences of the sweep
    workload (sequences first_seq, first_seq + stride, ...) until the budget is
    spent.  Returns (nodes, seconds, sequences)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle as O
    orc = O.get()
    sp = W.sweep_spec(variant)
    sh = sp.shape
    lp = W.layer_params(sp, 0, with_pools=False)
    nodes, secs, done = 0, 0.0, 0
    ri = W.round_inputs(sp, 0, 0)
    s = first_seq
    while True:
        sub = W.subset(sp, ri, [s % sh.n_seqs])
        n = int(sub.node_off[-1])
        # a one-slot pool holding this sequence's state and history
        ssm = W.Stream(sp.seed, 1000 + s, W.TID_STATE).normal(sh.h_v * sh.d * sh.d, 0.1).reshape(
            1, sh.h_v, sh.d, sh.d)
        hist = W.Stream(sp.seed, 1000 + s, W.TID_HIST).normal(3 * sh.conv_channels).reshape(1, 3, -1)
        dm = O.Dims(1, n, 1, sh.h_k, sh.h_v, sh.d)
        t0 = time.perf_counter()
        rc, xc, win = orc.conv_tree_step(dm, sub.x, lp.conv_w, hist, sub.parents, sub.node_off, [0])
        rc2, o, rep = orc.tree_verify(dm, xc.astype(np.float32), sub.ba, lp.dt_bias, lp.A, ssm,
                                      sub.parents, sub.node_off, [0])
        rc3 = orc.commit(dm, sub.accepted, sub.parents, sub.node_off, [0], rep, win, ssm, hist)
        secs += time.perf_counter() - t0
        assert rc == rc2 == rc3 == 0
        nodes += n
        done += 1
        s += stride
        if (seqs_per_step is not None and done >= seqs_per_step) or (seqs_per_step is None and secs >= budget_s):
            break
    return nodes, secs, done


def _oracle_worker(args):
    variant, budget_s, first, stride = args
    return oracle_sample(variant, budget_s, first_seq=first, stride=stride)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_all_cores(variant: str, budget_s: float = 8.0):
    """The oracle as independent per-sequence instances over every host core
    (a spawned process pool; sequences are independent).  Returns (nodes,
    seconds, sequences, cores): seconds is the longest worker's compute time."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle as O
    O.build()                       # once, before the workers load it
    n = host_cores()
    with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
        res = list(ex.map(_oracle_worker, [(variant, budget_s, w, n) for w in range(n)]))
    return sum(r[0] for r in res), max(r[1] for r in res), sum(r[2] for r in res), n


def parity_spot(wl: DeviceWorkload, seqs=(0, 63), r: int = 0):
    """One more (untimed) step of the benchmark's own device-drawn round r,
    checked against the oracle on a few sequences: the pools of their slots
    are read before the step, the oracle runs conv -> verify -> commit on the
    same inputs, and the outputs and committed state are compared."""
    import torch
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle as O
    sp, sh = wl.sp, wl.sp.shape
    sm = W.slot_map(sp)
    slots = [int(sm[s]) for s in seqs]
    ssm0 = wl.ssm[slots].cpu().numpy()
    hist0 = wl.hist[slots].cpu().numpy()
    wl.status.zero_()
    wl.step(r)
    torch.cuda.synchronize()
    ri = wl.host_rounds[r]
    sub = W.subset(sp, ri, list(seqs))
    rows = np.concatenate([np.arange(ri.node_off[s], ri.node_off[s + 1]) for s in seqs])
    x = wl.rounds[r]["x"].cpu().numpy()[rows]
    lp = W.layer_params(sp, 0, with_pools=False)
    orc = O.get()
    dm = O.Dims(len(seqs), len(rows), len(seqs), sh.h_k, sh.h_v, sh.d)
    slot_ids = list(range(len(seqs)))
    rc, xc, win = orc.conv_tree_step(dm, x, lp.conv_w, hist0, sub.parents, sub.node_off, slot_ids)
    rc2, o, rep = orc.tree_verify(dm, xc.astype(np.float32), sub.ba, lp.dt_bias, lp.A, ssm0, sub.parents,
                                  sub.node_off, slot_ids)
    ssm1, hist1 = ssm0.copy(), hist0.copy()
    rc3 = orc.commit(dm, sub.accepted, sub.parents, sub.node_off, slot_ids, rep, win, ssm1, hist1)
    assert rc == rc2 == rc3 == 0

    def rel(g, ref):
        g, ref = np.asarray(g, np.float64), np.asarray(ref, np.float64)
        rms = float(np.sqrt(np.mean(ref * ref)))
        return float(np.max(np.abs(g - ref) / np.maximum(np.abs(ref), 0.1 * rms)))

    d = sh.d
    g_rep = wl.replay.cpu().numpy()[rows, :, : 2 * d + 1]
    acc = [int(a) >= 0 for a in sub.accepted]
    out = {"sequences": list(seqs), "round": r, "status": int(wl.status.item()),
           "xc": rel(wl.xc.cpu().numpy()[rows], xc), "o": rel(wl.o.cpu().numpy()[rows], o),
           "replay_k": rel(g_rep[..., :d], rep[..., :d]), "replay_u": rel(g_rep[..., d:2 * d], rep[..., d:2 * d]),
           "replay_decay": rel(g_rep[..., 2 * d], rep[..., 2 * d]),
           "ssm": rel(wl.ssm[slots].cpu().numpy()[acc], ssm1[acc]) if any(acc) else 0.0,
           "win_bit_exact": bool(np.array_equal(wl.win.cpu().numpy()[rows], win)),
           "conv_hist_bit_exact": bool(np.array_equal(wl.hist[slots].cpu().numpy(), hist1))}
    out["pass"] = bool(out["status"] == 0 and out["win_bit_exact"] and out["conv_hist_bit_exact"] and
                       max(out[k] for k in ("xc", "o", "replay_k", "replay_u", "replay_decay", "ssm")) <= 1e-4)
    return {k: (f"{v:.2e}" if isinstance(v, float) else v) for k, v in out.items()}


# ---------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variants", default="all", help="'all', 'none' or a comma list of sweep variants")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default="1,2,3",
                    help="smaller workloads timed as whole steps (comma list of 1, 2, 3; 'none')")
    ap.add_argument("--l2-dirty", action="store_true", help="flush L2 by the write alone (no draining read)")
    args = ap.parse_args()
    global L2_DIRTY
    L2_DIRTY = bool(args.l2_dirty)
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    peak, peak_kind = measured_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        return reference_arm(args, peak, peak_kind)

    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    ranks = Ranks(dist, device)

    variants = (list(W.SWEEP_VARIANTS) + [HEADLINE + "_compact"] if args.variants == "all"
                else [] if args.variants in ("", "none") else args.variants.split(","))
    if HEADLINE in variants:
        variants.remove(HEADLINE)
    head = time_variant(HEADLINE, args.steps, args.warmup, device, seed_offset=rank, e2e=True, clocks=True,
                        ranks=ranks)
    others = {v: time_variant(v, args.steps, args.warmup, device, seed_offset=rank, ranks=ranks)
              for v in variants}
    extra = {"decode_step": time_decode(args.steps, args.warmup, device),
             "gated_rmsnorm_headline": time_gated_norm(head["wl"], args.steps, args.warmup)}
    cfg_ids = [] if args.configs in ("", "none") else [int(c) for c in args.configs.split(",")]
    configs = {W.SPEC_NAMES[c]: time_config(c, min(args.steps, 20), args.warmup, device) for c in cfg_ids}

    sp = head["sp"]
    N = head["wl"].N
    step_ms = statistics.mean(head["step_ms"])
    e2e_ms = head["e2e"]["ms_per_step"]
    e2e_ov_ms = head["e2e_overlapped"]["ms_per_step"]
    step_ms, e2e_ms, e2e_ov_ms = ranks.max([step_ms, e2e_ms, e2e_ov_ms])
    ranks.barrier()
    if not ranks.main:
        if dist is not None:
            dist.destroy_process_group()
        return

    nodes_total = N * world
    value = nodes_total / (step_ms * 1e-3)
    kern_ms = {k: statistics.mean(v) for k, v in head["per"].items()}
    kb = {k: statistics.mean(b[k] for b in head["bytes"]) for k in ("conv", "verify", "commit")}
    step_bytes = sum(kb.values())
    dom = max(kern_ms, key=kern_ms.get)
    achieved = kb[dom] / (kern_ms[dom] * 1e-3) / 1e9
    traffic = ncu_traffic(dom, HEADLINE)
    traffic_all = {k: ncu_traffic(k, HEADLINE) for k in kern_ms}
    measured = sum(traffic_all.values()) if all(traffic_all.values()) else None
    kernels = {k: {"ms": round(kern_ms[k], 5), "algo_bytes": int(kb[k]), "dram_bytes_ncu": traffic_all[k],
                   "gbs": round(kb[k] / (kern_ms[k] * 1e-3) / 1e9, 1),
                   "frac": round(kb[k] / (kern_ms[k] * 1e-3) / 1e9 / peak, 4),
                   "share": round(kern_ms[k] / sum(kern_ms.values()), 4)} for k in kern_ms}
    sweep = {}
    for v, r in others.items():
        ms = statistics.mean(r["step_ms"])
        b = statistics.mean(sum(x.values()) for x in r["bytes"])
        sweep[v] = {"nodes_per_s": round(r["wl"].N / (ms * 1e-3), 1), "ms_per_step": round(ms, 5),
                    "step_gbs": round(b / (ms * 1e-3) / 1e9, 1),
                    "frac_of_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                    "kernels_ms": {k: round(statistics.mean(x), 5) for k, x in r["per"].items()},
                    "verify_entry": r["wl"].verify.__name__}

    cpu = None
    spot = None
    if not args.no_cpu_baseline:
        spot = parity_spot(head["wl"])
        nodes1, secs1, nseq1 = oracle_sample(HEADLINE)
        nodes_n, secs_n, nseq_n, ncores = oracle_all_cores(HEADLINE)
        cpu = {"value": round(nodes_n / secs_n, 2), "unit": "nodes/s", "cores": ncores, "kind": "oracle",
               "sample": f"{nseq_n} whole sequences ({nodes_n} nodes) of the {HEADLINE} workload, "
                         f"conv+verify+commit, one single-threaded oracle process per core for "
                         f"{secs_n:.1f} s",
               "single_core": {"value": round(nodes1 / secs1, 2), "unit": "nodes/s", "cores": 1,
                               "sample": f"{nseq1} sequences ({nodes1} nodes), {secs1:.1f} s"}}

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "nodes/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 structure, Philox bulk tensors)",
        "config": {"workload": f"sweep_{HEADLINE}: 64 seqs x 16-node trees, 128-slot pool, H_k=16, "
                               f"H_v=32, d=128, d_conv=4, one layer, {N_ROUNDS} rounds",
                   "n_seqs": 64, "nodes_per_step": N, "h_k": 16, "h_v": 32, "d": 128,
                   "parallelism": f"replicas x{world}",
                   "l2": L2Flush.describe_static()},
        "hbm": {"step_algo_bytes": int(step_bytes),
                "step_algo_gbs": round(step_bytes / (step_ms * 1e-3) / 1e9, 1),
                "algo_frac_of_peak": round(step_bytes / (step_ms * 1e-3) / 1e9 / peak, 4),
                "step_dram_bytes_ncu": measured,
                "step_dram_gbs_ncu": (round(measured / (step_ms * 1e-3) / 1e9, 1) if measured else None),
                "peak_gbs": peak, "peak_kind": peak_kind,
                "note": "algorithmic bytes = what the method must move; the ncu figure is the DRAM traffic "
                        "of the same three kernels captured one launch each (null when a kernel changed "
                        "since its capture)",
                "ms_per_step_with_kernel_events": round(statistics.mean(head["step_ms_kernel_events"]), 5)},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": peak_kind},
        "kernels": kernels,
        "sweep": sweep,
        "e2e": {"value": round(nodes_total / (e2e_ms * 1e-3), 1), "unit": "nodes/s",
                "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": head["e2e"]["h2d_bytes_per_step"],
                "d2h_bytes_per_step": head["e2e"]["d2h_bytes_per_step"]},
        "e2e_overlapped": {"value": round(nodes_total / (e2e_ov_ms * 1e-3), 1),
                           "unit": "nodes/s", "ms_per_step": round(e2e_ov_ms, 5),
                           "h2d_bytes_per_step": head["e2e_overlapped"]["h2d_bytes_per_step"],
                           "d2h_bytes_per_step": head["e2e_overlapped"]["d2h_bytes_per_step"],
                           "note": "the same C-ABI steps with the input copy (one stream), the step (another) "
                                   "and the output copy (a third) of consecutive steps overlapped through "
                                   "double-buffered device buffers and events; e2e above is the serial figure"},
        "gpu_launches": 4 * args.steps * (1 + len(others)),
        "gpu_launches_note": "timed head steps x 4 launches (conv, verify, commit preflight, commit apply); "
                             "the second whole-step pass and the sweep variants launch the same per step",
        "clocks": head["clocks"],
        "cpu_baseline": cpu,
        "parity_spot": spot,
        "configs": configs,
        "other_stages": extra,
    }
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def reference_arm(args, peak, peak_kind):
    """The oracle, as it stands, on the host cores; each step a bounded sample
    (two whole sequences) of the headline workload."""
    for _ in range(args.warmup):
        oracle_sample(HEADLINE, seqs_per_step=1)
    nodes, secs = 0, 0.0
    for _ in range(args.steps):
        n, t, _ = oracle_sample(HEADLINE, seqs_per_step=2)
        nodes += n
        secs += t
    value = nodes / secs
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "nodes/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"sweep_{HEADLINE} (2 of 64 sequences per step)"},
        "cpu_baseline": {"value": round(value, 2), "unit": "nodes/s", "cores": 1, "kind": "oracle",
                         "sample": f"2 sequences (32 nodes) per step, {args.steps} steps"},
        "e2e": {"value": round(value, 2), "unit": "nodes/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
