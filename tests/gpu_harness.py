"""Runs the CUDA path through the C ABI on workloads from gdn_workloads and
the oracle on the same inputs.  Used by the -m gpu tests and the smoke check.

Outputs are filled with NaN before each call so that an element a kernel
forgets to write shows up as a mismatch.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import gated_deltanet_speculative_gdn_gb300 as G
import gdn_workloads as W
import oracle as O

# max relative error against the oracle (floored at 0.1 x RMS of the reference)
TOL = 1e-4


def relerr(got, ref, floor_frac: float = 0.1) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), floor_frac * rms if rms > 0 else 1e-30)
    return float(np.max(np.abs(got - ref) / den))


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def nan_like(shape, dtype=torch.float32):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


@dataclass
class Batch:
    """One round's inputs for one layer, in plain arrays."""
    S: int
    P: int
    Hk: int
    Hv: int
    d: int
    max_nodes: int
    x: np.ndarray
    ba: np.ndarray
    parents: np.ndarray
    node_off: np.ndarray
    slot_map: np.ndarray
    accepted: np.ndarray
    conv_w: np.ndarray
    dt_bias: np.ndarray
    A: np.ndarray

    @property
    def N(self) -> int:
        return int(self.node_off[-1])

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.d + self.Hv * self.d

    def gdims(self) -> G.GdnDims:
        return G.GdnDims.make(self.S, self.N, self.P, self.Hk, self.Hv, self.d, self.max_nodes)

    def odims(self) -> O.Dims:
        return O.Dims(self.S, self.N, self.P, self.Hk, self.Hv, self.d)


def batch_from(sp: W.Spec, lp: W.LayerParams, ri: W.RoundInputs, sm=None,
               max_nodes: Optional[int] = None) -> Batch:
    sh = sp.shape
    return Batch(len(ri.node_off) - 1, sh.n_slots, sh.h_k, sh.h_v, sh.d,
                 max_nodes or max(16, sp.max_seq_nodes), ri.x, ri.ba, ri.parents, ri.node_off,
                 W.slot_map(sp) if sm is None else sm, ri.accepted, lp.conv_w, lp.dt_bias, lp.A)


class GpuPools:
    """Device copies of a layer's pools (the persistent state)."""

    def __init__(self, ssm: np.ndarray, conv_hist: np.ndarray):
        self.ssm = dev(ssm)
        self.conv_hist = dev(conv_hist)


@dataclass
class GpuOut:
    xc: np.ndarray
    win: Optional[np.ndarray]      # None in the compact form
    o: np.ndarray
    replay: np.ndarray
    status: int
    win_ref: Optional[np.ndarray] = None   # [N][3] int32, compact form only


def run_gpu(b: Batch, pools: GpuPools, q_scale: float = 1.0, commit: bool = True,
            x_pad: int = 0, ba_pad: int = 0, replay_pad: int = 0,
            xc_override: Optional[np.ndarray] = None, compact: bool = False,
            chain: bool = False) -> GpuOut:
    """conv -> verify -> commit on the device (pools updated in place); with
    compact=True the windows travel as references (the compact entry points),
    with chain=True verify goes through gdn_chain_verify."""
    C, N, Hv, d = b.C, b.N, b.Hv, b.d
    dm = b.gdims()
    xs = C + x_pad
    xh = np.zeros((max(N, 1), xs), np.float32)
    xh[:N, :C] = b.x
    x = dev(xh)
    bas = 2 * Hv + ba_pad
    bah = np.zeros((max(N, 1), bas), np.float32)
    bah[:N, : 2 * Hv] = b.ba
    ba = dev(bah)
    w, dt, A = dev(b.conv_w), dev(b.dt_bias), dev(b.A)
    par = dev(b.parents if N else np.zeros(1, np.int32))
    off, sm, acc = dev(b.node_off), dev(b.slot_map), dev(b.accepted)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xc = nan_like((max(N, 1), C))
    win = nan_like((max(N, 1), 3, C))
    rs = G.gdn_replay_row_floats(d, d) + replay_pad
    o = nan_like((max(N, 1), Hv, d))
    rep = nan_like((max(N, 1), Hv, rs))
    wref = torch.full((max(N, 1), 3), -99, dtype=torch.int32, device="cuda")
    if compact:
        G.gdn_conv_tree_step_compact(dm, x, xs, w, pools.conv_hist, par, off, sm, xc, wref, status)
    else:
        G.gdn_conv_tree_step(dm, x, xs, w, pools.conv_hist, par, off, sm, xc, win, status)
    xin = xc if xc_override is None else dev(xc_override.astype(np.float32))
    verify = G.gdn_chain_verify if chain else G.gdn_tree_verify
    verify(dm, xin, ba, bas, dt, A, pools.ssm, q_scale, par, off, sm, o, rep, rs, status)
    if commit and compact:
        G.gdn_commit_compact(dm, acc, par, off, sm, rep, rs, x, xs, wref, pools.ssm, pools.conv_hist, status)
    elif commit:
        G.gdn_commit(dm, acc, par, off, sm, rep, rs, win, pools.ssm, pools.conv_hist, status)
    torch.cuda.synchronize()
    return GpuOut(xc.cpu().numpy()[:N], None if compact else win.cpu().numpy()[:N], o.cpu().numpy()[:N],
                  rep.cpu().numpy()[:N, :, : 2 * d + 1], int(status.item()),
                  wref.cpu().numpy()[:N] if compact else None)


@dataclass
class OracleOut:
    xc: np.ndarray
    win: np.ndarray
    o: np.ndarray
    replay: np.ndarray
    ssm: np.ndarray
    conv_hist: np.ndarray


def run_oracle(b: Batch, ssm: np.ndarray, conv_hist: np.ndarray, q_scale: float = 1.0,
               commit: bool = True, xc_override: Optional[np.ndarray] = None) -> OracleOut:
    orc = O.get()
    dm = b.odims()
    rc, xc, win = orc.conv_tree_step(dm, b.x, b.conv_w, conv_hist, b.parents, b.node_off, b.slot_map)
    assert rc == 0, rc
    xin = xc.astype(np.float32) if xc_override is None else xc_override.astype(np.float32)
    rc, o, rep = orc.tree_verify(dm, xin, b.ba, b.dt_bias, b.A, ssm, b.parents, b.node_off,
                                 b.slot_map, q_scale=q_scale)
    assert rc == 0, rc
    ssm2, hist2 = ssm.copy(), conv_hist.copy()
    if commit:
        rc = orc.commit(dm, b.accepted, b.parents, b.node_off, b.slot_map, rep, win, ssm2, hist2)
        assert rc == 0, rc
    return OracleOut(xc, win, o, rep, ssm2, hist2)


def replay_parts(rep: np.ndarray, d: int):
    """The three parts of replay rows [..., 2d + 1]: k^, u, decay."""
    return {"replay_k": rep[..., :d], "replay_u": rep[..., d:2 * d], "replay_decay": rep[..., 2 * d]}


def compare(g: GpuOut, r: OracleOut, tol: float = TOL, check_xc: bool = True):
    """Element-by-element parity; returns the error figures.  The replay rows
    are judged part by part (k^, u, decay), each against its own scale."""
    assert g.status == 0, G.gdn_status_str(g.status)
    errs = {}
    if check_xc:
        errs["xc"] = relerr(g.xc, r.xc)
        if g.win is not None:
            assert np.array_equal(g.win, r.win), "commit windows differ"
    errs["o"] = relerr(g.o, r.o)
    d = g.o.shape[-1] if g.o.size else (g.replay.shape[-1] - 1) // 2
    gp, rp = replay_parts(g.replay, d), replay_parts(r.replay, d)
    for k in gp:
        errs[k] = relerr(gp[k], rp[k])
    for k, v in errs.items():
        assert v <= tol, (k, v)
    return errs


def custom_batch(seed, Hk, Hv, d, sizes, P=None, kind="tree", forest=False, max_nodes=None,
                 accepted=None):
    """A batch of ragged sequences with the given node counts: random trees
    (or chains, kind="chain"; forest=True makes every fifth node a root),
    seeded inputs, the accepted node drawn per sequence unless given."""
    S = len(sizes)
    P = P or 2 * S + 1
    sp = W.Spec(f"edge{seed}", W.Shape(S, P, Hk, Hv, d), "tree", list(sizes), seed)
    lp = W.layer_params(sp)
    sm = W.slot_map(sp)
    off = np.zeros(S + 1, np.int32)
    off[1:] = np.cumsum(sizes)
    N = int(off[-1])
    parents = np.empty(N, np.int32)
    acc = np.empty(S, np.int32)
    for s, ns in enumerate(sizes):
        st = W.Stream(seed, 0, W.TID_TREE, 0, s)
        if kind == "chain":
            par = [i - 1 for i in range(ns)]
        else:
            par = W.random_tree(st, ns, 8 if ns <= 24 else 64, 3)
        if forest:
            par = [-1 if (i % 5 == 0) else p for i, p in enumerate(par)]
        parents[off[s]:off[s + 1]] = par
        acc[s] = -1 if ns == 0 else int(W.Stream(seed, 0, W.TID_ACC, 0, s).randint(1, ns + 1)[0]) - 1
    if accepted is not None:
        acc[:] = accepted
    C = 2 * Hk * d + Hv * d
    x = W.Stream(seed, 0, W.TID_X, 0).normal(N * C).reshape(N, C)
    ba = W.Stream(seed, 0, W.TID_BA, 0).normal(N * 2 * Hv).reshape(N, 2 * Hv)
    b = Batch(S, P, Hk, Hv, d, max_nodes or (16 if max(sizes) <= 16 else 64), x, ba, parents, off, sm,
              acc, lp.conv_w, lp.dt_bias, lp.A)
    return b, lp
