"""Seeded synthetic inputs for the GDN speculative tree-verify step.

This module only draws numbers: token trees, slot maps, accepted nodes and the
raw tensors (projected tokens, gate projections, weights, initial pools).  It
holds none of the method's arithmetic, so the oracle and the CUDA path can both
consume what it produces without sharing any computation.

Random numbers come from SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): a 64-bit counter advanced by the
golden-ratio increment and passed through the published finaliser.  Every
tensor has its own stream, keyed by (seed, layer, tensor id, round, sequence),
so the draw of one tensor never shifts another.  Uniforms use the top 24 bits
of an output; normals use Box-Muller in double precision on two 53-bit
uniforms and are then cast to float32.

The workloads are the five shapes of the GDN verify study:

  0 tiny   - one sequence, H_k = H_v = 2, d = 16, tree parents [-1,0,0,1,2],
             two slots mapped [1], accepted node 3 (path 0 -> 1 -> 3)
  1 chain  - one sequence, H_k = 16, H_v = 32, d = 128, chain of 8 drafts
  2 tree4  - four sequences of 16-node random draft trees, 8-slot pool
  3 stack  - 48 layers, five sequences with {4,8,12,16,16}-node trees,
             H_k = 16, H_v = 48, 16-slot pool per layer
  4 sweep  - 64 sequences in a 128-slot pool, grouped (16/32 heads) or
             non-grouped (32/32 heads), 16-node trees or 64-token chains

Value distributions: pre-conv q, k, v, z ~ N(0, 1); conv weights ~ N(0, 0.25)
(0.25 read as the standard deviation); b, a ~ N(0, 1); dt_bias ~ U(-1, 1);
A = -exp(U(0, ln 16)); initial recurrent state ~ N(0, 0.1); conv history
~ N(0, 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "Shape", "Spec", "LayerParams", "RoundInputs", "spec", "sweep_spec",
    "layer_params", "round_inputs", "slot_map", "Stream", "SPEC_NAMES",
    "SWEEP_VARIANTS",
]

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15

# tensor ids of the per-tensor streams
TID_W, TID_DT, TID_A, TID_STATE, TID_HIST = 1, 2, 3, 4, 5
TID_TREE, TID_X, TID_Z, TID_BA, TID_ACC, TID_SLOT = 6, 7, 8, 9, 10, 11


def _mix64(z: int) -> int:
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_key(*parts: int) -> int:
    """Fold integers into one 64-bit stream key."""
    h = 0x243F6A8885A308D3
    for p in parts:
        h = _mix64((h ^ ((int(p) + _GAMMA) & _MASK)) & _MASK)
    return h


class Stream:
    """A SplitMix64 stream: output i is mix(key + (i + 1) * gamma)."""

    def __init__(self, *key_parts: int):
        self.key = stream_key(*key_parts)
        self.pos = 0

    def raw(self, n: int) -> np.ndarray:
        i = np.arange(self.pos + 1, self.pos + n + 1, dtype=np.uint64)
        self.pos += n
        with np.errstate(over="ignore"):
            return _mix64_np(i * np.uint64(_GAMMA) + np.uint64(self.key))

    def uniform24(self, n: int) -> np.ndarray:
        """U[0, 1) from the top 24 bits (exact in float32)."""
        return (self.raw(n) >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))

    def uniform(self, n: int, lo: float, hi: float) -> np.ndarray:
        return (lo + (hi - lo) * self.uniform24(n)).astype(np.float32)

    def normal(self, n: int, std: float = 1.0) -> np.ndarray:
        z = self.raw(2 * n)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        r = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        return (r * std).astype(np.float32)

    def randint(self, n: int, hi: int) -> np.ndarray:
        """Uniform integers in [0, hi)."""
        u = (self.raw(n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        return np.minimum((u * hi).astype(np.int64), hi - 1)


@dataclass(frozen=True)
class Shape:
    n_seqs: int
    n_slots: int
    h_k: int
    h_v: int
    d: int
    d_conv: int = 4

    @property
    def conv_channels(self) -> int:
        return 2 * self.h_k * self.d + self.h_v * self.d


@dataclass(frozen=True)
class Spec:
    """A workload: shape, per-sequence tree kinds and sizes, seed."""
    name: str
    shape: Shape
    tree_kind: str                 # "fixed" | "tree" | "chain"
    seq_nodes: Sequence[int]       # nodes per sequence
    seed: int
    layers: int = 1
    rounds: int = 1
    fixed_parents: Optional[Sequence[int]] = None
    fixed_slot_map: Optional[Sequence[int]] = None
    fixed_accepted: Optional[Sequence[int]] = None
    max_path: int = 8              # nodes on any root-to-leaf path (trees)
    max_children: int = 3          # branching bound (trees)

    @property
    def n_nodes(self) -> int:
        return int(sum(self.seq_nodes))

    @property
    def max_seq_nodes(self) -> int:
        return int(max(self.seq_nodes)) if len(self.seq_nodes) else 0


SWEEP_VARIANTS = ("grouped_tree16", "grouped_chain64", "nongrouped_tree16", "nongrouped_chain64")


def sweep_spec(variant: str, rounds: int = 100) -> Spec:
    """Throughput sweep: 64 sequences in a 128-slot pool, d = 128."""
    grouped = variant.startswith("grouped")
    chain = variant.endswith("chain64")
    shape = Shape(n_seqs=64, n_slots=128, h_k=16 if grouped else 32, h_v=32, d=128)
    return Spec(name=f"sweep_{variant}", shape=shape,
                tree_kind="chain" if chain else "tree",
                seq_nodes=[64 if chain else 16] * 64, seed=4, rounds=rounds)


def spec(index: int, variant: str = "grouped_tree16") -> Spec:
    if index == 0:
        return Spec("tiny", Shape(1, 2, 2, 2, 16), "fixed", [5], seed=0,
                    fixed_parents=[-1, 0, 0, 1, 2], fixed_slot_map=[1],
                    fixed_accepted=[3])
    if index == 1:
        return Spec("chain8", Shape(1, 2, 16, 32, 128), "chain", [8], seed=1,
                    rounds=32, fixed_slot_map=[1])
    if index == 2:
        return Spec("tree4x16", Shape(4, 8, 16, 32, 128), "tree", [16] * 4,
                    seed=2, rounds=32)
    if index == 3:
        return Spec("stack48", Shape(5, 16, 16, 48, 128), "tree",
                    [4, 8, 12, 16, 16], seed=3, layers=48, rounds=10)
    if index == 4:
        return sweep_spec(variant)
    raise ValueError(f"no workload {index}")


SPEC_NAMES = {0: "tiny", 1: "chain8", 2: "tree4x16", 3: "stack48", 4: "sweep"}


@dataclass
class LayerParams:
    conv_w: np.ndarray      # [C][4] float32
    dt_bias: np.ndarray     # [H_v] float32
    A: np.ndarray           # [H_v] float32, negative
    ssm: np.ndarray         # [P][H_v][d][d] float32, row = value index
    conv_hist: np.ndarray   # [P][3][C] float32, tap 0 oldest


@dataclass
class RoundInputs:
    parents: np.ndarray     # [N] int32, local to the sequence, -1 = root
    node_off: np.ndarray    # [S + 1] int32
    x: np.ndarray           # [N][C] float32, q | k | v channels
    z: np.ndarray           # [N][H_v * d] float32 (drawn, not consumed)
    ba: np.ndarray          # [N][2 H_v] float32, b then a
    accepted: np.ndarray    # [S] int32 in {-1} U [0, N_s)


def layer_params(sp: Spec, layer: int = 0, with_pools: bool = True) -> LayerParams:
    sh = sp.shape
    C = sh.conv_channels
    w = Stream(sp.seed, layer, TID_W).normal(C * sh.d_conv, 0.25).reshape(C, sh.d_conv)
    dt = Stream(sp.seed, layer, TID_DT).uniform(sh.h_v, -1.0, 1.0)
    A = (-np.exp(Stream(sp.seed, layer, TID_A).uniform24(sh.h_v) * math.log(16.0))).astype(np.float32)
    if with_pools:
        ssm = Stream(sp.seed, layer, TID_STATE).normal(
            sh.n_slots * sh.h_v * sh.d * sh.d, 0.1).reshape(sh.n_slots, sh.h_v, sh.d, sh.d)
        hist = Stream(sp.seed, layer, TID_HIST).normal(
            sh.n_slots * (sh.d_conv - 1) * C, 1.0).reshape(sh.n_slots, sh.d_conv - 1, C)
    else:
        ssm = hist = None
    return LayerParams(w, dt, A, ssm, hist)


def slot_map(sp: Spec) -> np.ndarray:
    if sp.fixed_slot_map is not None:
        return np.asarray(sp.fixed_slot_map, dtype=np.int32)
    P = sp.shape.n_slots
    perm = list(range(P))
    st = Stream(sp.seed, 0, TID_SLOT)
    r = st.randint(P, P)
    for i in range(P - 1, 0, -1):               # Fisher-Yates
        j = int(r[i]) % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    return np.asarray(perm[: sp.shape.n_seqs], dtype=np.int32)


def random_tree(st: Stream, n: int, max_path: int, max_children: int) -> List[int]:
    """Parents of a random draft tree; node 0 is the root, order is topological."""
    parents = [-1]
    depth = [1]
    kids = [0]
    u = st.uniform24(max(n, 1))
    for i in range(1, n):
        cand = [j for j in range(i) if depth[j] < max_path and kids[j] < max_children]
        p = cand[min(int(u[i] * len(cand)), len(cand) - 1)]
        parents.append(p)
        depth.append(depth[p] + 1)
        kids.append(0)
        kids[p] += 1
    return parents


def round_inputs(sp: Spec, layer: int = 0, rnd: int = 0, with_x: bool = True) -> RoundInputs:
    sh = sp.shape
    C = sh.conv_channels
    S = sh.n_seqs
    off = np.zeros(S + 1, dtype=np.int32)
    off[1:] = np.cumsum(np.asarray(sp.seq_nodes, dtype=np.int64))
    N = int(off[-1])
    parents = np.empty(N, dtype=np.int32)
    acc = np.empty(S, dtype=np.int32)
    # trees and acceptances are shared by all layers of a round: the draft tree
    # is one per sequence, and every layer commits the same accepted node
    for s in range(S):
        ns = int(sp.seq_nodes[s])
        st = Stream(sp.seed, 0, TID_TREE, rnd, s)
        if sp.tree_kind == "fixed":
            par = list(sp.fixed_parents)
        elif sp.tree_kind == "chain":
            par = [i - 1 for i in range(ns)]
        else:
            par = random_tree(st, ns, sp.max_path, sp.max_children)
        parents[off[s]:off[s + 1]] = par
        if sp.fixed_accepted is not None:
            acc[s] = sp.fixed_accepted[s]
        else:
            ua = Stream(sp.seed, 0, TID_ACC, rnd, s)
            if sp.tree_kind == "chain":
                acc[s] = int(ua.randint(1, ns + 1)[0]) - 1     # m ~ U{0..N_s}
            else:
                acc[s] = int(ua.randint(1, ns)[0])             # uniform node
    if with_x:
        x = Stream(sp.seed, layer, TID_X, rnd).normal(N * C).reshape(N, C)
        z = Stream(sp.seed, layer, TID_Z, rnd).normal(N * sh.h_v * sh.d).reshape(N, sh.h_v * sh.d)
    else:
        x = z = None
    ba = Stream(sp.seed, layer, TID_BA, rnd).normal(N * 2 * sh.h_v).reshape(N, 2 * sh.h_v)
    return RoundInputs(parents, off, x, z, ba, acc)


def subset(sp: Spec, ri: RoundInputs, seqs: Sequence[int]) -> RoundInputs:
    """The same round restricted to some sequences (sequences are independent)."""
    rows = []
    off = [0]
    for s in seqs:
        a, b = int(ri.node_off[s]), int(ri.node_off[s + 1])
        rows.extend(range(a, b))
        off.append(off[-1] + (b - a))
    rows = np.asarray(rows, dtype=np.int64)
    pick = lambda t: None if t is None else np.ascontiguousarray(t[rows])
    return RoundInputs(np.ascontiguousarray(ri.parents[rows]), np.asarray(off, dtype=np.int32),
                       pick(ri.x), pick(ri.z), pick(ri.ba),
                       np.ascontiguousarray(ri.accepted[list(seqs)]))
