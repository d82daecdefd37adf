"""Pins of the oracle: each check_* runs the oracle and compares it with
something other than itself - a hand-worked example, a library routine over
the explicit column sequence, the literal matrix form of the gated delta rule,
a closed form or a structural invariant.  Each raises AssertionError on a
mismatch.  The mutation test runs every check against deliberately broken
oracle builds and requires each break to fail at least one check.
"""
from __future__ import annotations

import json
import os

import numpy as np

import gdn_workloads as W
import oracle as O
from pins_np import (conv_path, decode_path, gates, head_slices, l2n, path_to, relerr)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# closed forms and library formulations agree with a double-precision oracle
# to rounding: 1e-9 leaves room for different summation orders over d <= 32
TIGHT = 1e-9


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _dims(g):
    return O.Dims(**g["dims"])


def make_case(seed, S, h_k, h_v, d, seq_nodes, kind="tree", P=None, rnd=0):
    P = P if P is not None else max(2, 2 * S)
    sp = W.Spec(f"pin{seed}", W.Shape(S, P, h_k, h_v, d), kind, list(seq_nodes), seed)
    lp = W.layer_params(sp)
    ri = W.round_inputs(sp, rnd=rnd)
    sm = W.slot_map(sp)
    dm = O.Dims(S, sp.n_nodes, P, h_k, h_v, d)
    return sp, dm, lp, ri, sm


def _verify_inputs(orc, dm, lp, ri, sm):
    rc, xc, win = orc.conv_tree_step(dm, ri.x, lp.conv_w, lp.conv_hist, ri.parents, ri.node_off, sm)
    assert rc == 0, rc
    return xc.astype(np.float32), win


# ------------------------------------------------------------------ conv ----
def check_hand_conv(orc):
    g = _load("hand_conv_d1.json")
    dm = _dims(g)
    rc, xc, win = orc.conv_tree_step(dm, np.array(g["x"], np.float32), np.array(g["conv_w"], np.float32),
                                     np.array(g["conv_hist"], np.float32), g["parents"], g["node_off"],
                                     g["slot_map"])
    assert rc == 0
    assert np.max(np.abs(xc - np.array(g["expected_xc"]))) <= g["tolerance_abs"], xc
    assert np.array_equal(win[:, :, 0], np.array(g["expected_win_channel0"], np.float32)), win[:, :, 0]
    assert np.array_equal(win[:, :, 1], np.array(g["expected_win_channel1"], np.float32)), win[:, :, 1]


def check_conv_tree_is_path_correlation(orc, seed=11):
    """Every node's conv output and window equal the library cross-correlation
    over the explicit column sequence history ++ root..node tokens."""
    sp, dm, lp, ri, sm = make_case(seed, 3, 2, 4, 16, [12, 7, 1], P=5)
    rc, xc, win = orc.conv_tree_step(dm, ri.x, lp.conv_w, lp.conv_hist, ri.parents, ri.node_off, sm)
    assert rc == 0
    for s in range(dm.n_seqs):
        n0, n1 = int(ri.node_off[s]), int(ri.node_off[s + 1])
        par = ri.parents[n0:n1]
        for i in range(n1 - n0):
            path = path_to(par, i)
            _, act, w3 = conv_path(lp.conv_hist[sm[s]], ri.x[n0:n1][path], lp.conv_w)
            assert relerr(xc[n0 + i], act[-1]) <= TIGHT, (s, i)
            assert np.array_equal(win[n0 + i], w3.astype(np.float32)), (s, i)


def check_conv_chain_is_correlation(orc, seed=12):
    sp, dm, lp, ri, sm = make_case(seed, 1, 1, 2, 16, [9], kind="chain", P=3)
    rc, xc, win = orc.conv_tree_step(dm, ri.x, lp.conv_w, lp.conv_hist, ri.parents, ri.node_off, sm)
    assert rc == 0
    _, act, _ = conv_path(lp.conv_hist[sm[0]], ri.x, lp.conv_w)
    assert relerr(xc, act) <= TIGHT


# ------------------------------------------------------------ recurrence ----
def _hand_recurrence(orc, which):
    g = _load("hand_recurrence_d2.json")
    dm = _dims(g)
    case = g[which]
    ssm = np.array(g["ssm"], np.float32)
    rc, o, rep = orc.tree_verify(dm, np.array(g["xc"], np.float32), np.array(g["ba"], np.float32),
                                 g["dt_bias"], g["A"], ssm, case["parents"], g["node_off"],
                                 g["slot_map"])
    assert rc == 0
    tol = g["tolerance_abs"]
    assert np.max(np.abs(o - np.array(case["expected_o"]))) <= tol, o
    assert np.max(np.abs(rep[:, :, 2:4] - np.array(case["expected_u"]))) <= tol, rep
    return g, dm, ssm, rep


def check_hand_recurrence(orc):
    g, dm, ssm, rep = _hand_recurrence(orc, "chain")
    assert np.max(np.abs(rep[:, 0, 4] - np.array(g["chain"]["expected_decay"]))) <= 1e-15
    for acc, key in ((1, "expected_state_after_commit_1"), (0, "expected_state_after_commit_0")):
        S = ssm.copy()
        hist = np.zeros((1, 3, 6), np.float32)
        win = np.zeros((2, 3, 6), np.float32)
        rc = orc.commit(dm, [acc], g["chain"]["parents"], g["node_off"], g["slot_map"], rep, win, S, hist)
        assert rc == 0
        assert np.max(np.abs(S[0, 0] - np.array(g["chain"][key]))) <= g["tolerance_abs"], S
    _hand_recurrence(orc, "tree")


def check_chain_is_sequential_decode(orc, seed=21):
    """A chain verify equals token-by-token decode in the literal matrix form."""
    sp, dm, lp, ri, sm = make_case(seed, 1, 2, 4, 16, [8], kind="chain", P=3)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    assert rc == 0
    for h in range(dm.h_v):
        _, outs = decode_path(lp.ssm[sm[0], h], xc, ri.ba, lp.dt_bias[h], lp.A[h],
                              dm.h_k, dm.h_v, dm.d, h)
        assert relerr(o[:, h], outs) <= TIGHT, h


def check_tree_is_union_of_chains(orc, seed=22):
    sp, dm, lp, ri, sm = make_case(seed, 2, 2, 4, 16, [14, 9], P=4)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    assert rc == 0
    for s in range(dm.n_seqs):
        n0, n1 = int(ri.node_off[s]), int(ri.node_off[s + 1])
        par = ri.parents[n0:n1]
        for i in range(n1 - n0):
            path = [n0 + j for j in path_to(par, i)]
            for h in range(dm.h_v):
                _, outs = decode_path(lp.ssm[sm[s], h], xc[path], ri.ba[path], lp.dt_bias[h],
                                      lp.A[h], dm.h_k, dm.h_v, dm.d, h)
                assert relerr(o[n0 + i, h], outs[-1]) <= TIGHT, (s, i, h)


def check_beta_zero_closed_form(orc, seed=23):
    """beta = 0: nothing is written, o_t = (prod of decays on the path) S0 q_t."""
    sp, dm, lp, ri, sm = make_case(seed, 1, 1, 2, 16, [10], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    ba = ri.ba.copy()
    ba[:, : dm.h_v] = -1e30                         # sigmoid(-1e30) = 0 exactly
    rc, o, rep = orc.tree_verify(dm, xc, ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    assert rc == 0
    for h in range(dm.h_v):
        qs, ks, vs = head_slices(dm.h_k, dm.h_v, dm.d, h)
        S0 = lp.ssm[sm[0], h].astype(np.float64)
        for i in range(dm.n_nodes):
            gam = 1.0
            for j in path_to(ri.parents, i):
                gam *= gates(ba[j, h], ba[j, dm.h_v + h], lp.dt_bias[h], lp.A[h])[1]
            assert relerr(o[i, h], gam * (S0 @ l2n(xc[i, qs]))) <= TIGHT, (h, i)
            assert np.all(rep[i, h, dm.d: 2 * dm.d] == 0.0)


def check_zero_state_single_node(orc, seed=24):
    """S0 = 0, one node: o = beta (k_hat . q_hat) v and u = beta v."""
    sp, dm, lp, ri, sm = make_case(seed, 1, 2, 4, 32, [1], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    ssm = np.zeros_like(lp.ssm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, ssm, ri.parents, ri.node_off, sm,
                                 q_scale=0.5)
    assert rc == 0
    for h in range(dm.h_v):
        qs, ks, vs = head_slices(dm.h_k, dm.h_v, dm.d, h)
        beta, decay = gates(ri.ba[0, h], ri.ba[0, dm.h_v + h], lp.dt_bias[h], lp.A[h])
        v = xc[0, vs].astype(np.float64)
        assert relerr(o[0, h], 0.5 * beta * np.dot(l2n(xc[0, ks]), l2n(xc[0, qs])) * v) <= TIGHT
        assert relerr(rep[0, h, dm.d: 2 * dm.d], beta * v) <= TIGHT
        assert abs(rep[0, h, 2 * dm.d] - decay) <= TIGHT * decay


def check_gate_special_values(orc):
    """b = 0 -> beta = 1/2; a + dt_bias = 0 with A = -1 -> decay = 1/2."""
    sp, dm, lp, ri, sm = make_case(25, 1, 1, 2, 16, [1], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    ba = np.zeros_like(ri.ba)
    ba[0, dm.h_v:] = [0.25, -0.75]                 # a
    dt = np.array([-0.25, 0.75], np.float32)       # a + dt_bias = 0
    A = np.array([-1.0, -1.0], np.float32)
    rc, o, rep = orc.tree_verify(dm, xc, ba, dt, A, np.zeros_like(lp.ssm), ri.parents, ri.node_off, sm)
    assert rc == 0
    for h in range(2):
        assert abs(rep[0, h, 2 * dm.d] - 0.5) <= 1e-15
        v = xc[0, head_slices(1, 2, 16, h)[2]].astype(np.float64)
        assert np.max(np.abs(rep[0, h, dm.d: 2 * dm.d] - 0.5 * v)) <= 1e-15


def check_gates_match_library(orc, seed=26):
    sp, dm, lp, ri, sm = make_case(seed, 2, 2, 4, 16, [6, 5], P=4)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    assert rc == 0
    for t in range(dm.n_nodes):
        for h in range(dm.h_v):
            _, decay = gates(ri.ba[t, h], ri.ba[t, dm.h_v + h], lp.dt_bias[h], lp.A[h])
            assert abs(rep[t, h, 2 * dm.d] - decay) <= TIGHT * decay


def check_l2norm_property(orc, seed=27):
    """k_hat is k scaled to norm sqrt(|k|^2 / (|k|^2 + 1e-6))."""
    sp, dm, lp, ri, sm = make_case(seed, 1, 2, 4, 16, [4], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    assert rc == 0
    for t in range(dm.n_nodes):
        for h in range(dm.h_v):
            k = xc[t, head_slices(dm.h_k, dm.h_v, dm.d, h)[1]].astype(np.float64)
            kh = rep[t, h, : dm.d]
            n2 = np.dot(k, k)
            assert abs(np.dot(kh, kh) - n2 / (n2 + 1e-6)) <= 1e-12
            assert np.max(np.abs(kh * np.linalg.norm(k) - k * np.linalg.norm(kh))) <= 1e-9


def check_sibling_independence(orc, seed=28):
    """Appending a branch changes no existing node's output (bit for bit)."""
    sp, dm, lp, ri, sm = make_case(seed, 1, 2, 4, 16, [9], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o1, r1 = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    par2 = np.concatenate([ri.parents, [0, 9, 2]]).astype(np.int32)
    extra = W.Stream(seed, 0, 99).normal(3 * xc.shape[1]).reshape(3, -1)
    xc2 = np.concatenate([xc, extra]).astype(np.float32)
    ba2 = np.concatenate([ri.ba, W.Stream(seed, 0, 98).normal(3 * 2 * dm.h_v).reshape(3, -1)])
    dm2 = O.Dims(1, 12, dm.n_slots, dm.h_k, dm.h_v, dm.d)
    rc2, o2, r2 = orc.tree_verify(dm2, xc2, ba2, lp.dt_bias, lp.A, lp.ssm, par2, [0, 12], sm)
    assert rc == 0 and rc2 == 0
    assert np.array_equal(o1, o2[:9]) and np.array_equal(r1, r2[:9])


def check_grouped_mapping(orc, seed=29):
    """Value head h reads k-head floor(h / G): equal to a non-grouped run whose
    q/k channels of head h are copies of k-head floor(h / G)."""
    sp, dm, lp, ri, sm = make_case(seed, 1, 2, 6, 16, [7], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    d, Hk, Hv = dm.d, dm.h_k, dm.h_v
    q = xc[:, : Hk * d].reshape(-1, Hk, d)
    k = xc[:, Hk * d: 2 * Hk * d].reshape(-1, Hk, d)
    v = xc[:, 2 * Hk * d:]
    idx = np.arange(Hv) // (Hv // Hk)
    xc_flat = np.concatenate([q[:, idx].reshape(len(xc), -1), k[:, idx].reshape(len(xc), -1), v], axis=1)
    dm1 = O.Dims(1, dm.n_nodes, dm.n_slots, Hv, Hv, d)
    rc1, o1, rep1 = orc.tree_verify(dm1, xc_flat, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents,
                                    ri.node_off, sm)
    assert rc == 0 and rc1 == 0
    assert np.array_equal(o, o1) and np.array_equal(rep, rep1)


def check_q_scale_linear(orc, seed=30):
    sp, dm, lp, ri, sm = make_case(seed, 1, 1, 1, 16, [5], P=2)
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o1, r1 = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    rc, o2, r2 = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm,
                                 q_scale=0.25)
    assert np.max(np.abs(o2 - 0.25 * o1)) <= 1e-15 * np.max(np.abs(o1)) + 1e-300
    assert np.array_equal(r1, r2)


def check_verify_leaves_pool(orc, seed=31):
    sp, dm, lp, ri, sm = make_case(seed, 2, 2, 4, 16, [5, 6], P=4)
    ssm = lp.ssm.copy()
    xc, _ = _verify_inputs(orc, dm, lp, ri, sm)
    orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, ssm, ri.parents, ri.node_off, sm)
    assert np.array_equal(ssm, lp.ssm)


# ---------------------------------------------------------------- commit ----
def check_commit_equals_rerun(orc, seed=41):
    """Commit of node a leaves each head's slot at the state obtained by
    decoding the root..a tokens from the old state; the history becomes the
    last three raw columns of that path; other slots do not move."""
    sp, dm, lp, ri, sm = make_case(seed, 3, 2, 4, 16, [10, 8, 5], P=6)
    xc, win = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    acc = np.array([7, -1, 3], np.int32)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    assert orc.commit(dm, acc, ri.parents, ri.node_off, sm, rep, win, ssm, hist) == 0
    for s in range(dm.n_seqs):
        n0, n1 = int(ri.node_off[s]), int(ri.node_off[s + 1])
        slot = sm[s]
        if acc[s] < 0:
            assert np.array_equal(ssm[slot], lp.ssm[slot]) and np.array_equal(hist[slot], lp.conv_hist[slot])
            continue
        path = [n0 + j for j in path_to(ri.parents[n0:n1], int(acc[s]))]
        for h in range(dm.h_v):
            S, _ = decode_path(lp.ssm[slot, h], xc[path], ri.ba[path], lp.dt_bias[h], lp.A[h],
                               dm.h_k, dm.h_v, dm.d, h)
            # the slot stores float32: one rounding of the committed state
            assert relerr(ssm[slot, h], S) <= 1e-6, (s, h)
        _, _, w3 = conv_path(lp.conv_hist[slot], ri.x[path], lp.conv_w)
        assert np.array_equal(hist[slot], w3.astype(np.float32))
    untouched = sorted(set(range(dm.n_slots)) - {int(sm[s]) for s in range(dm.n_seqs) if acc[s] >= 0})
    assert np.array_equal(ssm[untouched], lp.ssm[untouched])
    assert np.array_equal(hist[untouched], lp.conv_hist[untouched])


def check_commit_zero_length_identity(orc, seed=42):
    sp, dm, lp, ri, sm = make_case(seed, 2, 2, 4, 16, [6, 4], P=4)
    xc, win = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    assert orc.commit(dm, [-1, -1], ri.parents, ri.node_off, sm, rep, win, ssm, hist) == 0
    assert np.array_equal(ssm, lp.ssm) and np.array_equal(hist, lp.conv_hist)


def check_multi_round_equals_stream_decode(orc, seed=43, rounds=4):
    """Rounds of conv + verify + commit equal a plain decode of the stream of
    accepted tokens: same outputs on the accepted nodes, same final state and
    history."""
    S, Hk, Hv, d = 2, 2, 4, 16
    sp = W.Spec("pinmr", W.Shape(S, 4, Hk, Hv, d), "tree", [9, 6], seed, rounds=rounds)
    lp = W.layer_params(sp)
    sm = W.slot_map(sp)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    streams = [[] for _ in range(S)]        # (x row, ba row, o of the node) per accepted token
    for r in range(rounds):
        ri = W.round_inputs(sp, rnd=r)
        dm = O.Dims(S, sp.n_nodes, 4, Hk, Hv, d)
        rc, xc, win = orc.conv_tree_step(dm, ri.x, lp.conv_w, hist, ri.parents, ri.node_off, sm)
        rc2, o, rep = orc.tree_verify(dm, xc.astype(np.float32), ri.ba, lp.dt_bias, lp.A, ssm,
                                      ri.parents, ri.node_off, sm)
        assert rc == 0 and rc2 == 0
        assert orc.commit(dm, ri.accepted, ri.parents, ri.node_off, sm, rep, win, ssm, hist) == 0
        for s in range(S):
            n0, n1 = int(ri.node_off[s]), int(ri.node_off[s + 1])
            if ri.accepted[s] >= 0:
                for j in path_to(ri.parents[n0:n1], int(ri.accepted[s])):
                    streams[s].append((ri.x[n0 + j], ri.ba[n0 + j], o[n0 + j]))
    for s in range(S):
        xs = np.array([e[0] for e in streams[s]])
        bas = np.array([e[1] for e in streams[s]])
        os_ = np.array([e[2] for e in streams[s]])
        _, act, w3 = conv_path(lp.conv_hist[sm[s]], xs, lp.conv_w)
        assert np.array_equal(hist[sm[s]], w3.astype(np.float32))
        for h in range(Hv):
            Sfin, outs = decode_path(lp.ssm[sm[s], h], act.astype(np.float32), bas, lp.dt_bias[h],
                                     lp.A[h], Hk, Hv, d, h)
            # float32 storage of xc and of the state between rounds
            assert relerr(os_[:, h], outs) <= 2e-5, (s, h)
            assert relerr(ssm[sm[s], h], Sfin) <= 2e-5, (s, h)


def check_preflight_rejects(orc, seed=44):
    """Every failed check returns its code and leaves both pools bit-identical."""
    sp, dm, lp, ri, sm = make_case(seed, 3, 2, 4, 16, [5, 5, 5], P=6)
    xc, win = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    cases = []
    cases.append(("dup", [1, 2, 3], ri.parents, [sm[0], sm[1], sm[0]], O.DUP_SLOT))
    cases.append(("acc_hi", [1, 5, 3], ri.parents, sm, O.BAD_ACCEPTED))
    cases.append(("acc_lo", [1, -2, 3], ri.parents, sm, O.BAD_ACCEPTED))
    bad = ri.parents.copy(); bad[5 + 3] = 3                        # self parent
    cases.append(("self_parent", [1, 3, 0], bad, sm, O.BAD_PARENT))
    cases.append(("slot_range", [1, 2, 3], ri.parents, [sm[0], 6, sm[2]], O.BAD_SLOT))
    for name, acc, par, smap, code in cases:
        ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
        got = orc.commit(dm, acc, par, ri.node_off, smap, rep, win, ssm, hist)
        assert got == code, (name, got)
        assert np.array_equal(ssm, lp.ssm) and np.array_equal(hist, lp.conv_hist), name
    # a duplicated slot is fine when one of the two sequences commits nothing
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    assert orc.commit(dm, [1, -1, 2], ri.parents, ri.node_off, [sm[0], sm[0], sm[2]], rep, win, ssm,
                      hist) == 0


def check_tiny_regression(orc):
    """The oracle's own outputs on the tiny workload, frozen (make_tiny_golden.py)."""
    path = os.path.join(GOLDEN, "tiny_oracle.json")
    with open(path) as f:
        g = json.load(f)
    sp = W.spec(0)
    lp, ri, sm = W.layer_params(sp), W.round_inputs(sp), W.slot_map(sp)
    sh = sp.shape
    dm = O.Dims(sh.n_seqs, sp.n_nodes, sh.n_slots, sh.h_k, sh.h_v, sh.d)
    rc, xc, win = orc.conv_tree_step(dm, ri.x, lp.conv_w, lp.conv_hist, ri.parents, ri.node_off, sm)
    rc2, o, rep = orc.tree_verify(dm, xc.astype(np.float32), ri.ba, lp.dt_bias, lp.A, lp.ssm,
                                  ri.parents, ri.node_off, sm)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    rc3 = orc.commit(dm, ri.accepted, ri.parents, ri.node_off, sm, rep, win, ssm, hist)
    assert rc == rc2 == rc3 == 0
    assert relerr(xc, np.array(g["xc"])) <= 1e-12
    assert relerr(o, np.array(g["o"])) <= 1e-12
    assert relerr(rep, np.array(g["replay"])) <= 1e-12
    assert relerr(ssm[sm[0]], np.array(g["committed_state"])) <= 1e-7


# ------------------------------------------------------- compact windows ----
def check_hand_window_refs(orc):
    g = _load("hand_window_refs.json")
    rc, refs = orc.window_refs(_dims(g), g["parents"], g["node_off"])
    assert rc == 0
    assert refs.tolist() == g["expected_refs"], refs.tolist()


def check_window_refs_gather_windows(orc, seed=51):
    """Gathering x rows and the slot's history columns through the references
    gives the conv step's commit windows exactly (trees with several roots,
    chains, a one-node sequence)."""
    for kind, sizes in (("tree", [12, 1, 7]), ("chain", [9, 2])):
        sp, dm, lp, ri, sm = make_case(seed, len(sizes), 1, 2, 16, sizes, kind=kind)
        parents = ri.parents.copy()
        if kind == "tree":
            for s in range(dm.n_seqs):
                n0 = int(ri.node_off[s])
                for i in range(5, sizes[s], 5):
                    parents[n0 + i] = -1
        rc, xc, win = orc.conv_tree_step(dm, ri.x, lp.conv_w, lp.conv_hist, parents, ri.node_off, sm)
        assert rc == 0
        rc, refs = orc.window_refs(dm, parents, ri.node_off)
        assert rc == 0
        for s in range(dm.n_seqs):
            for n in range(int(ri.node_off[s]), int(ri.node_off[s + 1])):
                for j in range(dm.d_conv - 1):
                    r = int(refs[n, j])
                    got = ri.x[r] if r >= 0 else lp.conv_hist[sm[s], -1 - r]
                    assert np.array_equal(got, win[n, j]), (kind, s, n, j, r)


def check_commit_compact_equals_commit(orc, seed=52):
    """The commit through references leaves both pools bit-identical to the
    commit with materialised windows."""
    sp, dm, lp, ri, sm = make_case(seed, 3, 2, 4, 16, [10, 8, 5], P=6)
    xc, win = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o, rep = orc.tree_verify(dm, xc, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm)
    rc, refs = orc.window_refs(dm, ri.parents, ri.node_off)
    acc = np.array([0, -1, 4], np.int32)
    ssm1, hist1 = lp.ssm.copy(), lp.conv_hist.copy()
    ssm2, hist2 = lp.ssm.copy(), lp.conv_hist.copy()
    assert orc.commit(dm, acc, ri.parents, ri.node_off, sm, rep, win, ssm1, hist1) == 0
    assert orc.commit_compact(dm, acc, ri.parents, ri.node_off, sm, rep, ri.x, refs, ssm2, hist2) == 0
    assert np.array_equal(ssm1, ssm2) and np.array_equal(hist1, hist2)
    assert not np.array_equal(hist2, lp.conv_hist)


# ------------------------------------------------------- gated RMS norm ----
def check_hand_gated_norm(orc):
    g = _load("hand_gated_norm.json")
    dm = O.Dims(1, 1, 1, 1, 1, 2)
    for c in g["cases"]:
        rc, y = orc.gated_rmsnorm(dm, np.array([[c["o"]]], np.float32), np.array([c["z"]], np.float32),
                                  np.array(c["w"], np.float32), c["eps"], c["gate_mode"])
        assert rc == 0
        assert np.max(np.abs(y[0, 0] - np.array(c["expected_y"]))) <= g["tolerance_abs"], (c, y)


def _norm_case(seed, N=5, Hv=3, d=16):
    st = W.Stream(seed, 0, 99)
    o = st.normal(N * Hv * d).reshape(N, Hv, d)
    z = st.normal(N * Hv * d, 2.0).reshape(N, Hv * d)
    w = st.normal(d, 0.5)
    return O.Dims(1, N, 1, 1, Hv, d), o, z, w


def check_gated_norm_constant_head(orc, seed=61):
    """A head whose outputs all equal c normalises to c / sqrt(c^2 + eps)."""
    dm, o, z, w = _norm_case(seed)
    o[:] = np.float32(-1.5)
    eps = 0.25
    for mode, gate in ((0, lambda v: v / (1 + np.exp(-v))), (1, lambda v: 1 / (1 + np.exp(-v)))):
        rc, y = orc.gated_rmsnorm(dm, o, z, w, eps, mode)
        want = (-1.5 / np.sqrt(2.25 + eps)) * w.astype(np.float64) * gate(z.astype(np.float64).reshape(y.shape))
        assert relerr(y, want) <= TIGHT


def check_gated_norm_modes_relation(orc, seed=62):
    """SiLU(z) = z sigmoid(z), so the SiLU-gated output is z times the
    sigmoid-gated one, element by element."""
    dm, o, z, w = _norm_case(seed)
    rc0, ys = orc.gated_rmsnorm(dm, o, z, w, 1e-6, 0)
    rc1, yg = orc.gated_rmsnorm(dm, o, z, w, 1e-6, 1)
    assert rc0 == rc1 == 0
    assert relerr(ys, z.astype(np.float64).reshape(yg.shape) * yg) <= TIGHT


def check_gated_norm_scale_invariance(orc, seed=63):
    """With eps = 0 the norm removes any power-of-two scale of o exactly."""
    dm, o, z, w = _norm_case(seed)
    rc, y1 = orc.gated_rmsnorm(dm, o, z, w, 0.0, 1)
    rc, y2 = orc.gated_rmsnorm(dm, (o * np.float32(2.0 ** 20)).astype(np.float32), z, w, 0.0, 1)
    assert relerr(y1, y2) <= TIGHT
    rc, y3 = orc.gated_rmsnorm(dm, o, z, w, 0.0, 2)
    assert rc != 0


# ---------------------------------------------------------- decode step ----
def _decode_case(seed, S=3, Hk=2, Hv=4, d=16, P=5):
    sp = W.Spec(f"dec{seed}", W.Shape(S, P, Hk, Hv, d), "chain", [1] * S, seed)
    lp = W.layer_params(sp)
    ri = W.round_inputs(sp)
    sm = W.slot_map(sp)
    return sp, O.Dims(S, S, P, Hk, Hv, d), lp, ri, sm


def check_decode_step_is_one_node_tree_committed(orc, seed=71):
    """A decode step equals the tree path on one-node trees with the node
    accepted: same xc and o, same state and history afterwards."""
    sp, dm, lp, ri, sm = _decode_case(seed)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    rc, xc, o = orc.decode_step(dm, ri.x, lp.conv_w, hist, ri.ba, lp.dt_bias, lp.A, ssm, sm, q_scale=0.5)
    assert rc == 0
    xcf, win = _verify_inputs(orc, dm, lp, ri, sm)
    rc, o2, rep = orc.tree_verify(dm, xcf, ri.ba, lp.dt_bias, lp.A, lp.ssm, ri.parents, ri.node_off, sm,
                                  q_scale=0.5)
    ssm2, hist2 = lp.ssm.copy(), lp.conv_hist.copy()
    assert orc.commit(dm, np.zeros(dm.n_seqs, np.int32), ri.parents, ri.node_off, sm, rep, win, ssm2, hist2) == 0
    rc, xc2, _ = orc.conv_tree_step(dm, ri.x, lp.conv_w, lp.conv_hist, ri.parents, ri.node_off, sm)
    assert relerr(xc, xc2) <= TIGHT
    assert relerr(o, o2) <= TIGHT
    assert np.array_equal(hist, hist2)
    # the committed state rounds once to fp32 on both paths
    assert relerr(ssm, ssm2) <= 1e-6


def check_decode_steps_match_literal_decode(orc, seed=72, steps=5):
    """Several decode steps equal the literal matrix form S (I - beta k k^T)
    + beta v k^T applied token by token, with the conv as a correlation over
    the history and the tokens so far."""
    sp, dm, lp, ri, sm = _decode_case(seed, S=2)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    xs, bas, outs = [], [], []
    for r in range(steps):
        ri = W.round_inputs(sp, 0, r)
        rc, xc, o = orc.decode_step(dm, ri.x, lp.conv_w, hist, ri.ba, lp.dt_bias, lp.A, ssm, sm)
        assert rc == 0
        xs.append(ri.x)
        bas.append(ri.ba)
        outs.append(o)
    for s in range(dm.n_seqs):
        slot = sm[s]
        toks = np.stack([x[s] for x in xs])
        _, act, w3 = conv_path(lp.conv_hist[slot], toks, lp.conv_w)
        assert np.array_equal(hist[slot], w3.astype(np.float32))
        for h in range(dm.h_v):
            S, o = decode_path(lp.ssm[slot, h], act.astype(np.float32), np.stack([b[s] for b in bas]),
                               lp.dt_bias[h], lp.A[h], dm.h_k, dm.h_v, dm.d, h)
            assert relerr(np.stack([out[s, h] for out in outs]), o) <= 1e-5, (s, h)
            assert relerr(ssm[slot, h], S) <= 1e-5, (s, h)


def check_decode_step_rejects_shared_slots(orc, seed=73):
    sp, dm, lp, ri, sm = _decode_case(seed)
    sm = sm.copy()
    sm[2] = sm[0]
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    rc, _, _ = orc.decode_step(dm, ri.x, lp.conv_w, hist, ri.ba, lp.dt_bias, lp.A, ssm, sm)
    assert rc == O.DUP_SLOT
    assert np.array_equal(ssm, lp.ssm) and np.array_equal(hist, lp.conv_hist)


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
