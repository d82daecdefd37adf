"""Writes tiny_oracle.json: the oracle's outputs on the tiny workload (one
sequence, H_k = H_v = 2, d = 16, parents [-1,0,0,1,2], accepted node 3).

Calls only the oracle and the seeded input generators.  The file freezes the
oracle so that any later change to its arithmetic shows up as a failing pin
and has to be justified.  Run from the repository root:
    python tests/golden/make_tiny_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import gdn_workloads as W  # noqa: E402
import oracle as O  # noqa: E402


def main():
    orc = O.get()
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
    out = {
        "what": "oracle outputs on the tiny workload (seed 0); regression fixture written by make_tiny_golden.py",
        "xc": np.round(xc, 17).tolist(),
        "o": o.tolist(),
        "replay": rep.tolist(),
        "committed_state": ssm[sm[0]].astype(np.float64).tolist(),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, separators=(",", ":"))


if __name__ == "__main__":
    main()
