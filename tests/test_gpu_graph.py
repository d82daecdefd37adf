"""The library's calls captured in a CUDA graph.

Three carried rounds of conv -> verify -> commit are captured once into a
CUDA graph and replayed.  The replay must give bit-identical outputs, replay
rows and pools to the same calls launched one by one (the kernels are
deterministic and the graph holds the same launches, with the same
programmatic dependencies), and the pools after each pass must match the
oracle's.  Covered for the tensor-core tree path and the chain path.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gdn_gb300 as G
import gdn_workloads as W
from gpu_harness import TOL, batch_from, dev, relerr, run_oracle
from test_gpu_parity import custom_batch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


class Setup:
    """Device buffers for a few rounds of one layer, allocated before any
    launch, so that the launches can be captured."""

    def __init__(self, batches, ssm, hist, chain):
        b0 = batches[0]
        self.batches, self.chain = batches, chain
        self.dm = b0.gdims()
        N, C, Hv, d = b0.N, b0.C, b0.Hv, b0.d
        assert all(b.N == N for b in batches)
        self.rs = G.gdn_replay_row_floats(d, d)
        self.rounds = [dict(x=dev(b.x), ba=dev(b.ba), par=dev(b.parents), off=dev(b.node_off), acc=dev(b.accepted))
                       for b in batches]
        self.sm, self.w = dev(b0.slot_map), dev(b0.conv_w)
        self.dt, self.A = dev(b0.dt_bias), dev(b0.A)
        self.ssm, self.hist = dev(ssm), dev(hist)
        self.xc = torch.zeros((N, C), device="cuda")
        self.win = torch.zeros((N, 3, C), device="cuda")
        self.o = torch.zeros((N, Hv, d), device="cuda")
        self.rep = torch.zeros((N, Hv, self.rs), device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def launch(self):
        b0 = self.batches[0]
        C, Hv = b0.C, b0.Hv
        verify = G.gdn_chain_verify if self.chain else G.gdn_tree_verify
        for R in self.rounds:
            G.gdn_conv_tree_step(self.dm, R["x"], C, self.w, self.hist, R["par"], R["off"], self.sm, self.xc,
                                 self.win, self.status)
            verify(self.dm, self.xc, R["ba"], 2 * Hv, self.dt, self.A, self.ssm, 1.0, R["par"], R["off"], self.sm,
                   self.o, self.rep, self.rs, self.status)
            G.gdn_commit(self.dm, R["acc"], R["par"], R["off"], self.sm, self.rep, self.rs, self.win, self.ssm,
                         self.hist, self.status)

    def snapshot(self):
        torch.cuda.synchronize()
        return {k: getattr(self, k).cpu().numpy().copy() for k in ("xc", "win", "o", "rep", "ssm", "hist", "status")}


def oracle_pass(batches, ssm, hist):
    for b in batches:
        ref = run_oracle(b, ssm, hist)
        ssm, hist = ref.ssm, ref.conv_hist
    return ssm, hist


def check_graph(batches, ssm0, hist0, chain):
    eager = Setup(batches, ssm0, hist0, chain)
    graph = Setup(batches, ssm0, hist0, chain)
    eager.launch()                       # the launches also warm up lazy set-up
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graph.launch()
    ref_ssm, ref_hist = ssm0, hist0
    for _ in range(2):                   # two passes: the pools carry over
        g.replay()
        e, q = eager.snapshot(), graph.snapshot()
        for k in e:
            assert np.array_equal(e[k], q[k]), f"graph replay differs from the eager launches in {k}"
        assert int(q["status"][0]) == 0, G.gdn_status_str(int(q["status"][0]))
        ref_ssm, ref_hist = oracle_pass(batches, ref_ssm, ref_hist)
        assert np.array_equal(q["hist"], ref_hist), "conv history differs from the oracle"
        assert relerr(q["ssm"], ref_ssm) <= TOL
        eager.launch()


def test_tree_rounds_in_a_graph():
    """Four 16-node trees (the tensor-core verify), three rounds per graph."""
    sp = W.spec(2)
    lp = W.layer_params(sp)
    sm = W.slot_map(sp)
    batches = [batch_from(sp, lp, W.round_inputs(sp, 0, r), sm) for r in range(3)]
    check_graph(batches, lp.ssm, lp.conv_hist, chain=False)


def test_chain_rounds_in_a_graph():
    """Chains of 40 and 23 nodes through gdn_chain_verify, three rounds per graph."""
    batches = []
    lp = None
    for r in range(3):
        b, l = custom_batch(5000 + r, 2, 4, 128, [40, 23], kind="chain", max_nodes=64)
        lp = lp or l
        # one layer: every round uses the first round's weights and slot map
        b.conv_w, b.dt_bias, b.A = lp.conv_w, lp.dt_bias, lp.A
        if batches:
            b.slot_map = batches[0].slot_map
        batches.append(b)
    check_graph(batches, lp.ssm, lp.conv_hist, chain=True)
