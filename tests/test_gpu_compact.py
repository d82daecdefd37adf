"""Compact commit windows: the conv step names each node's window by three
references instead of copying it, and the commit gathers it from x and the
slot's history.  CUDA path vs the oracle through the C ABI: references and
the committed history bit-exact, everything else at the usual 1e-4."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gdn_gb300 as G
import gdn_workloads as W
import oracle as O
from gpu_harness import GpuPools, batch_from, compare, dev, run_gpu, run_oracle
from test_gpu_parity import check_commit, custom_batch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def oracle_refs(b):
    rc, refs = O.get().window_refs(b.odims(), b.parents, b.node_off)
    assert rc == 0
    return refs


def run_compact(b, ssm, hist, pools, **kw):
    before = pools.ssm.cpu().numpy()
    g = run_gpu(b, pools, compact=True, **kw)
    ref = run_oracle(b, ssm, hist)
    errs = compare(g, ref)
    assert np.array_equal(g.win_ref, oracle_refs(b)), "window references differ"
    errs["ssm"] = check_commit(b, pools, ref.ssm, ref.conv_hist, before, hist)
    return errs, ref


@pytest.mark.parametrize("cfg,rounds", [(0, 1), (2, 8)])
def test_compact_rounds(cfg, rounds):
    sp = W.spec(cfg)
    lp = W.layer_params(sp)
    sm = W.slot_map(sp)
    pools = GpuPools(lp.ssm, lp.conv_hist)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    for r in range(rounds):
        b = batch_from(sp, lp, W.round_inputs(sp, 0, r), sm)
        errs, ref = run_compact(b, ssm, hist, pools)
        ssm, hist = ref.ssm, ref.conv_hist
    print(cfg, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("d,kind,sizes", [(128, "tree", [9, 0, 14, 0, 3, 16]), (64, "chain", [64, 1, 17]),
                                          (16, "tree", [1, 2, 3])])
def test_compact_forests_chains_short_sequences(d, kind, sizes):
    """Several roots, empty sequences, sequences shorter than the window (the
    window then reaches into the history), chains through the 64-node kernel."""
    b, lp = custom_batch(3000 + d, 2, 4, d, sizes, kind=kind, forest=(kind == "tree"))
    pools = GpuPools(lp.ssm, lp.conv_hist)
    run_compact(b, lp.ssm, lp.conv_hist, pools, x_pad=8)


def test_compact_sweep_full_size():
    """The benchmark's headline workload at full size, three carried rounds."""
    sp = W.sweep_spec("grouped_tree16")
    lp = W.layer_params(sp)
    sm = W.slot_map(sp)
    pools = GpuPools(lp.ssm, lp.conv_hist)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    for r in range(3):
        b = batch_from(sp, lp, W.round_inputs(sp, 0, r), sm, max_nodes=sp.max_seq_nodes)
        errs, ref = run_compact(b, ssm, hist, pools)
        ssm, hist = ref.ssm, ref.conv_hist
    print({k: f"{v:.2e}" for k, v in errs.items()})


def test_compact_bad_reference_is_rejected_whole():
    b, lp = custom_batch(3100, 1, 2, 16, [5, 6], accepted=[3, 4])
    pools = GpuPools(lp.ssm, lp.conv_hist)
    dm = b.gdims()
    C, N = b.C, b.N
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs = G.gdn_replay_row_floats(b.d, b.d)
    wref = torch.from_numpy(oracle_refs(b)).cuda()
    wref[5 + 4, 1] = N                       # past the last node
    x = dev(b.x)
    rep = torch.zeros((N, b.Hv, rs), device="cuda")
    G.gdn_commit_compact(dm, dev(b.accepted), dev(b.parents), dev(b.node_off), dev(b.slot_map), rep, rs, x, C,
                         wref, pools.ssm, pools.conv_hist, status)
    torch.cuda.synchronize()
    assert int(status.item()) == G.GDN_DEV_BAD_WINDOW
    assert np.array_equal(pools.ssm.cpu().numpy(), lp.ssm)
    assert np.array_equal(pools.conv_hist.cpu().numpy(), lp.conv_hist)
