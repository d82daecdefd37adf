"""Device-detected errors: each bad input yields its exact status code, and a
failed commit leaves both pools bit-identical.  Every bad index here is caught
by the kernels' own checks before it is used; no test faults the GPU."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gdn_gb300 as G
from gpu_harness import GpuPools, custom_batch, dev, run_gpu

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def status_of(b, lp, commit=True):
    pools = GpuPools(lp.ssm, lp.conv_hist)
    g = run_gpu(b, pools, commit=commit)
    return g.status, pools


def assert_pools_unchanged(pools, lp):
    assert np.array_equal(pools.ssm.cpu().numpy(), lp.ssm)
    assert np.array_equal(pools.conv_hist.cpu().numpy(), lp.conv_hist)


def test_bad_parent():
    b, lp = custom_batch(10, 1, 2, 16, [5, 6])
    b.parents = b.parents.copy()
    b.parents[5 + 3] = 3                       # a node that is its own parent
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_BAD_PARENT
    assert_pools_unchanged(pools, lp)
    b.parents[5 + 3] = -2
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_BAD_PARENT


def test_bad_slot():
    b, lp = custom_batch(11, 1, 2, 16, [5, 6])
    b.slot_map = b.slot_map.copy()
    b.slot_map[1] = b.P
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_BAD_SLOT
    assert_pools_unchanged(pools, lp)


def test_bad_node_offsets_and_too_many_nodes():
    b, lp = custom_batch(12, 1, 2, 16, [5, 6])
    b.node_off = b.node_off.copy()
    b.node_off[1] = 12                         # 0, 12, 11: past the end, not monotone
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_BAD_NODE_OFF
    assert_pools_unchanged(pools, lp)
    b, lp = custom_batch(13, 1, 2, 16, [20, 6], max_nodes=16)    # 20 > max_seq_nodes
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_BAD_NODE_OFF
    assert_pools_unchanged(pools, lp)


@pytest.mark.parametrize("d,max_nodes", [(16, None), (128, 16), (128, 64)])
def test_commit_duplicate_slot_is_rejected_whole(d, max_nodes):
    """At d = 128 through the streaming apply (both ring shapes)."""
    b, lp = custom_batch(14, 1, 2, d, [5, 6, 4], accepted=[2, 3, 1], max_nodes=max_nodes)
    b.slot_map = b.slot_map.copy()
    b.slot_map[2] = b.slot_map[0]
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_DUP_SLOT
    assert_pools_unchanged(pools, lp)
    # a shared slot is fine when one of the two commits nothing
    b.accepted = np.array([2, 3, -1], np.int32)
    st, pools = status_of(b, lp)
    assert st == 0


@pytest.mark.parametrize("acc", [[5, 0], [0, -2]])
def test_commit_bad_accepted(acc):
    b, lp = custom_batch(15, 1, 2, 16, [5, 6], accepted=acc)
    st, pools = status_of(b, lp)
    assert st == G.GDN_DEV_BAD_ACCEPTED
    assert_pools_unchanged(pools, lp)


@pytest.mark.parametrize("d,max_nodes", [(16, None), (128, 16), (128, 64)])
def test_commit_refuses_after_an_earlier_error(d, max_nodes):
    """A non-zero status on entry (e.g. left by verify) blocks the commit; at
    d = 128 through the streaming apply (both ring shapes)."""
    b, lp = custom_batch(16, 1, 2, d, [5, 6], accepted=[2, 3], max_nodes=max_nodes)
    pools = GpuPools(lp.ssm, lp.conv_hist)
    g = run_gpu(b, pools, commit=False)
    assert g.status == 0
    dm = b.gdims()
    status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    rs = G.gdn_replay_row_floats(b.d, b.d)
    rep = torch.zeros((b.N, b.Hv, rs), device="cuda")
    win = torch.zeros((b.N, 3, b.C), device="cuda")
    G.gdn_commit(dm, dev(b.accepted), dev(b.parents), dev(b.node_off), dev(b.slot_map), rep, rs, win,
                 pools.ssm, pools.conv_hist, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 99
    assert_pools_unchanged(pools, lp)


def test_verify_wait_that_runs_out_reports_timeout_and_the_context_survives():
    """A test hook makes one team of the first CTA of the tensor-core verify
    wait on a barrier that nothing completes; the wait runs out (20 ms), every
    role drains and leaves, *status reads GDN_DEV_TIMEOUT and the commit that
    follows writes nothing.  The next call on the same context is exact."""
    from gpu_harness import compare, run_oracle
    b, lp = custom_batch(18, 2, 4, 128, [16, 9, 12], max_nodes=16)
    pools = GpuPools(lp.ssm, lp.conv_hist)
    G.gdn_test_stall_next_verify(20_000_000)
    g = run_gpu(b, pools)
    assert g.status == G.GDN_DEV_TIMEOUT, G.gdn_status_str(g.status)
    assert_pools_unchanged(pools, lp)
    g2 = run_gpu(b, pools)
    compare(g2, run_oracle(b, lp.ssm, lp.conv_hist))


def test_chain_verify_wait_that_runs_out_reports_timeout_and_the_context_survives():
    """The same hook on the chain kernel: a d = 64 tree round first runs
    another kernel and leaves the hook pending (its result is exact); the
    chain round that follows takes it, the producer of its first CTA gives up
    before issuing a copy, the other roles' waits run out in turn, *status
    reads GDN_DEV_TIMEOUT and the commit writes nothing.  The next chain round
    on the same context is exact."""
    from gpu_harness import compare, run_oracle
    bt, lt = custom_batch(19, 2, 4, 64, [16, 7])
    G.gdn_test_stall_next_verify(20_000_000)
    pt = GpuPools(lt.ssm, lt.conv_hist)
    gt = run_gpu(bt, pt)
    assert gt.status == 0, G.gdn_status_str(gt.status)
    compare(gt, run_oracle(bt, lt.ssm, lt.conv_hist))
    b, lp = custom_batch(20, 2, 4, 128, [40, 23, 16], kind="chain", max_nodes=64)
    pools = GpuPools(lp.ssm, lp.conv_hist)
    g = run_gpu(b, pools, chain=True)
    assert g.status == G.GDN_DEV_TIMEOUT, G.gdn_status_str(g.status)
    assert_pools_unchanged(pools, lp)
    g2 = run_gpu(b, pools, chain=True)
    compare(g2, run_oracle(b, lp.ssm, lp.conv_hist))
