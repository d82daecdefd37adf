"""The tensor-core verify path (d = 128, at most 16 nodes per sequence) on the
method's edge cases, its device status codes, and a sweep over the scale of
the state, the values and the q/k rows.  CUDA path vs the oracle through the
C ABI, same parity bar as the other GPU tests.

The scale sweep matters because the kernel splits fp32 operands into parts
for the tensor cores: a part that loses range would show up as an error that
grows as the data shrinks or grows, although the method itself is
homogeneous in (state, values) and normalises q and k.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gdn_gb300 as G
from gpu_harness import GpuPools, compare, dev, nan_like, relerr, run_gpu, run_oracle
from test_gpu_parity import check_commit, custom_batch, run_edge

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

D = 128


def tc_batch(seed, Hk, Hv, sizes, **kw):
    """A d = 128 batch whose max_seq_nodes (16) selects the tensor-core kernel."""
    return custom_batch(seed, Hk, Hv, D, sizes, max_nodes=16, **kw)


# ----------------------------------------------------------------- edge cases
def test_forest_and_empty_sequences():
    """Several roots per sequence (every fifth node), empty sequences between
    full ones."""
    b, lp = tc_batch(1400, 2, 4, [9, 0, 14, 0, 3, 16], forest=True)
    run_edge(b, lp)


def test_padded_strides_and_q_scale():
    b, lp = tc_batch(1500, 2, 4, [12, 7, 16])
    run_edge(b, lp, q_scale=0.125, x_pad=12, ba_pad=3, replay_pad=8)


def test_nothing_accepted():
    b, lp = tc_batch(1700, 2, 4, [6, 4, 16], accepted=[-1, -1, -1])
    run_edge(b, lp)


@pytest.mark.parametrize("Hk,Hv", [(3, 3), (2, 4), (2, 6), (1, 5)])
def test_group_ratios(Hk, Hv):
    """G = H_v / H_k in {1, 2, 3, 5}; 3:1 is the 48-layer stack's ratio."""
    b, lp = tc_batch(1600 + 10 * Hk + Hv, Hk, Hv, [16, 5, 11, 1])
    run_edge(b, lp)


def test_more_items_than_one_pass_of_the_grid():
    """10,000 (sequence, head) items: more than one CTA per SM takes, so CTAs
    queue behind the first wave.  Verify only reads the pool, so sequences
    may share slots; only the first eight commit (distinct slots)."""
    S, P = 1250, 8
    sizes = [(s * 7) % 17 for s in range(S)]
    b, lp = custom_batch(1800, 2, 8, D, sizes, P=P, max_nodes=16)
    b.slot_map = (np.arange(S) % P).astype(np.int32)
    acc = np.full(S, -1, np.int32)
    for s in range(P):
        if sizes[s]:
            acc[s] = sizes[s] - 1
    b.accepted = acc
    run_edge(b, lp)


# ----------------------------------------------------------- device statuses
def verify_status(b, lp):
    """Runs verify alone with a fresh status word; returns (status, pool after)."""
    dm = b.gdims()
    N, C, Hv = max(b.N, 1), b.C, b.Hv
    rs = G.gdn_replay_row_floats(D, D)
    ssm = dev(lp.ssm)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xc = dev(np.zeros((N, C), np.float32))
    G.gdn_tree_verify(dm, xc, dev(b.ba), 2 * Hv, dev(b.dt_bias), dev(b.A), ssm, 1.0,
                      dev(b.parents), dev(b.node_off), dev(b.slot_map), nan_like((N, Hv, D)),
                      nan_like((N, Hv, rs)), rs, status)
    torch.cuda.synchronize()
    return int(status.item()), ssm.cpu().numpy()


def test_status_bad_parent():
    b, lp = tc_batch(20, 1, 2, [5, 6])
    b.parents = b.parents.copy()
    b.parents[5 + 3] = 3                       # its own parent
    st, ssm = verify_status(b, lp)
    assert st == G.GDN_DEV_BAD_PARENT
    assert np.array_equal(ssm, lp.ssm)
    b.parents[5 + 3] = -2
    assert verify_status(b, lp)[0] == G.GDN_DEV_BAD_PARENT


def test_status_bad_node_offsets():
    b, lp = tc_batch(21, 1, 2, [5, 6])
    b.node_off = b.node_off.copy()
    b.node_off[1] = 12                         # past the end, and not monotone
    st, ssm = verify_status(b, lp)
    assert st == G.GDN_DEV_BAD_NODE_OFF
    assert np.array_equal(ssm, lp.ssm)


def test_status_sequence_longer_than_max_seq_nodes():
    b, lp = tc_batch(22, 1, 2, [20, 6])        # 20 > max_seq_nodes = 16
    assert b.max_nodes == 16
    st, ssm = verify_status(b, lp)
    assert st == G.GDN_DEV_BAD_NODE_OFF
    assert np.array_equal(ssm, lp.ssm)


def test_status_bad_slot():
    b, lp = tc_batch(23, 1, 2, [5, 6])
    b.slot_map = b.slot_map.copy()
    b.slot_map[1] = b.P
    st, ssm = verify_status(b, lp)
    assert st == G.GDN_DEV_BAD_SLOT
    assert np.array_equal(ssm, lp.ssm)


# ------------------------------------------------------------------ scale sweep
def shared_xc(b, lp):
    """The oracle's conv output as fp32: both sides then verify on identical xc."""
    return run_oracle(b, lp.ssm, lp.conv_hist, commit=False).xc.astype(np.float32)


def run_scaled(b, lp, xc, ssm):
    pools = GpuPools(ssm, lp.conv_hist)
    g = run_gpu(b, pools, xc_override=xc)
    ref = run_oracle(b, ssm, lp.conv_hist, xc_override=xc)
    errs = compare(g, ref, check_xc=False)
    errs["ssm"] = check_commit(b, pools, ref.ssm, ref.conv_hist, ssm, lp.conv_hist)
    return errs


@pytest.mark.parametrize("k", [-24, -16, -8, 0, 8])
def test_state_and_value_scale(k):
    """S0 and v multiplied by 2^k (exact in fp32): o, u and the committed state
    scale by 2^k, so the relative error must not depend on k."""
    b, lp = tc_batch(1900, 2, 4, [16, 9, 13])
    xc = shared_xc(b, lp)
    f = np.float32(2.0 ** k)
    xc[:, 2 * b.Hk * D:] *= f
    ssm = np.ascontiguousarray(lp.ssm * f, dtype=np.float32)
    errs = run_scaled(b, lp, xc, ssm)
    print(f"2^{k}", {n: f"{v:.2e}" for n, v in errs.items()})


@pytest.mark.parametrize("e", [-4, -3, -2, -1, 0, 1, 2, 3])
def test_qk_scale(e):
    """q and k multiplied by 10^e.  The L2 norm's epsilon (1e-6) makes the
    method only approximately scale-invariant for small q/k, but both sides
    evaluate the same formula on the same fp32 inputs."""
    b, lp = tc_batch(1950, 2, 4, [16, 9, 13])
    xc = shared_xc(b, lp)
    xc[:, : 2 * b.Hk * D] *= np.float32(10.0 ** e)
    errs = run_scaled(b, lp, xc, lp.ssm)
    print(f"10^{e}", {n: f"{v:.2e}" for n, v in errs.items()})


def test_qk_scale_mixed_within_a_sequence():
    """Node t's q and k rows multiplied by 10^((t mod 7) - 3): rows seven
    orders of magnitude apart share one tensor-core operand."""
    b, lp = tc_batch(1960, 2, 4, [16, 16, 7])
    xc = shared_xc(b, lp)
    for s in range(b.S):
        n0, n1 = int(b.node_off[s]), int(b.node_off[s + 1])
        for t in range(n1 - n0):
            xc[n0 + t, : 2 * b.Hk * D] *= np.float32(10.0 ** ((t % 7) - 3))
    errs = run_scaled(b, lp, xc, lp.ssm)
    print("mixed", {n: f"{v:.2e}" for n, v in errs.items()})


def test_contraction_with_full_low_mantissas():
    """beta = 0 and decay = 1 reduce each single-node sequence to o = S0 q^,
    the bare contraction.  Every S0 and q entry has its low 13 mantissa bits
    set, so an operand part that counted those bits twice (or dropped them)
    would be off by ~2^-11; the split must reach fp32 accuracy (2^-17 here,
    against fp64)."""
    b, lp = tc_batch(2000, 2, 4, [1, 1, 1, 1, 1])
    b.ba = np.full_like(b.ba, -100.0)           # sigmoid -> 0, softplus -> 0, decay -> 1
    xc = shared_xc(b, lp)
    qs = slice(0, b.Hk * D)
    xc[:, qs] = (xc[:, qs].view(np.uint32) | np.uint32(0x1FFF)).view(np.float32)
    ssm = np.ascontiguousarray((lp.ssm.view(np.uint32) | np.uint32(0x1FFF)).view(np.float32))
    pools = GpuPools(ssm, lp.conv_hist)
    g = run_gpu(b, pools, xc_override=xc, commit=False)
    assert g.status == 0
    G_ = b.Hv // b.Hk
    want = np.empty((b.N, b.Hv, D))
    for t in range(b.N):
        s = t                                   # one node per sequence
        for h in range(b.Hv):
            q = xc[t, (h // G_) * D:(h // G_ + 1) * D].astype(np.float64)
            qhat = q / np.sqrt(np.dot(q, q) + 1e-6)
            want[t, h] = ssm[b.slot_map[s], h].astype(np.float64) @ qhat
    err = relerr(g.o, want)
    print(f"o = S0 q^: {err:.2e}")
    assert err <= 2.0 ** -17, err
