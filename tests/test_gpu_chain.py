"""The chain verify (gdn_chain_verify: chunked form, d = 128) against the
oracle through the C ABI: chains of every length class (one node, within one
16-node chunk, ragged tails, the 64-node maximum), grouping ratios, padded
strides, a grid with more items than resident CTAs, carried rounds at the
benchmark's full size, the scale of the state and of q/k, and the device
status codes.  Same parity bar as the other GPU tests: outputs, replay rows
and committed state within 1e-4, pools and status codes exact.  The oracle
is the tree verify (a chain is a tree); nothing here depends on the chunk
size except the choice of lengths.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gdn_gb300 as G
import gdn_workloads as W
from gpu_harness import GpuPools, batch_from, compare, dev, nan_like, run_gpu, run_oracle
from test_gpu_parity import check_commit, custom_batch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

D = 128


def chain_batch(seed, Hk, Hv, sizes, **kw):
    return custom_batch(seed, Hk, Hv, D, sizes, kind="chain", max_nodes=kw.pop("max_nodes", 64), **kw)


def run_chain(b, lp, q_scale=1.0, ssm=None, xc=None, **kw):
    ssm = lp.ssm if ssm is None else ssm
    pools = GpuPools(ssm, lp.conv_hist)
    g = run_gpu(b, pools, q_scale=q_scale, chain=True, xc_override=xc, **kw)
    ref = run_oracle(b, ssm, lp.conv_hist, q_scale=q_scale, xc_override=xc)
    errs = compare(g, ref, check_xc=xc is None)
    errs["ssm"] = check_commit(b, pools, ref.ssm, ref.conv_hist, ssm, lp.conv_hist)
    return errs


# ------------------------------------------------------------------- lengths
@pytest.mark.parametrize("sizes", [[1, 2, 3], [16, 15, 8], [17, 31, 32, 33], [64, 63, 48, 49], [64, 0, 5, 0]])
def test_chain_lengths(sizes):
    """One node, one chunk, a chunk plus a ragged tail, exact multiples of
    16, the 64-node maximum, empty sequences between full ones."""
    b, lp = chain_batch(3000 + sum(sizes), 2, 4, sizes)
    print(sizes, {k: f"{v:.2e}" for k, v in run_chain(b, lp).items()})


@pytest.mark.parametrize("Hk,Hv", [(3, 3), (2, 6), (1, 5), (16, 32)])
def test_group_ratios(Hk, Hv):
    b, lp = chain_batch(3100 + 10 * Hk + Hv, Hk, Hv, [64, 20, 9])
    run_chain(b, lp)


def test_padded_strides_q_scale_nothing_accepted():
    b, lp = chain_batch(3200, 2, 4, [40, 7, 64])
    run_chain(b, lp, q_scale=0.125, x_pad=12, ba_pad=3, replay_pad=8)
    b, lp = chain_batch(3201, 2, 4, [40, 7, 64], accepted=[-1, -1, -1])
    run_chain(b, lp)


def test_more_items_than_resident_ctas():
    """1,400 (sequence, head) items of mixed lengths (empty ones included):
    each persistent CTA takes several.  Verify only reads the pool, so
    sequences may share slots; only the first eight commit."""
    S, P = 700, 8
    sizes = [(s * 7) % 23 for s in range(S)]
    b, lp = chain_batch(3300, 1, 2, sizes, P=P, max_nodes=32)
    b.slot_map = (np.arange(S) % P).astype(np.int32)
    acc = np.full(S, -1, np.int32)
    for s in range(P):
        if sizes[s]:
            acc[s] = sizes[s] - 1
    b.accepted = acc
    run_chain(b, lp)


def test_more_items_than_one_pass_of_the_grid():
    """5,200 items of one to three nodes: more than the persistent grid takes
    in one pass at two CTAs per SM, so the grid grows to keep each CTA's list
    within its bound."""
    S, P = 2600, 8
    sizes = [1 + s % 3 for s in range(S)]
    b, lp = chain_batch(3350, 1, 2, sizes, P=P, max_nodes=16)
    b.slot_map = (np.arange(S) % P).astype(np.int32)
    acc = np.full(S, -1, np.int32)
    acc[:P] = [sizes[s] - 1 for s in range(P)]
    b.accepted = acc
    run_chain(b, lp)


def test_chain_kernel_matches_tree_kernel_closely():
    """Both kernels on the same chains: each is within the bar of the oracle,
    and the two agree with each other to the same bar."""
    b, lp = chain_batch(3400, 2, 4, [64, 33, 16])
    pa, pb = GpuPools(lp.ssm, lp.conv_hist), GpuPools(lp.ssm, lp.conv_hist)
    ga = run_gpu(b, pa, chain=True, commit=False)
    gb = run_gpu(b, pb, chain=False, commit=False)
    ref = run_oracle(b, lp.ssm, lp.conv_hist, commit=False)
    compare(ga, ref)
    compare(gb, ref)
    from gpu_harness import relerr
    assert relerr(ga.o, gb.o) <= 1e-4
    assert relerr(ga.replay[..., D:2 * D], gb.replay[..., D:2 * D]) <= 1e-4


def test_verify_leaves_pools_and_is_deterministic():
    b, lp = chain_batch(3500, 2, 4, [64, 17])
    pools = GpuPools(lp.ssm, lp.conv_hist)
    g1 = run_gpu(b, pools, commit=False, chain=True)
    assert np.array_equal(pools.ssm.cpu().numpy(), lp.ssm)
    g2 = run_gpu(b, pools, commit=False, chain=True)
    for f in ("o", "replay"):
        assert np.array_equal(getattr(g1, f), getattr(g2, f)), f


# ------------------------------------------------------------------ full size
@pytest.mark.parametrize("variant", ["grouped_chain64", "nongrouped_chain64"])
def test_sweep_chain64_full_size_three_rounds(variant):
    """The benchmark's chain workload at full size (64 sequences of 64-node
    chains, 128-slot pool) through the chain kernel: rounds 0-2, pools carried
    on both sides, every sequence compared with the oracle."""
    sp = W.sweep_spec(variant)
    lp = W.layer_params(sp)
    sm = W.slot_map(sp)
    pools = GpuPools(lp.ssm, lp.conv_hist)
    ssm, hist = lp.ssm.copy(), lp.conv_hist.copy()
    worst = {}
    for r in range(3):
        ri = W.round_inputs(sp, 0, r)
        b = batch_from(sp, lp, ri, sm, sp.max_seq_nodes)
        before = pools.ssm.cpu().numpy()
        g = run_gpu(b, pools, chain=True)
        ref = run_oracle(b, ssm, hist)
        errs = compare(g, ref)
        errs["ssm"] = check_commit(b, pools, ref.ssm, ref.conv_hist, before, hist)
        ssm, hist = ref.ssm, ref.conv_hist
        for k, v in errs.items():
            worst[k] = max(worst.get(k, 0.0), v)
    print(variant, {k: f"{v:.2e}" for k, v in worst.items()})


# -------------------------------------------------------------------- scales
@pytest.mark.parametrize("k", [-20, -6, 0, 6, 20])
def test_state_and_value_scale(k):
    """State and v scaled by 2^k together (the method is homogeneous in them)."""
    b, lp = chain_batch(3600, 2, 4, [64, 23])
    ref0 = run_oracle(b, lp.ssm, lp.conv_hist, commit=False)
    xc = ref0.xc.astype(np.float32)
    C0 = 2 * b.Hk * D
    xc[:, C0:] *= np.float32(2.0 ** k)
    ssm = (lp.ssm * np.float32(2.0 ** k)).astype(np.float32)
    run_chain(b, lp, ssm=ssm, xc=xc)


@pytest.mark.parametrize("e", [-30, -8, 8, 30])
def test_qk_scale(e):
    """q and k scaled by 2^e: only the 1e-6 inside the norm sees the scale."""
    b, lp = chain_batch(3700, 2, 4, [64, 9])
    xc = run_oracle(b, lp.ssm, lp.conv_hist, commit=False).xc.astype(np.float32)
    C0 = 2 * b.Hk * D
    xc[:, :C0] *= np.float32(2.0 ** e)
    run_chain(b, lp, xc=xc)


# ------------------------------------------------------------ device statuses
def chain_status(b, lp):
    dm = b.gdims()
    N, C, Hv = max(b.N, 1), b.C, b.Hv
    rs = G.gdn_replay_row_floats(D, D)
    ssm = dev(lp.ssm)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gdn_chain_verify(dm, dev(np.zeros((N, C), np.float32)), dev(b.ba), 2 * Hv, dev(b.dt_bias), dev(b.A),
                       ssm, 1.0, dev(b.parents), dev(b.node_off), dev(b.slot_map), nan_like((N, Hv, D)),
                       nan_like((N, Hv, rs)), rs, status)
    torch.cuda.synchronize()
    return int(status.item()), ssm.cpu().numpy()


def test_status_not_a_chain():
    b, lp = chain_batch(40, 1, 2, [5, 40])
    b.parents = b.parents.copy()
    b.parents[5 + 20] = 3                      # a branch: a valid tree, not a chain
    st, ssm = chain_status(b, lp)
    assert st == G.GDN_DEV_BAD_PARENT
    assert np.array_equal(ssm, lp.ssm)
    b.parents[5 + 20] = -1                     # a second root
    assert chain_status(b, lp)[0] == G.GDN_DEV_BAD_PARENT


def test_status_bad_node_offsets_slot_and_length():
    b, lp = chain_batch(41, 1, 2, [5, 6])
    b.node_off = b.node_off.copy()
    b.node_off[1] = 12
    assert chain_status(b, lp)[0] == G.GDN_DEV_BAD_NODE_OFF
    b, lp = chain_batch(42, 1, 2, [5, 6])
    b.slot_map = b.slot_map.copy()
    b.slot_map[0] = -1
    assert chain_status(b, lp)[0] == G.GDN_DEV_BAD_SLOT
    b, lp = chain_batch(43, 1, 2, [40, 6], max_nodes=32)  # 40 > max_seq_nodes
    assert chain_status(b, lp)[0] == G.GDN_DEV_BAD_NODE_OFF


def test_contraction_with_full_low_mantissas():
    """beta = 0 and decay = 1 leave the state at S0 through every chunk, so
    o_t = S0 q^_t for every node, across chunk boundaries (the state passes
    through the scale and the rank-16 update with u = 0).  Every S0 and q entry
    has its low 13 mantissa bits set: the kernel reads the state from tensor
    memory as its tf32 part and adds the rest from the fp16 lo product, so an
    operand part that counted those bits twice (or dropped them) would be off
    by ~2^-11.  The lo product rounds both of its operands to fp16 (11
    significant bits), so each term is exact to ~2^-20 of |S| |q| (the tree
    kernel, with exact lo parts of q, to ~2^-21), and the metric's floor at
    0.1 x RMS magnifies small outputs up to 10x: the bound is 2^-16, against
    fp64, still far below the ~2^-11 of a wrong split."""
    from gpu_harness import relerr
    b, lp = chain_batch(3800, 2, 4, [40, 1, 17])
    b.ba = np.full_like(b.ba, -100.0)           # sigmoid -> 0, softplus -> 0, decay -> 1
    xc = run_oracle(b, lp.ssm, lp.conv_hist, commit=False).xc.astype(np.float32)
    qs = slice(0, b.Hk * D)
    xc[:, qs] = (xc[:, qs].view(np.uint32) | np.uint32(0x1FFF)).view(np.float32)
    ssm = np.ascontiguousarray((lp.ssm.view(np.uint32) | np.uint32(0x1FFF)).view(np.float32))
    pools = GpuPools(ssm, lp.conv_hist)
    g = run_gpu(b, pools, xc_override=xc, commit=False, chain=True)
    assert g.status == 0
    G_ = b.Hv // b.Hk
    want = np.empty((b.N, b.Hv, D))
    for s in range(b.S):
        for t in range(int(b.node_off[s]), int(b.node_off[s + 1])):
            for h in range(b.Hv):
                q = xc[t, (h // G_) * D:(h // G_ + 1) * D].astype(np.float64)
                qhat = q / np.sqrt(np.dot(q, q) + 1e-6)
                want[t, h] = ssm[b.slot_map[s], h].astype(np.float64) @ qhat
    err = relerr(g.o, want)
    print(f"o = S0 q^ over chunks: {err:.2e}")
    assert err <= 2.0 ** -16, err
