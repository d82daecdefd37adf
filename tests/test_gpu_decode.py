"""Plain decode step (one token per sequence, state and history advanced in
place): CUDA path vs the oracle through the C ABI over several carried steps,
widths and head groupings, the headline shape, and the slot checks."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gdn_gb300 as G
import gdn_workloads as W
import oracle as O
from gpu_harness import TOL, dev, nan_like, relerr

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def decode_case(seed, S, P, Hk, Hv, d):
    sp = W.Spec(f"dec{seed}", W.Shape(S, P, Hk, Hv, d), "chain", [1] * S, seed)
    return sp, W.layer_params(sp), W.slot_map(sp)


def run_steps(sp, lp, sm, steps, q_scale=1.0, x_pad=0):
    sh = sp.shape
    S, C = sh.n_seqs, sh.conv_channels
    dm = G.GdnDims.make(S, S, sh.n_slots, sh.h_k, sh.h_v, sh.d, 16)
    odm = O.Dims(S, S, sh.n_slots, sh.h_k, sh.h_v, sh.d)
    ssm_d, hist_d = dev(lp.ssm), dev(lp.conv_hist)
    ssm_o, hist_o = lp.ssm.copy(), lp.conv_hist.copy()
    w, dt, A, smd = dev(lp.conv_w), dev(lp.dt_bias), dev(lp.A), dev(sm)
    worst = {}
    for r in range(steps):
        ri = W.round_inputs(sp, 0, r)
        xs = C + x_pad
        xh = np.zeros((S, xs), np.float32)
        xh[:, :C] = ri.x
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        xc, o = nan_like((S, C)), nan_like((S, sh.h_v, sh.d))
        G.gdn_decode_step(dm, dev(xh), xs, w, hist_d, dev(ri.ba), 2 * sh.h_v, dt, A, ssm_d, q_scale, smd, xc, o,
                          status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        rc, xc_r, o_r = O.get().decode_step(odm, ri.x, lp.conv_w, hist_o, ri.ba, lp.dt_bias, lp.A, ssm_o, sm,
                                            q_scale=q_scale)
        assert rc == 0
        errs = {"xc": relerr(xc.cpu().numpy(), xc_r), "o": relerr(o.cpu().numpy(), o_r),
                "ssm": relerr(ssm_d.cpu().numpy()[sm], ssm_o[sm])}
        assert np.array_equal(hist_d.cpu().numpy(), hist_o), "conv history differs"
        for k, v in errs.items():
            assert v <= TOL, (r, k, v)
            worst[k] = max(worst.get(k, 0.0), v)
    others = sorted(set(range(sp.shape.n_slots)) - set(int(s) for s in sm))
    assert np.array_equal(ssm_d.cpu().numpy()[others], lp.ssm[others])
    return worst


@pytest.mark.parametrize("d,Hk,Hv", [(16, 2, 2), (32, 2, 6), (64, 2, 4), (128, 3, 3), (128, 2, 6)])
def test_decode_steps(d, Hk, Hv):
    sp, lp, sm = decode_case(4000 + d + Hv, 5, 9, Hk, Hv, d)
    worst = run_steps(sp, lp, sm, 6, q_scale=0.75, x_pad=4)
    print(d, Hk, Hv, {k: f"{v:.2e}" for k, v in worst.items()})


def test_decode_headline_shape():
    """64 sequences in a 128-slot pool, 16 q/k and 32 value heads, d = 128."""
    sp, lp, sm = decode_case(4300, 64, 128, 16, 32, 128)
    worst = run_steps(sp, lp, sm, 3)
    print({k: f"{v:.2e}" for k, v in worst.items()})


@pytest.mark.parametrize("bad", ["dup", "range"])
def test_decode_bad_slots_write_nothing(bad):
    sp, lp, sm = decode_case(4400, 4, 6, 1, 2, 16)
    sm = sm.copy()
    if bad == "dup":
        sm[3] = sm[1]
    else:
        sm[2] = 6
    sh = sp.shape
    S, C = sh.n_seqs, sh.conv_channels
    dm = G.GdnDims.make(S, S, sh.n_slots, sh.h_k, sh.h_v, sh.d, 16)
    ri = W.round_inputs(sp)
    ssm_d, hist_d = dev(lp.ssm), dev(lp.conv_hist)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gdn_decode_step(dm, dev(ri.x), C, dev(lp.conv_w), hist_d, dev(ri.ba), 2 * sh.h_v, dev(lp.dt_bias),
                      dev(lp.A), ssm_d, 1.0, dev(sm), nan_like((S, C)), nan_like((S, sh.h_v, sh.d)), status)
    torch.cuda.synchronize()
    assert int(status.item()) == (G.GDN_DEV_DUP_SLOT if bad == "dup" else G.GDN_DEV_BAD_SLOT)
    assert np.array_equal(ssm_d.cpu().numpy(), lp.ssm)
    assert np.array_equal(hist_d.cpu().numpy(), lp.conv_hist)
