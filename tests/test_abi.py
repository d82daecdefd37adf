"""The C-ABI library loads and exports every symbol include/gdn.h declares,
and host-side validation rejects bad arguments before any CUDA call.  CPU only:
every call here fails validation (or has nothing to do), so no kernel is ever
launched."""
import ctypes
import os
import re

import pytest

import gated_deltanet_speculative_gdn_gb300 as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(G.EXPORTED_SYMBOLS)


@pytest.mark.parametrize("name", declared_functions())
def test_symbol_exported(name):
    assert hasattr(G.lib, name)
    assert ctypes.cast(getattr(G.lib, name), ctypes.c_void_p).value


def test_status_strings():
    for name in dir(G):
        if name.startswith("GDN_OK") or name.startswith("GDN_ERR_") or name.startswith("GDN_DEV_"):
            assert G.gdn_status_str(getattr(G, name)) == name
    assert G.gdn_status_str(12345) == "unknown"


def test_replay_row_floats():
    assert G.gdn_replay_row_floats(128, 128) == 260
    assert G.gdn_replay_row_floats(16, 16) == 36
    assert G.gdn_replay_row_floats(64, 64) == 132
    assert G.gdn_replay_row_floats(48, 48) == 0


FAKE = 1 << 20          # a 16-byte aligned address that is never dereferenced


def dims(**kw):
    base = dict(n_seqs=2, n_nodes=8, n_slots=4, h_k=1, h_v=2, d=16, max_seq_nodes=16)
    base.update(kw)
    return G.GdnDims.make(**base)


def conv(d, **kw):
    C = d.conv_channels
    args = dict(x=FAKE, x_stride=C, conv_w=FAKE * 2, conv_hist=FAKE * 3, parents=FAKE * 4,
                node_off=FAKE * 5, slot_map=FAKE * 6, xc=FAKE * 7, win=FAKE * 8, status=FAKE * 9)
    args.update(kw)
    return G.gdn_conv_tree_step(d, args["x"], args["x_stride"], args["conv_w"], args["conv_hist"],
                                args["parents"], args["node_off"], args["slot_map"], args["xc"],
                                args["win"], args["status"], stream=0, raise_on_error=False)


def verify(d, **kw):
    args = dict(xc=FAKE, ba=FAKE * 2, ba_stride=2 * d.h_v, dt_bias=FAKE * 3, A=FAKE * 4, ssm=FAKE * 5,
                parents=FAKE * 6, node_off=FAKE * 7, slot_map=FAKE * 8, o=FAKE * 9, replay=FAKE * 10,
                replay_stride=G.gdn_replay_row_floats(d.d_k, d.d_v), status=FAKE * 11)
    args.update(kw)
    return G.gdn_tree_verify(d, args["xc"], args["ba"], args["ba_stride"], args["dt_bias"], args["A"],
                             args["ssm"], 1.0, args["parents"], args["node_off"], args["slot_map"],
                             args["o"], args["replay"], args["replay_stride"], args["status"],
                             stream=0, raise_on_error=False)


def chain_verify(d, **kw):
    args = dict(xc=FAKE, ba=FAKE * 2, ba_stride=2 * d.h_v, dt_bias=FAKE * 3, A=FAKE * 4, ssm=FAKE * 5,
                parents=FAKE * 6, node_off=FAKE * 7, slot_map=FAKE * 8, o=FAKE * 9, replay=FAKE * 10,
                replay_stride=G.gdn_replay_row_floats(d.d_k, d.d_v), status=FAKE * 11)
    args.update(kw)
    return G.gdn_chain_verify(d, args["xc"], args["ba"], args["ba_stride"], args["dt_bias"], args["A"],
                              args["ssm"], 1.0, args["parents"], args["node_off"], args["slot_map"],
                              args["o"], args["replay"], args["replay_stride"], args["status"],
                              stream=0, raise_on_error=False)


def commit(d, **kw):
    args = dict(accepted=FAKE, parents=FAKE * 2, node_off=FAKE * 3, slot_map=FAKE * 4, replay=FAKE * 5,
                replay_stride=G.gdn_replay_row_floats(d.d_k, d.d_v), win=FAKE * 6, ssm=FAKE * 7,
                conv_hist=FAKE * 8, status=FAKE * 9)
    args.update(kw)
    return G.gdn_commit(d, args["accepted"], args["parents"], args["node_off"], args["slot_map"],
                        args["replay"], args["replay_stride"], args["win"], args["ssm"],
                        args["conv_hist"], args["status"], stream=0, raise_on_error=False)


@pytest.mark.parametrize("bad", [
    dict(d=48), dict(d=8), dict(h_k=3, h_v=4), dict(max_seq_nodes=0), dict(max_seq_nodes=65),
    dict(n_slots=0), dict(n_seqs=-1), dict(h_v=0)])
def test_bad_dims(bad):
    d = dims(**bad)
    assert conv(d) == G.GDN_ERR_DIMS
    assert verify(d) == G.GDN_ERR_DIMS
    assert commit(d) == G.GDN_ERR_DIMS


def test_bad_d_conv_and_unequal_widths():
    d = dims()
    d.d_conv = 3
    assert conv(d) == G.GDN_ERR_DIMS
    d = dims()
    d.d_v = 32
    assert verify(d) == G.GDN_ERR_DIMS


def test_null_pointers():
    d = dims()
    assert conv(d, status=None) == G.GDN_ERR_NULL
    assert conv(d, x=None) == G.GDN_ERR_NULL
    assert verify(d, ssm=None) == G.GDN_ERR_NULL
    assert verify(d, replay=None) == G.GDN_ERR_NULL
    assert commit(d, accepted=None) == G.GDN_ERR_NULL
    assert commit(d, win=None) == G.GDN_ERR_NULL
    args = [None, None, None, 0, None, None, None, ctypes.c_float(1.0), None, None, None, None, None, 0,
            None, None]
    assert G.lib.gdn_tree_verify(*args) == G.GDN_ERR_NULL           # dims itself NULL


def test_strides():
    d = dims()
    assert conv(d, x_stride=d.conv_channels - 4) == G.GDN_ERR_STRIDE
    assert conv(d, x_stride=d.conv_channels + 2) == G.GDN_ERR_STRIDE
    assert verify(d, ba_stride=2 * d.h_v - 1) == G.GDN_ERR_STRIDE
    assert verify(d, replay_stride=2 * d.d_k) == G.GDN_ERR_STRIDE
    assert verify(d, replay_stride=2 * d.d_k + 2) == G.GDN_ERR_STRIDE
    assert commit(d, replay_stride=33) == G.GDN_ERR_STRIDE


def test_alignment():
    d = dims()
    assert conv(d, x=FAKE + 4) == G.GDN_ERR_ALIGN
    assert verify(d, ssm=FAKE * 5 + 8) == G.GDN_ERR_ALIGN
    assert commit(d, ssm=FAKE * 7 + 4) == G.GDN_ERR_ALIGN


def test_aliasing():
    d = dims()
    assert conv(d, xc=FAKE) == G.GDN_ERR_ALIAS                       # output on the input
    assert conv(d, win=FAKE * 7 + 16) == G.GDN_ERR_ALIAS             # outputs overlap
    assert verify(d, o=FAKE * 5 + 64) == G.GDN_ERR_ALIAS             # output inside the pool
    assert commit(d, conv_hist=FAKE * 6) == G.GDN_ERR_ALIAS          # history on the windows
    assert commit(d, ssm=FAKE * 9) == G.GDN_ERR_ALIAS                # pool on the status word


def test_empty_batches_are_no_ops():
    # nothing to do: returns before touching memory or the device
    d = dims(n_seqs=0, n_nodes=0)
    assert conv(d, x=None) == G.GDN_OK
    assert verify(d, xc=None) == G.GDN_OK
    assert commit(d, accepted=None) == G.GDN_OK
    d = dims(n_nodes=0)
    assert conv(d) == G.GDN_OK
    assert verify(d) == G.GDN_OK


def test_gated_norm_host_validation():
    d = dims()
    base = dict(o=FAKE, z=FAKE * 2, z_stride=d.h_v * d.d_v, w=FAKE * 3, eps=1e-6, mode=0, y=FAKE * 4)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return G.gdn_gated_rmsnorm(d, a["o"], a["z"], a["z_stride"], a["w"], a["eps"], a["mode"], a["y"],
                                   stream=0, raise_on_error=False)

    assert call(mode=2) == G.GDN_ERR_ARG
    assert call(eps=-1.0) == G.GDN_ERR_ARG
    assert call(eps=float("nan")) == G.GDN_ERR_ARG
    assert call(z_stride=d.h_v * d.d_v - 4) == G.GDN_ERR_STRIDE
    assert call(o=None) == G.GDN_ERR_NULL
    assert call(y=FAKE + 4) == G.GDN_ERR_ALIGN
    assert call(y=FAKE) == G.GDN_ERR_ALIAS


def test_compact_host_validation():
    d = dims()
    C = d.conv_channels
    assert G.gdn_conv_tree_step_compact(d, FAKE, C, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6,
                                        FAKE * 7, None, FAKE * 9, stream=0, raise_on_error=False) == G.GDN_ERR_NULL
    rs = G.gdn_replay_row_floats(d.d_k, d.d_v)
    assert G.gdn_commit_compact(d, FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, rs, FAKE * 6, C - 4, FAKE * 7,
                                FAKE * 8, FAKE * 9, FAKE * 10, stream=0, raise_on_error=False) == G.GDN_ERR_STRIDE
    assert G.gdn_commit_compact(d, FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, rs, FAKE * 6, C, None,
                                FAKE * 8, FAKE * 9, FAKE * 10, stream=0, raise_on_error=False) == G.GDN_ERR_NULL


def test_chain_verify_host_validation():
    """The chain verify takes gdn_tree_verify's arguments and checks them the
    same way; it serves d = 128 only."""
    for d in (16, 32, 64):
        assert chain_verify(dims(d=d)) == G.GDN_ERR_DIMS
    for bad in (dict(max_seq_nodes=65), dict(h_k=3, h_v=4), dict(n_slots=0)):
        assert chain_verify(dims(d=128, **bad)) == G.GDN_ERR_DIMS
    d = dims(d=128)
    assert chain_verify(d, ssm=None) == G.GDN_ERR_NULL
    assert chain_verify(d, status=None) == G.GDN_ERR_NULL
    assert chain_verify(d, ba_stride=2 * d.h_v - 1) == G.GDN_ERR_STRIDE
    assert chain_verify(d, replay_stride=2 * 128) == G.GDN_ERR_STRIDE
    assert chain_verify(d, replay_stride=2 * 128 + 2) == G.GDN_ERR_STRIDE
    assert chain_verify(d, ssm=FAKE * 5 + 8) == G.GDN_ERR_ALIGN
    assert chain_verify(d, o=FAKE * 5 + 64) == G.GDN_ERR_ALIAS
    assert chain_verify(dims(d=128, n_nodes=0)) == G.GDN_OK
    assert chain_verify(dims(d=128, n_seqs=0, n_nodes=0), xc=None) == G.GDN_OK
