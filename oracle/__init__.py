"""ctypes front end of the C oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The library under test never does.

``build()`` compiles ``gdn_oracle.c`` with gcc (-O2, -ffp-contract=off, no
fast-math) into ``liboracle_gdn.so`` beside it.  ``compile_source`` compiles
another copy of the source the same way; the mutation test uses it to build
deliberately broken copies and checks that every planted mistake fails at
least one pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gdn_oracle.c")
LIB = os.path.join(_HERE, "liboracle_gdn.so")

OK, BAD_NODE_OFF, BAD_PARENT, BAD_SLOT, DUP_SLOT, BAD_ACCEPTED, BAD_DIMS, NOMEM = range(8)


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -ffp-contract=off (no fast-math) of one oracle source file into
    a shared library at ``out``."""
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC",
           "-shared", "-I", _HERE, "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
            os.path.getmtime(SOURCE), os.path.getmtime(os.path.join(_HERE, "gdn_oracle.h"))):
        return LIB
    return compile_source(SOURCE, LIB)


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_seqs", "n_nodes", "n_slots", "h_k", "h_v", "d", "d_conv")]


@dataclass(frozen=True)
class Dims:
    n_seqs: int
    n_nodes: int
    n_slots: int
    h_k: int
    h_v: int
    d: int
    d_conv: int = 4

    @property
    def conv_channels(self) -> int:
        return 2 * self.h_k * self.d + self.h_v * self.d

    def c(self) -> _Dims:
        return _Dims(self.n_seqs, self.n_nodes, self.n_slots, self.h_k, self.h_v,
                     self.d, self.d_conv)


_P = ctypes.c_void_p


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


class Oracle:
    def __init__(self, lib_path: Optional[str] = None):
        self.lib = ctypes.CDLL(lib_path or build())
        self.lib.gdn_oracle_conv_tree_step.argtypes = [
            ctypes.POINTER(_Dims), _P, ctypes.c_long, _P, _P, _P, _P, _P, _P, _P]
        self.lib.gdn_oracle_tree_verify.argtypes = [
            ctypes.POINTER(_Dims), _P, _P, ctypes.c_long, _P, _P, _P, ctypes.c_double,
            _P, _P, _P, _P, _P]
        self.lib.gdn_oracle_commit.argtypes = [
            ctypes.POINTER(_Dims), _P, _P, _P, _P, _P, _P, _P, _P]
        self.lib.gdn_oracle_window_refs.argtypes = [ctypes.POINTER(_Dims), _P, _P, _P]
        self.lib.gdn_oracle_commit_compact.argtypes = [
            ctypes.POINTER(_Dims), _P, _P, _P, _P, _P, _P, ctypes.c_long, _P, _P, _P]
        self.lib.gdn_oracle_gated_rmsnorm.argtypes = [
            ctypes.POINTER(_Dims), _P, _P, ctypes.c_long, _P, ctypes.c_double, ctypes.c_int, _P]
        self.lib.gdn_oracle_decode_step.argtypes = [
            ctypes.POINTER(_Dims), _P, ctypes.c_long, _P, _P, _P, ctypes.c_long, _P, _P, _P, ctypes.c_double,
            _P, _P, _P]
        for f in ("gdn_oracle_conv_tree_step", "gdn_oracle_tree_verify", "gdn_oracle_commit",
                  "gdn_oracle_window_refs", "gdn_oracle_commit_compact", "gdn_oracle_gated_rmsnorm",
                  "gdn_oracle_decode_step"):
            getattr(self.lib, f).restype = ctypes.c_int

    def conv_tree_step(self, dm: Dims, x, conv_w, conv_hist, parents, node_off, slot_map):
        """Returns (status, xc [N][C] float64, win [N][K-1][C] float32)."""
        x = _f32(x)
        C = dm.conv_channels
        xc = np.zeros((dm.n_nodes, C), dtype=np.float64)
        win = np.zeros((dm.n_nodes, dm.d_conv - 1, C), dtype=np.float32)
        cd = dm.c()
        w, hist, par, off, sm = _f32(conv_w), _f32(conv_hist), _i32(parents), _i32(node_off), _i32(slot_map)
        rc = self.lib.gdn_oracle_conv_tree_step(
            ctypes.byref(cd), _ptr(x), x.shape[1] if x.ndim == 2 else C, _ptr(w), _ptr(hist),
            _ptr(par), _ptr(off), _ptr(sm), _ptr(xc), _ptr(win))
        return rc, xc, win

    def tree_verify(self, dm: Dims, xc, ba, dt_bias, A, ssm, parents, node_off, slot_map,
                    q_scale: float = 1.0):
        """Returns (status, o [N][H_v][d] float64, replay [N][H_v][2d+1] float64)."""
        xc, ba = _f32(xc), _f32(ba)
        o = np.zeros((dm.n_nodes, dm.h_v, dm.d), dtype=np.float64)
        rep = np.zeros((dm.n_nodes, dm.h_v, 2 * dm.d + 1), dtype=np.float64)
        cd = dm.c()
        dt, Aa, S = _f32(dt_bias), _f32(A), _f32(ssm)
        par, off, sm = _i32(parents), _i32(node_off), _i32(slot_map)
        rc = self.lib.gdn_oracle_tree_verify(
            ctypes.byref(cd), _ptr(xc), _ptr(ba), ba.shape[1] if ba.ndim == 2 else 2 * dm.h_v,
            _ptr(dt), _ptr(Aa), _ptr(S), float(q_scale), _ptr(par), _ptr(off), _ptr(sm),
            _ptr(o), _ptr(rep))
        return rc, o, rep

    def commit(self, dm: Dims, accepted, parents, node_off, slot_map, replay, win, ssm, conv_hist):
        """Commits in place into ``ssm`` and ``conv_hist`` (float32, C-contiguous)."""
        assert ssm.dtype == np.float32 and ssm.flags.c_contiguous
        assert conv_hist.dtype == np.float32 and conv_hist.flags.c_contiguous
        rep = np.ascontiguousarray(replay, dtype=np.float64)
        w = _f32(win)
        cd = dm.c()
        acc, par, off, sm = _i32(accepted), _i32(parents), _i32(node_off), _i32(slot_map)
        return self.lib.gdn_oracle_commit(
            ctypes.byref(cd), _ptr(acc), _ptr(par), _ptr(off), _ptr(sm), _ptr(rep), _ptr(w),
            _ptr(ssm), _ptr(conv_hist))


    def window_refs(self, dm: Dims, parents, node_off):
        """Returns (status, refs [N][d_conv - 1] int32): the commit window of every
        node as references (x row >= 0, or -1 - k for history column k)."""
        refs = np.zeros((dm.n_nodes, dm.d_conv - 1), dtype=np.int32)
        cd = dm.c()
        par, off = _i32(parents), _i32(node_off)
        rc = self.lib.gdn_oracle_window_refs(ctypes.byref(cd), _ptr(par), _ptr(off), _ptr(refs))
        return rc, refs


    def commit_compact(self, dm: Dims, accepted, parents, node_off, slot_map, replay, x, refs, ssm,
                        conv_hist):
        """gdn_oracle_commit with the accepted windows gathered through refs."""
        assert ssm.dtype == np.float32 and ssm.flags.c_contiguous
        assert conv_hist.dtype == np.float32 and conv_hist.flags.c_contiguous
        rep = np.ascontiguousarray(replay, dtype=np.float64)
        xx = _f32(x)
        cd = dm.c()
        acc, par, off, sm, rf = _i32(accepted), _i32(parents), _i32(node_off), _i32(slot_map), _i32(refs)
        return self.lib.gdn_oracle_commit_compact(
            ctypes.byref(cd), _ptr(acc), _ptr(par), _ptr(off), _ptr(sm), _ptr(rep), _ptr(xx),
            xx.shape[1] if xx.ndim == 2 else dm.conv_channels, _ptr(rf), _ptr(ssm), _ptr(conv_hist))

    def gated_rmsnorm(self, dm: Dims, o, z, w, eps: float, gate_mode: int):
        """Returns (status, y [N][h_v][d] float64)."""
        oo, zz, ww = _f32(o), _f32(z), _f32(w)
        y = np.zeros((dm.n_nodes, dm.h_v, dm.d), dtype=np.float64)
        cd = dm.c()
        rc = self.lib.gdn_oracle_gated_rmsnorm(ctypes.byref(cd), _ptr(oo), _ptr(zz),
                                               zz.shape[1] if zz.ndim == 2 else dm.h_v * dm.d, _ptr(ww),
                                               float(eps), int(gate_mode), _ptr(y))
        return rc, y

    def decode_step(self, dm: Dims, x, conv_w, conv_hist, ba, dt_bias, A, ssm, slot_map, q_scale: float = 1.0):
        """One token per sequence, in place into ``ssm`` and ``conv_hist``
        (float32, C-contiguous).  Returns (status, xc [S][C], o [S][h_v][d])."""
        assert ssm.dtype == np.float32 and ssm.flags.c_contiguous
        assert conv_hist.dtype == np.float32 and conv_hist.flags.c_contiguous
        xx, bb = _f32(x), _f32(ba)
        xc = np.zeros((dm.n_seqs, dm.conv_channels), dtype=np.float64)
        o = np.zeros((dm.n_seqs, dm.h_v, dm.d), dtype=np.float64)
        cd = dm.c()
        w, dt, Aa, sm = _f32(conv_w), _f32(dt_bias), _f32(A), _i32(slot_map)
        rc = self.lib.gdn_oracle_decode_step(
            ctypes.byref(cd), _ptr(xx), xx.shape[1], _ptr(w), _ptr(conv_hist), _ptr(bb), bb.shape[1], _ptr(dt),
            _ptr(Aa), _ptr(ssm), float(q_scale), _ptr(sm), _ptr(xc), _ptr(o))
        return rc, xc, o


_default: Optional[Oracle] = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default

