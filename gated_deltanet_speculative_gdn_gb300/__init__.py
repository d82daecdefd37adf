"""Python binding of the GB300 GDN speculative tree-verify library.

Argument marshalling only: every step runs in the CUDA kernels of
``libgdn_gb300.so`` behind the C ABI declared in ``include/gdn.h``.  The
functions carry the C names and the C argument order.  Tensor arguments may be
torch tensors (their ``data_ptr()`` is passed) or raw device addresses
(ints); ``stream`` may be a ``torch.cuda.Stream``, a raw handle or None (the
current torch stream when torch has initialised CUDA, else the legacy default
stream).

A non-zero host return code raises :class:`GdnError`.  Device-side errors are
written into the caller's ``status`` tensor and are read by the caller.

There is no CPU fallback: importing this package fails if the library has not
been built (``python gated_deltanet_speculative_gdn_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn_gb300.so")

GDN_OK = 0
GDN_ERR_NULL, GDN_ERR_DIMS, GDN_ERR_STRIDE, GDN_ERR_ALIGN = -1, -2, -3, -4
GDN_ERR_ALIAS, GDN_ERR_LAUNCH, GDN_ERR_TMA, GDN_ERR_ARG = -5, -6, -7, -8
GDN_DEV_BAD_NODE_OFF, GDN_DEV_BAD_PARENT, GDN_DEV_BAD_SLOT = 1, 2, 3
GDN_DEV_DUP_SLOT, GDN_DEV_BAD_ACCEPTED, GDN_DEV_TIMEOUT = 4, 5, 6
GDN_DEV_BAD_WINDOW = 7

EXPORTED_SYMBOLS = ("gdn_conv_tree_step", "gdn_tree_verify", "gdn_chain_verify", "gdn_commit",
                    "gdn_conv_tree_step_compact", "gdn_commit_compact", "gdn_gated_rmsnorm",
                    "gdn_decode_step", "gdn_test_stall_next_verify",
                    "gdn_status_str", "gdn_replay_row_floats")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python gated_deltanet_speculative_gdn_gb300/build.py)")

lib = ctypes.CDLL(LIB_PATH)


class GdnDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_seqs", "n_nodes", "n_slots", "h_k", "h_v", "d_k", "d_v", "d_conv", "max_seq_nodes")]

    @classmethod
    def make(cls, n_seqs, n_nodes, n_slots, h_k, h_v, d, max_seq_nodes, d_conv=4):
        return cls(n_seqs, n_nodes, n_slots, h_k, h_v, d, d, d_conv, max_seq_nodes)

    @property
    def conv_channels(self) -> int:
        return 2 * self.h_k * self.d_k + self.h_v * self.d_v


class GdnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({gdn_status_str(code)})")
        self.code = code


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_DP = ctypes.POINTER(GdnDims)

lib.gdn_conv_tree_step.argtypes = [_DP, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P]
lib.gdn_tree_verify.argtypes = [_DP, _P, _P, _I64, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                                _P, _P, _I64, _P, _P]
lib.gdn_chain_verify.argtypes = lib.gdn_tree_verify.argtypes
lib.gdn_commit.argtypes = [_DP, _P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _P]
lib.gdn_conv_tree_step_compact.argtypes = [_DP, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P]
lib.gdn_commit_compact.argtypes = [_DP, _P, _P, _P, _P, _P, _I64, _P, _I64, _P, _P, _P, _P, _P]
lib.gdn_gated_rmsnorm.argtypes = [_DP, _P, _P, _I64, _P, ctypes.c_float, ctypes.c_int, _P, _P]
lib.gdn_test_stall_next_verify.argtypes = [ctypes.c_uint64]
lib.gdn_test_stall_next_verify.restype = None
lib.gdn_decode_step.argtypes = [_DP, _P, _I64, _P, _P, _P, _I64, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P,
                                _P]
for _f in ("gdn_conv_tree_step", "gdn_tree_verify", "gdn_chain_verify", "gdn_commit", "gdn_conv_tree_step_compact",
           "gdn_commit_compact", "gdn_gated_rmsnorm", "gdn_decode_step"):
    getattr(lib, _f).restype = ctypes.c_int
lib.gdn_status_str.argtypes = [ctypes.c_int]
lib.gdn_status_str.restype = ctypes.c_char_p
lib.gdn_replay_row_floats.argtypes = [ctypes.c_int, ctypes.c_int]
lib.gdn_replay_row_floats.restype = ctypes.c_size_t


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int, raise_on_error: bool) -> int:
    if rc != GDN_OK and raise_on_error:
        raise GdnError(fn, rc)
    return rc


def gdn_status_str(code: int) -> str:
    return lib.gdn_status_str(int(code)).decode()


def gdn_replay_row_floats(d_k: int, d_v: int) -> int:
    return int(lib.gdn_replay_row_floats(int(d_k), int(d_v)))


def gdn_conv_tree_step(dims: GdnDims, x, x_stride: int, conv_w, conv_hist, parents, node_off,
                       slot_map, xc, win, status, stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_conv_tree_step(ctypes.byref(dims), _ptr(x), int(x_stride), _ptr(conv_w),
                                _ptr(conv_hist), _ptr(parents), _ptr(node_off), _ptr(slot_map),
                                _ptr(xc), _ptr(win), _ptr(status), _stream(stream))
    return _check("gdn_conv_tree_step", rc, raise_on_error)


def gdn_tree_verify(dims: GdnDims, xc, ba, ba_stride: int, dt_bias, A, ssm, q_scale: float,
                    parents, node_off, slot_map, o, replay, replay_stride: int, status,
                    stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_tree_verify(ctypes.byref(dims), _ptr(xc), _ptr(ba), int(ba_stride), _ptr(dt_bias),
                             _ptr(A), _ptr(ssm), float(q_scale), _ptr(parents), _ptr(node_off),
                             _ptr(slot_map), _ptr(o), _ptr(replay), int(replay_stride),
                             _ptr(status), _stream(stream))
    return _check("gdn_tree_verify", rc, raise_on_error)


def gdn_chain_verify(dims: GdnDims, xc, ba, ba_stride: int, dt_bias, A, ssm, q_scale: float,
                     parents, node_off, slot_map, o, replay, replay_stride: int, status,
                     stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_chain_verify(ctypes.byref(dims), _ptr(xc), _ptr(ba), int(ba_stride), _ptr(dt_bias),
                              _ptr(A), _ptr(ssm), float(q_scale), _ptr(parents), _ptr(node_off),
                              _ptr(slot_map), _ptr(o), _ptr(replay), int(replay_stride),
                              _ptr(status), _stream(stream))
    return _check("gdn_chain_verify", rc, raise_on_error)


def gdn_commit(dims: GdnDims, accepted, parents, node_off, slot_map, replay, replay_stride: int,
               win, ssm, conv_hist, status, stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_commit(ctypes.byref(dims), _ptr(accepted), _ptr(parents), _ptr(node_off),
                        _ptr(slot_map), _ptr(replay), int(replay_stride), _ptr(win), _ptr(ssm),
                        _ptr(conv_hist), _ptr(status), _stream(stream))
    return _check("gdn_commit", rc, raise_on_error)


def gdn_conv_tree_step_compact(dims: GdnDims, x, x_stride: int, conv_w, conv_hist, parents, node_off,
                               slot_map, xc, win_ref, status, stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_conv_tree_step_compact(ctypes.byref(dims), _ptr(x), int(x_stride), _ptr(conv_w),
                                        _ptr(conv_hist), _ptr(parents), _ptr(node_off), _ptr(slot_map),
                                        _ptr(xc), _ptr(win_ref), _ptr(status), _stream(stream))
    return _check("gdn_conv_tree_step_compact", rc, raise_on_error)


def gdn_commit_compact(dims: GdnDims, accepted, parents, node_off, slot_map, replay, replay_stride: int,
                       x, x_stride: int, win_ref, ssm, conv_hist, status, stream=None,
                       raise_on_error: bool = True) -> int:
    rc = lib.gdn_commit_compact(ctypes.byref(dims), _ptr(accepted), _ptr(parents), _ptr(node_off),
                                _ptr(slot_map), _ptr(replay), int(replay_stride), _ptr(x), int(x_stride),
                                _ptr(win_ref), _ptr(ssm), _ptr(conv_hist), _ptr(status), _stream(stream))
    return _check("gdn_commit_compact", rc, raise_on_error)


def gdn_gated_rmsnorm(dims: GdnDims, o, z, z_stride: int, norm_w, eps: float, gate_mode: int, y,
                      stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_gated_rmsnorm(ctypes.byref(dims), _ptr(o), _ptr(z), int(z_stride), _ptr(norm_w), float(eps),
                               int(gate_mode), _ptr(y), _stream(stream))
    return _check("gdn_gated_rmsnorm", rc, raise_on_error)


def gdn_decode_step(dims: GdnDims, x, x_stride: int, conv_w, conv_hist, ba, ba_stride: int, dt_bias, A, ssm,
                    q_scale: float, slot_map, xc, o, status, stream=None, raise_on_error: bool = True) -> int:
    rc = lib.gdn_decode_step(ctypes.byref(dims), _ptr(x), int(x_stride), _ptr(conv_w), _ptr(conv_hist), _ptr(ba),
                             int(ba_stride), _ptr(dt_bias), _ptr(A), _ptr(ssm), float(q_scale), _ptr(slot_map),
                             _ptr(xc), _ptr(o), _ptr(status), _stream(stream))
    return _check("gdn_decode_step", rc, raise_on_error)


def gdn_test_stall_next_verify(wait_ns: int) -> None:
    lib.gdn_test_stall_next_verify(int(wait_ns))
