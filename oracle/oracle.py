"""ctypes wrapper of the CPU oracle (moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg use it. The product path never imports it.
It takes plain numpy arrays (bf16 as uint16 bit patterns) and returns numpy
arrays; it knows nothing of the CUDA library or of torch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain IEEE fp64: no -ffast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-ffp-contract=off", "-std=c++17", "-shared", "-fPIC",
                               "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


class _QMat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("gate", _QMat), ("up", _QMat), ("down", _QMat),
                ("s_gate", _QMat), ("s_up", _QMat), ("s_down", _QMat)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        vp, ci = ctypes.c_void_p, ctypes.c_int
        _lib.oracle_dequant.argtypes = [ctypes.POINTER(_QMat), ci, ci, ci, vp]
        _lib.oracle_route.argtypes = [ctypes.POINTER(_Layer), vp, ci, vp, vp, vp, ci]
        _lib.oracle_topk.argtypes = [vp, ci, ci, vp, vp]
        _lib.oracle_route_tables.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, ci]
        _lib.oracle_expert_h.argtypes = [ctypes.POINTER(_Layer), ci, vp, vp]
        _lib.oracle_moe_forward.argtypes = [ctypes.POINTER(_Layer), vp, ci, vp, ci, vp, ci]
        _lib.oracle_moe_forward_dense_masked.argtypes = [ctypes.POINTER(_Layer), vp, ci, vp, ci]
        _lib.oracle_threads_used.argtypes = [ci]
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleLayer:
    """Holds contiguous host copies of one layer (anything with the fields of
    synth.Layer) and the ctypes struct pointing at them."""

    def __init__(self, layer):
        self.D, self.E, self.k, self.I = layer.D, layer.E, layer.k, layer.I
        keep = []

        def qm(m):
            c, s, b = _c(m.codes, np.uint32), _c(m.scales, np.uint16), _c(m.biases, np.uint16)
            keep.extend([c, s, b])
            return _QMat(_p(c), _p(s), _p(b))

        wr = _c(layer.router_w, np.float32)
        rb = None if layer.router_bias is None else _c(layer.router_bias, np.float32)
        keep.extend([wr, rb])
        self._keep = keep
        self.s = _Layer(layer.D, layer.E, layer.k, layer.I, _p(wr), _p(rb),
                        qm(layer.gate), qm(layer.up), qm(layer.down),
                        qm(layer.s_gate), qm(layer.s_up), qm(layer.s_down))


def dequant(m, expert: int, rows: int, K: int) -> np.ndarray:
    c, s, b = _c(m.codes, np.uint32), _c(m.scales, np.uint16), _c(m.biases, np.uint16)
    q = _QMat(_p(c), _p(s), _p(b))
    out = np.empty((rows, K), dtype=np.float64)
    assert lib().oracle_dequant(ctypes.byref(q), expert, rows, K, _p(out)) == 0
    return out


def route(ol: OracleLayer, x: np.ndarray, n_threads: int = 0):
    """Returns (logits fp32 [T,E], topk_idx int32 [T,k], topk_w fp64 [T,k])."""
    x = _c(x, np.uint16)
    T = x.shape[0]
    logits = np.empty((T, ol.E), dtype=np.float32)
    idx = np.empty((T, ol.k), dtype=np.int32)
    w = np.empty((T, ol.k), dtype=np.float64)
    assert lib().oracle_route(ctypes.byref(ol.s), _p(x), T, _p(logits), _p(idx), _p(w), n_threads) == 0
    return logits, idx, w


def topk(logits: np.ndarray, k: int):
    """Top-k of one token's given fp32 logits [E]: (indices int32 [k], weights fp64 [k])."""
    lg = _c(logits, np.float32)
    idx = np.empty(k, np.int32)
    w = np.empty(k, np.float64)
    assert lib().oracle_topk(_p(lg), lg.shape[0], k, _p(idx), _p(w)) == 0
    return idx, w


def route_tables(topk_idx: np.ndarray, E: int, BM: int):
    """Returns dict(count [E], off [E+1], perm [T*k], inv [T*k], blocks [n,3])."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    A = T * k
    count = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    perm = np.empty(max(A, 1), np.int32)
    inv = np.empty(max(A, 1), np.int32)
    maxb = A // BM + E + T // BM + 2
    blocks = np.empty((maxb, 3), np.int32)
    nb = lib().oracle_route_tables(_p(idx), T, k, E, BM, _p(count), _p(off), _p(perm), _p(inv),
                                   _p(blocks), maxb)
    assert nb >= 0
    return dict(count=count, off=off, perm=perm[:A], inv=inv[:A], blocks=blocks[:nb])


def expert_h(ol: OracleLayer, expert: int, x_row: np.ndarray) -> np.ndarray:
    """Intermediate silu(g)*u [I] of one expert (-1 = shared) for one token row."""
    xr = _c(x_row, np.uint16)
    h = np.empty(ol.I, np.float64)
    assert lib().oracle_expert_h(ctypes.byref(ol.s), expert, _p(xr), _p(h)) == 0
    return h


def forward(ol: OracleLayer, x: np.ndarray, tokens=None, n_threads: int = 0) -> np.ndarray:
    """fp64 layer output for the listed tokens (all tokens if None)."""
    x = _c(x, np.uint16)
    T = x.shape[0]
    tk = None if tokens is None else _c(tokens, np.int32)
    n = T if tk is None else len(tk)
    y = np.empty((n, ol.D), np.float64)
    assert lib().oracle_moe_forward(ctypes.byref(ol.s), _p(x), T, _p(tk), n, _p(y), n_threads) == 0
    return y


def forward_dense_masked(ol: OracleLayer, x: np.ndarray, n_threads: int = 0) -> np.ndarray:
    x = _c(x, np.uint16)
    y = np.empty((x.shape[0], ol.D), np.float64)
    assert lib().oracle_moe_forward_dense_masked(ctypes.byref(ol.s), _p(x), x.shape[0], _p(y),
                                                 n_threads) == 0
    return y


def threads_used(n_threads: int = 0) -> int:
    return lib().oracle_threads_used(n_threads)
