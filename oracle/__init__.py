"""ctypes front end of the fp64 CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product library never imports it.
The C file is compiled with gcc on first use (or by ``build()``); numpy arrays
are passed by pointer.

Functions mirror the C entry points; every array argument is a numpy array
of the exact dtype (bf16 as ``uint16`` bit patterns, packed words as
``uint32``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs = {}


def build(plant: int = 0, out_dir: Optional[str] = None, openmp: bool = True) -> str:
    """Compile the oracle (optionally with planted mistake ``plant``)."""
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so"
    path = os.path.join(out_dir, name)
    if os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORACLE_PLANT={plant}",
           _SRC, "-o", path + ".tmp", "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    subprocess.run(cmd, check=True)
    os.replace(path + ".tmp", path)
    return path


_P = ctypes.c_void_p
_I = ctypes.c_int


def _bind(lib):
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_dequant.argtypes = [_P, _P, _P, _I, _I, _I, _P]
    lib.oracle_router_logits.argtypes = [_P, _I, _I, _P, _P, _I, _P]
    lib.oracle_topk.argtypes = [_P, _I, _I, _I, _P, _P, _P]
    lib.oracle_route_maps.restype = _I
    lib.oracle_route_maps.argtypes = [_P, _I, _I, _I, _I] + [_P] * 6
    lib.oracle_expert_ffn.argtypes = [_P, _I, _I, _I, _I] + [_P] * 9 + [_P]
    lib.oracle_moe_rows.argtypes = ([_P, _I, _I, _I, _I, _I, _I, _P, _P] + [_P] * 18
                                    + [_P, _I, _I, _P, _P, _P, _P, _P])
    lib.oracle_residual.argtypes = [_P, _P, _I, ctypes.c_double, _P]
    lib.oracle_rmsnorm.argtypes = [_P, _I, _I, ctypes.c_double, _P]
    lib.oracle_w4_bits_per_weight.restype = ctypes.c_double
    lib.oracle_w4_bits_per_weight.argtypes = [_I]
    lib.oracle_planted.restype = _I
    return lib


class Oracle:
    """One loaded oracle library (the real one, or a planted mutant)."""

    def __init__(self, plant: int = 0, out_dir: Optional[str] = None):
        self.lib = _bind(ctypes.CDLL(build(plant, out_dir)))
        self.plant = plant

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _p(a):
        if a is None:
            return None
        assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
        return a.ctypes.data_as(ctypes.c_void_p)

    # -- scalar conversions ---------------------------------------------
    def bf16_to_f64(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_f64(int(bits))

    def f64_to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_f64_to_bf16(float(v)))

    def bits_per_weight(self, G: int) -> float:
        return self.lib.oracle_w4_bits_per_weight(G)

    # -- array functions --------------------------------------------------
    def dequant(self, q, s, b, G: int) -> np.ndarray:
        """Dense fp64 ``[N, K]`` of one packed matrix ``q [N, K/8]``."""
        q = np.ascontiguousarray(q, np.uint32)
        s = np.ascontiguousarray(s, np.uint16)
        b = np.ascontiguousarray(b, np.uint16)
        N, K = q.shape[0], q.shape[1] * 8
        W = np.empty((N, K), np.float64)
        self.lib.oracle_dequant(self._p(q), self._p(s), self._p(b), N, K, G, self._p(W))
        return W

    def router_logits(self, x, wr, bias) -> np.ndarray:
        x = np.ascontiguousarray(x, np.uint16)
        wr = np.ascontiguousarray(wr, np.uint16)
        T, H = x.shape
        E = wr.shape[1]
        out = np.empty((T, E), np.float64)
        bias = None if bias is None else np.ascontiguousarray(bias, np.float32)
        self.lib.oracle_router_logits(self._p(x), T, H, self._p(wr), self._p(bias), E,
                                      self._p(out))
        return out

    def topk(self, logits, k: int):
        logits = np.ascontiguousarray(logits, np.float64)
        T, E = logits.shape
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float64)
        gap = np.empty(T, np.float64)
        self.lib.oracle_topk(self._p(logits), T, E, k, self._p(idx), self._p(w), self._p(gap))
        return idx, w, gap

    def route_maps(self, idx, E: int, BM: int = 128) -> dict:
        idx = np.ascontiguousarray(idx, np.int32)
        T, k = idx.shape
        cnt = np.empty(E, np.int32)
        off = np.empty(E + 1, np.int32)
        toff = np.empty(E + 1, np.int32)
        perm = np.empty(T * k, np.int32)
        inv = np.empty(T * k, np.int32)
        max_tiles = (T * k + BM - 1) // BM + E
        bmap = np.zeros((max_tiles, 3), np.int32)
        nt = self.lib.oracle_route_maps(self._p(idx), T, k, E, BM, self._p(cnt), self._p(off),
                                        self._p(toff), self._p(perm), self._p(inv),
                                        self._p(bmap))
        return dict(counts=cnt, offsets=off, tile_offsets=toff, perm=perm, inv=inv,
                    block_map=bmap[:nt].copy(), num_tiles=int(nt))

    def expert_ffn(self, x, e: int, gate, up, down, G: int) -> np.ndarray:
        """One routed expert ``e`` of a set applied to fp64 token ``x [H]``.

        ``gate``/``up``/``down`` are ``(q, s, b)`` triples of arrays
        ``[E, N, K/8]`` / ``[E, N, K/G]``."""
        x = np.ascontiguousarray(x, np.float64)
        H = x.shape[0]
        I = gate[0].shape[1]
        arrs = []
        for m in (gate, up, down):
            arrs += [np.ascontiguousarray(m[0], np.uint32), np.ascontiguousarray(m[1], np.uint16),
                     np.ascontiguousarray(m[2], np.uint16)]
        out = np.empty(H, np.float64)
        self.lib.oracle_expert_ffn(self._p(x), H, I, G, e, *[self._p(a) for a in arrs],
                                   self._p(out))
        return out

    def moe_rows(self, x, router_w, router_bias, routed: dict, shared: Optional[dict],
                 k: int, G: int, rows=None, nthreads: int = 1) -> dict:
        """The full layer for the listed token rows (all rows by default).

        ``routed``/``shared`` map "gate"/"up"/"down" to ``(q, s, b)``."""
        x = np.ascontiguousarray(x, np.uint16)
        T, H = x.shape
        wr = np.ascontiguousarray(router_w, np.uint16)
        E = wr.shape[1]
        I = routed["gate"][0].shape[1]
        rb = None if router_bias is None else np.ascontiguousarray(router_bias, np.float32)
        keep = []

        def trip(m):
            a = (np.ascontiguousarray(m[0], np.uint32), np.ascontiguousarray(m[1], np.uint16),
                 np.ascontiguousarray(m[2], np.uint16))
            keep.extend(a)
            return [self._p(t) for t in a]

        ptrs = []
        for name in ("gate", "up", "down"):
            ptrs += trip(routed[name])
        for name in ("gate", "up", "down"):
            ptrs += trip(shared[name]) if shared is not None else [None] * 3
        if rows is None:
            rows_a = None
            n = T
        else:
            rows_a = np.ascontiguousarray(rows, np.int32)
            n = rows_a.shape[0]
        logits = np.empty((n, E), np.float64)
        idx = np.empty((n, k), np.int32)
        w = np.empty((n, k), np.float64)
        gap = np.empty(n, np.float64)
        y = np.empty((n, H), np.float64)
        self.lib.oracle_moe_rows(self._p(x), T, H, I, E, k, G, self._p(wr), self._p(rb), *ptrs,
                                 self._p(rows_a), n, int(nthreads), self._p(logits),
                                 self._p(idx), self._p(w), self._p(gap), self._p(y))
        return dict(logits=logits, topk_idx=idx, topk_w=w, gap=gap, y=y)

    def rmsnorm(self, x, eps: float = 1e-6) -> np.ndarray:
        """Row-wise x / sqrt(mean(x^2) + eps) of bf16 rows, rounded to bf16."""
        x = np.ascontiguousarray(x, np.uint16)
        rows, H = (1, x.shape[0]) if x.ndim == 1 else x.shape
        out = np.empty_like(x)
        self.lib.oracle_rmsnorm(self._p(x), rows, H, float(eps), self._p(out))
        return out

    def residual(self, x, y, alpha: float) -> np.ndarray:
        x = np.ascontiguousarray(x, np.uint16)
        y = np.ascontiguousarray(y, np.float64)
        out = np.empty_like(x)
        self.lib.oracle_residual(self._p(x), self._p(y), x.size, float(alpha), self._p(out))
        return out


def get(plant: int = 0) -> Oracle:
    with _lock:
        if plant not in _libs:
            _libs[plant] = Oracle(plant)
        return _libs[plant]
