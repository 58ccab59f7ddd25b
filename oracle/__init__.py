"""Plain CPU oracle for one GLM-5.2 routed-MoE layer (ctypes over moe_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it.

Every wrapper takes and returns numpy arrays; the arithmetic lives in
``moe_oracle.c`` (plain C11, fp32 as the pages fix it, exact int32 dots).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_SRC = os.path.join(_HERE, "moe_oracle.c")
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so next to it (gcc, C11)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "moe_oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Expert(ctypes.Structure):
    _fields_ = [("gq", ctypes.c_void_p), ("uq", ctypes.c_void_p), ("dq", ctypes.c_void_p),
                ("gs", ctypes.c_void_p), ("us", ctypes.c_void_p), ("ds", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("K", ctypes.c_int), ("n_shared", ctypes.c_int),
                ("routed_scale", ctypes.c_float),
                ("Wr", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("experts", ctypes.POINTER(_Expert)), ("top_p", ctypes.c_float), ("weight_bits", ctypes.c_int)]


class _Debug(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("idx", "w", "xq", "sx", "gate_acc", "up_acc", "hq", "sh", "down_acc", "y",
                 "uniq", "n_uniq")]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, ci, cf = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        L.orc_pack_int4.argtypes = [vp, vp, vp, i64, i64]
        L.orc_unpack_int4.argtypes = [vp, vp, i64, i64]
        L.orc_qrow_i8.argtypes = [vp, vp, i64]
        L.orc_qrow_i8.restype = cf
        L.orc_quant_act.argtypes = [vp, vp, vp, i64, i64]
        L.orc_dot_i4_i8.argtypes = [vp, vp, i64]
        L.orc_dot_i4_i8.restype = ctypes.c_int32
        L.orc_quantize_rows.argtypes = [vp, vp, vp, i64, i64, ci]
        L.orc_dot_i8_i8.argtypes = [vp, vp, i64]
        L.orc_dot_i8_i8.restype = ctypes.c_int32
        L.orc_router.argtypes = [vp, vp, vp, ci, ci, ci, ci, cf, vp, vp, vp]
        L.orc_router_gap_f64.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
        L.orc_topp_keff.argtypes = [vp, ci, cf]
        L.orc_topp_keff.restype = ci
        L.orc_union.argtypes = [vp, ci, ci, ci, vp]
        L.orc_union.restype = ci
        L.orc_rmsnorm.argtypes = [vp, vp, vp, ci, cf]
        L.orc_layer_forward.argtypes = [ctypes.POINTER(_Layer), vp, ci, vp, ctypes.POINTER(_Debug)]
        L.orc_layer_forward.restype = ci
        L.orc_block_forward.argtypes = [ctypes.POINTER(_Layer), vp, vp, cf, ci]
        L.orc_block_forward.restype = ci
        L.orc_fp8_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_fp8_e4m3_decode.restype = cf
        L.orc_fp8_block_dequant.argtypes = [vp, vp, vp, i64, i64]
        L.orc_fp8_block_to_int4.argtypes = [vp, vp, vp, vp, i64, i64]
        L.orc_set_threads.argtypes = [ci]
        L.orc_max_threads.restype = ci
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def pack_int4(w):
    """w [O, I] fp32 -> (q4 [O, ceil(I/2)] uint8, scale [O] fp32)."""
    w = _c(w, np.float32)
    O, I = w.shape
    q4 = np.empty((O, (I + 1) // 2), np.uint8)
    s = np.empty(O, np.float32)
    lib().orc_pack_int4(_p(w), _p(q4), _p(s), O, I)
    return q4, s


def fp8_e4m3_decode(b):
    """uint8 array of FP8 E4M3 codes -> fp32 values (same shape)."""
    b = np.asarray(b, dtype=np.uint8)
    f = lib().orc_fp8_e4m3_decode
    return np.array([f(int(v)) for v in b.reshape(-1)], np.float32).reshape(b.shape)


def fp8_block_dequant(w8, scale_inv):
    """w8 [O, I] uint8 E4M3 codes, scale_inv [ceil(O/128), ceil(I/128)] fp32 -> fp32 [O, I]."""
    w8 = _c(w8, np.uint8)
    O, I = w8.shape
    si = _c(scale_inv, np.float32)
    assert si.shape == ((O + 127) // 128, (I + 127) // 128)
    w = np.empty((O, I), np.float32)
    lib().orc_fp8_block_dequant(_p(w8), _p(si), _p(w), O, I)
    return w


def fp8_block_to_int4(w8, scale_inv):
    """The converter step: block dequantisation then int4 packing -> (q4, scale)."""
    w8 = _c(w8, np.uint8)
    O, I = w8.shape
    si = _c(scale_inv, np.float32)
    assert si.shape == ((O + 127) // 128, (I + 127) // 128)
    q4 = np.empty((O, (I + 1) // 2), np.uint8)
    s = np.empty(O, np.float32)
    lib().orc_fp8_block_to_int4(_p(w8), _p(si), _p(q4), _p(s), O, I)
    return q4, s


def unpack_int4(q4, I):
    """q4 [O, ceil(I/2)] uint8 -> int8 values [O, I] in [-8, 7]."""
    q4 = _c(q4, np.uint8)
    O = q4.shape[0]
    v = np.empty((O, I), np.int8)
    lib().orc_unpack_int4(_p(q4), _p(v), O, I)
    return v


def qrow_i8(x):
    x = _c(x, np.float32).reshape(-1)
    q = np.empty(x.shape[0], np.int8)
    s = lib().orc_qrow_i8(_p(x), _p(q), x.shape[0])
    return q, np.float32(s)


def quant_act(x):
    x = _c(x, np.float32)
    T, D = x.shape
    xq = np.empty((T, D), np.int8)
    sx = np.empty(T, np.float32)
    lib().orc_quant_act(_p(x), _p(xq), _p(sx), T, D)
    return xq, sx


def dot_i4_i8(q4row, x):
    q4row = _c(q4row, np.uint8).reshape(-1)
    x = _c(x, np.int8).reshape(-1)
    assert q4row.shape[0] == (x.shape[0] + 1) // 2
    return int(lib().orc_dot_i4_i8(_p(q4row), _p(x), x.shape[0]))


def quantize_rows(w, bits=8):
    """w [O, I] fp32 -> (q [O, I] int8, scale [O] fp32), per-row symmetric."""
    w = _c(w, np.float32)
    O, I = w.shape
    q = np.empty((O, I), np.int8)
    s = np.empty(O, np.float32)
    lib().orc_quantize_rows(_p(w), _p(q), _p(s), O, I, int(bits))
    return q, s


def dot_i8_i8(w, x):
    w = _c(w, np.int8).reshape(-1)
    x = _c(x, np.int8).reshape(-1)
    assert w.shape == x.shape
    return int(lib().orc_dot_i8_i8(_p(w), _p(x), x.shape[0]))


def router(x, Wr, bias, K, routed_scale=2.5):
    """-> (idx [T,K] int32, w [T,K] fp32, p [T,E] fp32)."""
    x = _c(x, np.float32)
    Wr = _c(Wr, np.float32)
    bias = _c(bias, np.float32)
    T, D = x.shape
    E = Wr.shape[0]
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    p = np.empty((T, E), np.float32)
    lib().orc_router(_p(x), _p(Wr), _p(bias), T, D, E, K, float(routed_scale), _p(idx), _p(w), _p(p))
    return idx, w, p


def router_gap_f64(x, Wr, bias, K):
    x = _c(x, np.float32)
    Wr = _c(Wr, np.float32)
    bias = _c(bias, np.float32)
    T, D = x.shape
    gap = np.empty(T, np.float64)
    lib().orc_router_gap_f64(_p(x), _p(Wr), _p(bias), T, D, Wr.shape[0], K, _p(gap))
    return gap


def topp_keff(w, top_p):
    """w [K] or [T, K] routing weights in selection order -> keff (int or [T])."""
    w = _c(w, np.float32)
    if w.ndim == 1:
        return int(lib().orc_topp_keff(_p(w), w.shape[0], float(top_p)))
    return np.array([lib().orc_topp_keff(_p(np.ascontiguousarray(r)), w.shape[1], float(top_p)) for r in w], np.int32)


def union(idx, E):
    idx = _c(idx, np.int32)
    T, K = idx.shape
    u = np.empty(E, np.int32)
    n = lib().orc_union(_p(idx), T, K, E, _p(u))
    return u[:n].copy()


def rmsnorm(x, w, eps):
    x = _c(x, np.float32).reshape(-1)
    w = _c(w, np.float32).reshape(-1)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(w), _p(out), x.shape[0], float(eps))
    return out


@dataclass
class PackedExpert:
    """One expert's packed int4 weights as the oracle packed them."""
    gq: np.ndarray
    gs: np.ndarray
    uq: np.ndarray
    us: np.ndarray
    dq: np.ndarray
    ds: np.ndarray


def pack_expert(gate, up, down, bits=4) -> PackedExpert:
    """bits 4: packed int4 rows (pack_int4); bits 8: int8 rows (quantize_rows)."""
    pack = pack_int4 if bits == 4 else (lambda w: quantize_rows(w, 8))
    gq, gs = pack(gate)
    uq, us = pack(up)
    dq, ds = pack(down)
    return PackedExpert(gq, gs, uq, us, dq, ds)


class Layer:
    """Keeps the numpy buffers alive for the ctypes layer description."""

    def __init__(self, D, I, E, K, n_shared, routed_scale, Wr, bias, experts, top_p=0.0, weight_bits=4):
        """experts: dict or list, index -> PackedExpert (shared expert at index E).
        Missing entries are passed as NULL and must not be selected.  top_p in
        (0, 1) turns on adaptive expert top-p (dropped selections: id -1).
        weight_bits 8: the experts hold int8 rows (pack_expert(..., bits=8))."""
        self.D, self.I, self.E, self.K, self.n_shared = D, I, E, K, n_shared
        self.Wr = _c(Wr, np.float32)
        self.bias = _c(bias, np.float32)
        self._experts = dict(experts) if isinstance(experts, dict) else dict(enumerate(experts))
        arr = (_Expert * (E + n_shared))()
        for e, px in self._experts.items():
            if px is None:
                continue
            arr[e] = _Expert(_p(px.gq), _p(px.uq), _p(px.dq), _p(px.gs), _p(px.us), _p(px.ds))
        self._arr = arr
        self.top_p = float(top_p)
        self.weight_bits = int(weight_bits)
        self._c = _Layer(D, I, E, K, n_shared, float(routed_scale), _p(self.Wr), _p(self.bias), arr, self.top_p,
                         self.weight_bits)

    def forward(self, x, debug: bool = False):
        x = _c(x, np.float32)
        T = x.shape[0]
        out = np.empty((T, self.D), np.float32)
        dbg = None
        S = self.K + self.n_shared
        if debug:
            d = dict(idx=np.empty((T, self.K), np.int32), w=np.empty((T, self.K), np.float32),
                     xq=np.empty((T, self.D), np.int8), sx=np.empty(T, np.float32),
                     gate_acc=np.empty((T, S, self.I), np.int32),
                     up_acc=np.empty((T, S, self.I), np.int32),
                     hq=np.empty((T, S, self.I), np.int8), sh=np.empty((T, S), np.float32),
                     down_acc=np.empty((T, S, self.D), np.int32),
                     y=np.empty((T, S, self.D), np.float32),
                     uniq=np.empty(self.E, np.int32), n_uniq=np.empty(1, np.int32))
            dbg = d
            cd = _Debug(*[_p(d[n]) for n, _ in _Debug._fields_])
            rc = lib().orc_layer_forward(ctypes.byref(self._c), _p(x), T, _p(out), ctypes.byref(cd))
        else:
            rc = lib().orc_layer_forward(ctypes.byref(self._c), _p(x), T, _p(out), None)
        if rc != 0:
            raise RuntimeError(f"oracle layer forward failed ({rc}): missing expert weights?")
        if debug:
            dbg["uniq"] = dbg["uniq"][: int(dbg["n_uniq"][0])].copy()
            return out, dbg
        return out

    def block_forward(self, x, norm_w, eps):
        x = _c(x, np.float32).copy()
        nw = _c(norm_w, np.float32)
        rc = lib().orc_block_forward(ctypes.byref(self._c), _p(x), _p(nw), float(eps), x.shape[0])
        if rc != 0:
            raise RuntimeError(f"oracle block forward failed ({rc})")
        return x


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
