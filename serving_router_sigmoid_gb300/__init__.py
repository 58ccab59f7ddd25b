"""Thin Python binding of libmoe_int4.so, the GB300 routed-MoE layer library.

Argument marshalling only: every function passes device pointers of torch
tensors (and the current CUDA stream) to the C ABI declared in
include/moe_int4.h and raises on a non-zero status.  Every step of the layer
runs in the library's CUDA kernels; there is no CPU path.  Importing the
package fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_int4.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_SHAPE = -2
MOE_ERR_CUDA = -3
MOE_ERR_NOMEM = -4
MOE_ERR_DEVICE = -5
MOE_PROBE_NONE, MOE_PROBE_GATE_UP, MOE_PROBE_DOWN, MOE_PROBE_ROUTER = 0, 1, 2, 3
MOE_OPT_DECODE_SINGLE_KERNEL, MOE_OPT_DECODE_SINGLE_KERNEL_AVAILABLE, MOE_OPT_TCGEN05_GEMM = 1, 2, 3
MOE_OPT_DECODE_TEST_WAIT_TIMEOUT = 4
MOE_OPT_TCGEN05_GEMM_AVAILABLE = 5
MOE_OPT_TCGEN05_TMA_WEIGHTS = 6

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'`")


class MoeLayerDesc(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int), ("K", ctypes.c_int),
                ("n_shared", ctypes.c_int), ("routed_scale", ctypes.c_float), ("max_tokens", ctypes.c_int),
                ("top_p", ctypes.c_float), ("weight_bits", ctypes.c_int)]


class MoeExpertW(ctypes.Structure):
    _fields_ = [("gate_q", ctypes.c_void_p), ("up_q", ctypes.c_void_p), ("down_q", ctypes.c_void_p),
                ("gate_s", ctypes.c_void_p), ("up_s", ctypes.c_void_p), ("down_s", ctypes.c_void_p)]


class MoeDebugOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("idx", "w", "xq", "sx", "gate_acc", "up_acc", "hq", "sh", "down_acc", "union_experts",
                 "n_union")]


_lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _ci, _cf = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
_SIGS = {
    "moe_version": ([], _ci),
    "moe_last_error": ([], ctypes.c_char_p),
    "moe_pack_int4": ([_vp, _vp, _vp, _i64, _i64, _vp], _ci),
    "moe_quant_act_int8": ([_vp, _vp, _vp, _ci, _ci, _vp], _ci),
    "moe_fp8_block_to_int4": ([_vp, _vp, _vp, _vp, _i64, _i64, _vp], _ci),
    "moe_pack_int8": ([_vp, _vp, _vp, _i64, _i64, _vp], _ci),
    "moe_router_topk": ([_vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _vp, _vp, _vp], _ci),
    "moe_layer_create": ([ctypes.POINTER(MoeLayerDesc), _vp, _vp, ctypes.POINTER(MoeExpertW),
                          ctypes.POINTER(_vp)], _ci),
    "moe_layer_destroy": ([_vp], _ci),
    "moe_layer_forward": ([_vp, _vp, _ci, _vp, _vp], _ci),
    "moe_block_forward": ([_vp, _vp, _vp, _cf, _ci, _vp], _ci),
    "moe_layer_debug": ([_vp, _vp, _ci, _vp, ctypes.POINTER(MoeDebugOut), _vp], _ci),
    "moe_layer_device_status": ([_vp, _vp, ctypes.POINTER(_ci)], _ci),
    "moe_layer_set_probe": ([_vp, _ci, _vp, _vp], _ci),
    "moe_layer_forward_host": ([_vp, _vp, _ci, _vp, _vp], _ci),
    "moe_layer_set_option": ([_vp, _ci, _ci], _ci),
    "moe_layer_set_trace": ([_vp, _vp, _ci], _ci),
    "moe_layer_get_option": ([_vp, _ci, ctypes.POINTER(_ci)], _ci),
    "moe_layer_workspace_bytes": ([ctypes.POINTER(MoeLayerDesc), ctypes.POINTER(ctypes.c_size_t)], _ci),
    "moe_layer_forward_static": ([ctypes.POINTER(MoeLayerDesc), _vp, _vp, _vp, _vp, _ci, _vp, _vp], _ci),
    "moe_layer_static_status": ([_vp, ctypes.POINTER(_ci)], _ci),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def _check(rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, _lib.moe_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def version() -> int:
    return int(_lib.moe_version())


def library():
    """The ctypes handle of libmoe_int4.so."""
    return _lib


def moe_pack_int4(w, q4, scale, stream=None):
    O, I = w.shape
    _check(_lib.moe_pack_int4(_ptr(w), _ptr(q4), _ptr(scale), O, I, _stream(stream)))


def moe_quant_act_int8(x, xq, sx, stream=None):
    T, D = x.shape
    _check(_lib.moe_quant_act_int8(_ptr(x), _ptr(xq), _ptr(sx), T, D, _stream(stream)))


def moe_router_topk(x, Wr, bias, K, routed_scale, idx, w, stream=None):
    T, D = x.shape
    E = Wr.shape[0]
    _check(_lib.moe_router_topk(_ptr(x), _ptr(Wr), _ptr(bias), T, D, E, K, float(routed_scale),
                                _ptr(idx), _ptr(w), _stream(stream)))


def moe_fp8_block_to_int4(w8, scale_inv, q4, scale, stream=None):
    """w8 [O, I] uint8 E4M3 codes, scale_inv [ceil(O/128), ceil(I/128)] fp32 -> q4, scale (outputs)."""
    O, I = w8.shape
    if tuple(scale_inv.shape) != ((O + 127) // 128, (I + 127) // 128):
        raise ValueError("scale_inv must be [ceil(O/128), ceil(I/128)]")
    _check(_lib.moe_fp8_block_to_int4(_ptr(w8), _ptr(scale_inv), _ptr(q4), _ptr(scale), O, I, _stream(stream)))


def fp8_block_to_int4(w8, scale_inv, stream=None):
    """Allocating convenience wrapper of moe_fp8_block_to_int4 -> (q4, scale)."""
    O, I = w8.shape
    q4 = torch.empty((O, (I + 1) // 2), dtype=torch.uint8, device=w8.device)
    s = torch.empty(O, dtype=torch.float32, device=w8.device)
    moe_fp8_block_to_int4(w8, scale_inv, q4, s, stream)
    return q4, s


def moe_pack_int8(w, q8, scale, stream=None):
    O, I = w.shape
    _check(_lib.moe_pack_int8(_ptr(w), _ptr(q8), _ptr(scale), O, I, _stream(stream)))


def pack_int8(w, stream=None):
    """Allocating convenience wrapper: w [O, I] fp32 (cuda) -> (q8 int8 [O, I], scale)."""
    O, I = w.shape
    q8 = torch.empty((O, I), dtype=torch.int8, device=w.device)
    s = torch.empty(O, dtype=torch.float32, device=w.device)
    moe_pack_int8(w, q8, s, stream)
    return q8, s


def pack_int4(w, stream=None):
    """Allocating convenience wrapper: w [O, I] fp32 (cuda) -> (q4, scale)."""
    O, I = w.shape
    q4 = torch.empty((O, (I + 1) // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty(O, dtype=torch.float32, device=w.device)
    moe_pack_int4(w, q4, s, stream)
    return q4, s


class MoeLayer:
    """Owns a library handle; borrows (and keeps alive) the weight tensors.

    experts: list of E + n_shared tuples (gate_q, gate_s, up_q, up_s, down_q, down_s)
    of CUDA tensors as moe_pack_int4 (weight_bits 4) or moe_pack_int8
    (weight_bits 8) writes them; entry E is the shared expert.
    """

    def __init__(self, D, I, E, K, n_shared, routed_scale, max_tokens, Wr, bias, experts, top_p=0.0,
                 weight_bits=4):
        self.D, self.I, self.E, self.K, self.n_shared = D, I, E, K, n_shared
        self.S = K + n_shared
        self.max_tokens = max_tokens
        self.top_p = float(top_p)
        self._keep = (Wr, bias, list(experts))
        self.weight_bits = int(weight_bits)
        desc = MoeLayerDesc(D, I, E, K, n_shared, float(routed_scale), max_tokens, self.top_p, self.weight_bits)
        arr = (MoeExpertW * (E + n_shared))()
        for e, (gq, gs, uq, us, dq, ds) in enumerate(experts):
            arr[e] = MoeExpertW(_ptr(gq), _ptr(uq), _ptr(dq), _ptr(gs), _ptr(us), _ptr(ds))
        h = ctypes.c_void_p()
        _check(_lib.moe_layer_create(ctypes.byref(desc), _ptr(Wr), _ptr(bias), arr, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            _check(_lib.moe_layer_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def moe_layer_forward(self, x, out, stream=None):
        _check(_lib.moe_layer_forward(self.handle, _ptr(x), x.shape[0], _ptr(out), _stream(stream)))

    def forward(self, x, stream=None):
        out = torch.empty_like(x)
        self.moe_layer_forward(x, out, stream)
        return out

    def forward_host(self, x_host, out_host, stream=None):
        """moe_layer_forward_host: x_host / out_host are CPU float32 tensors
        [n_tokens, D] (pinned memory keeps the copies asynchronous); the
        result is in out_host once the stream has been synchronised."""
        for name, t in (("x_host", x_host), ("out_host", out_host)):
            if t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.dim() != 2 or \
                    t.shape[1] != self.D:
                raise ValueError(f"{name} must be a contiguous CPU float32 tensor [n_tokens, {self.D}]")
        if out_host.shape[0] != x_host.shape[0]:
            raise ValueError("x_host and out_host must have the same number of rows")
        _check(_lib.moe_layer_forward_host(self.handle, ctypes.c_void_p(x_host.data_ptr()), x_host.shape[0],
                                           ctypes.c_void_p(out_host.data_ptr()), _stream(stream)))

    def moe_block_forward(self, x_inout, norm_w, eps, stream=None):
        _check(_lib.moe_block_forward(self.handle, _ptr(x_inout), _ptr(norm_w), float(eps), x_inout.shape[0],
                                      _stream(stream)))

    def moe_layer_debug(self, x, out=None, stream=None, **want):
        """Runs a forward and returns the requested intermediates as tensors.
        want: any of idx, w, xq, sx, gate_acc, up_acc, hq, sh, down_acc, union (True to request)."""
        T, dev = x.shape[0], x.device
        S = self.S
        shapes = dict(idx=((T, self.K), torch.int32), w=((T, self.K), torch.float32),
                      xq=((T, self.D), torch.int8), sx=((T,), torch.float32),
                      gate_acc=((T, S, self.I), torch.int32), up_acc=((T, S, self.I), torch.int32),
                      hq=((T, S, self.I), torch.int8), sh=((T, S), torch.float32),
                      down_acc=((T, S, self.D), torch.int32))
        res = {}
        for k, (shp, dt) in shapes.items():
            if want.get(k):
                res[k] = torch.full(shp, -1, dtype=dt, device=dev) if dt != torch.float32 else \
                    torch.full(shp, float("nan"), dtype=dt, device=dev)
        if want.get("union"):
            res["union_experts"] = torch.full((self.E + 1,), -1, dtype=torch.int32, device=dev)
            res["n_union"] = torch.zeros(1, dtype=torch.int32, device=dev)
        d = MoeDebugOut(*[_ptr(res.get(n)) for n, _ in MoeDebugOut._fields_])
        _check(_lib.moe_layer_debug(self.handle, _ptr(x), T, _ptr(out), ctypes.byref(d), _stream(stream)))
        return res

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int(0)
        rc = _lib.moe_layer_device_status(self.handle, _stream(stream), ctypes.byref(v))
        if rc not in (MOE_OK, MOE_ERR_DEVICE):
            _check(rc)
        return int(v.value)

    def set_option(self, option, value):
        _check(_lib.moe_layer_set_option(self.handle, int(option), int(value)))

    def get_option(self, option) -> int:
        v = ctypes.c_int(0)
        _check(_lib.moe_layer_get_option(self.handle, int(option), ctypes.byref(v)))
        return int(v.value)

    def set_trace(self, stamps=None):
        """stamps: int64 CUDA tensor (10 per CTA) for the decode kernel's phase
        stamps, or None to stop tracing."""
        if stamps is None:
            _check(_lib.moe_layer_set_trace(self.handle, None, 0))
        else:
            if stamps.dtype != torch.int64 or not stamps.is_cuda or not stamps.is_contiguous():
                raise ValueError("stamps must be a contiguous int64 CUDA tensor")
            _check(_lib.moe_layer_set_trace(self.handle, ctypes.c_void_p(stamps.data_ptr()), stamps.numel()))
        self._trace = stamps

    def set_probe(self, which, begin=None, end=None):
        for ev in (begin, end):  # torch creates the CUDA event at its first record
            if ev is not None and not ev.cuda_event:
                ev.record()
        _check(_lib.moe_layer_set_probe(self.handle, int(which),
                                        ctypes.c_void_p(begin.cuda_event if begin is not None else 0),
                                        ctypes.c_void_p(end.cuda_event if end is not None else 0)))


def workspace_bytes(D, I, E, K, n_shared, max_tokens, routed_scale=2.5) -> int:
    desc = MoeLayerDesc(D, I, E, K, n_shared, float(routed_scale), max_tokens, 0.0)
    n = ctypes.c_size_t(0)
    _check(_lib.moe_layer_workspace_bytes(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def expert_table_device(experts, device):
    """Device copy of a MoeExpertW array (entry E = shared expert) for
    moe_layer_forward_static; experts as for MoeLayer.  The entry point cannot
    inspect a device table, so the requirements moe_layer_create checks are
    checked here, on the host: no missing tensor, 16-byte aligned weights."""
    for e, ts in enumerate(experts):
        if len(ts) != 6 or any(t is None for t in ts):
            raise ValueError(f"expert {e}: need six tensors (gate_q, gate_s, up_q, up_s, down_q, down_s)")
        for name, t in (("gate_q", ts[0]), ("up_q", ts[2]), ("down_q", ts[4])):
            if t.data_ptr() % 16:
                raise ValueError(f"expert {e}: {name} must be 16-byte aligned")
    arr = (MoeExpertW * len(experts))()
    for e, (gq, gs, uq, us, dq, ds) in enumerate(experts):
        arr[e] = MoeExpertW(_ptr(gq), _ptr(uq), _ptr(dq), _ptr(gs), _ptr(us), _ptr(ds))
    return torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8).to(device)


def moe_layer_forward_static(D, I, E, K, n_shared, routed_scale, Wr, bias, experts_dev, x, out, stream=None,
                             top_p=0.0):
    """The allocation-free forward: experts_dev from expert_table_device."""
    desc = MoeLayerDesc(D, I, E, K, n_shared, float(routed_scale), max(1, x.shape[0]), float(top_p))
    _check(_lib.moe_layer_forward_static(ctypes.byref(desc), _ptr(Wr), _ptr(bias), _ptr(experts_dev), _ptr(x),
                                         x.shape[0], _ptr(out), _stream(stream)))


def static_status(stream=None) -> int:
    """Reads and clears the device-side flags that moe_layer_forward_static
    calls on the current device collected (0 when none)."""
    v = ctypes.c_int(0)
    rc = _lib.moe_layer_static_status(_stream(stream), ctypes.byref(v))
    if rc not in (MOE_OK, MOE_ERR_DEVICE):
        _check(rc)
    return int(v.value)
