"""ctypes binding of ``libmoe_w4.so`` (include/moe_w4.h): argument marshalling
only. Every step of the block runs in the library's CUDA kernels; there is no
Python or CPU fallback, and a missing or unloadable library raises.

Functions keep the C names. Tensors are torch CUDA tensors (bf16 tensors are
passed by pointer as bit patterns; packed weights as int32/uint32 tensors).
``stream`` is a ``torch.cuda.Stream``, a raw handle (int) or ``None`` for
torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_w4.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_CUDA", 4: "MOE_ERR_CAPACITY", 5: "MOE_ERR_DEVICE_TIMEOUT",
                6: "MOE_ERR_OPERAND_RANGE"}
KERNEL_KINDS = ("router", "scan", "scatter", "gather", "gate_up_gemm", "down_gemm",
                "combine", "residual", "topk", "decode_layer")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class MoePlanDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int),
                ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("group_size", ctypes.c_int), ("has_shared", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("block_m", ctypes.c_int),
                ("gemm_path", ctypes.c_int), ("small_m_max_tokens", ctypes.c_int),
                ("wait_limit_ms", ctypes.c_int)]


class MoeW4(ctypes.Structure):
    _fields_ = [("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p)]


class MoeExperts(ctypes.Structure):
    _fields_ = [("gate", MoeW4), ("up", MoeW4), ("down", MoeW4)]


class MoeLayer(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("routed", MoeExperts), ("shared", MoeExperts)]


class MoeRouting(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "counts", "offsets", "tile_offsets", "perm", "inv",
                 "block_map", "num_tiles", "logits")]


class MoeTiming(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * len(KERNEL_KINDS)),
                ("launches", ctypes.c_longlong * len(KERNEL_KINDS))]


_lib = None


def load_library(path: Optional[str] = None):
    """Load (once) and bind the C-ABI library. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m bit_grouped_gemm_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sig = {
        "moe_plan_create": (S, [ctypes.POINTER(MoePlanDesc), I, ctypes.POINTER(P)]),
        "moe_plan_destroy": (S, [P]),
        "moe_plan_scratch_bytes": (S, [ctypes.POINTER(MoePlanDesc), ctypes.POINTER(ctypes.c_size_t)]),
        "moe_route": (S, [P, P, I, P, P, ctypes.POINTER(MoeRouting), P]),
        "moe_grouped_w4_ffn": (S, [P, P, I, ctypes.POINTER(MoeRouting), ctypes.POINTER(MoeExperts),
                                   ctypes.POINTER(MoeExperts), P, P]),
        "moe_forward_layer": (S, [P, P, I, P, P, ctypes.POINTER(MoeExperts),
                                  ctypes.POINTER(MoeExperts), P, P]),
        "moe_forward_layer_residual": (S, [P, P, I, P, P, ctypes.POINTER(MoeExperts),
                                           ctypes.POINTER(MoeExperts), ctypes.c_float, P, P, P]),
        "moe_residual_add": (S, [P, P, P, I, ctypes.c_float, P, P, P]),
        "moe_forward_stack": (S, [P, P, P, I, ctypes.POINTER(MoeLayer), I, ctypes.c_float, P]),
        "moe_get_error": (S, [P]),
        "moe_debug_wait_timeout": (S, [P, I, P]),
        "moe_enable_timing": (S, [P, I]),
        "moe_set_tail_split": (S, [P, I]),
        "moe_read_timing": (S, [P, ctypes.POINTER(MoeTiming)]),
        "moe_last_gemm_path": (I, [P]),
        "moe_debug_buffer": (P, [P, I]),
        "moe_route_noalloc": (S, [P, I, I, P, P, I, I, ctypes.POINTER(MoeRouting), P]),
        "moe_route_noalloc_get_error": (S, []),
        "moe_route_noalloc_debug_wait_timeout": (S, [I, P]),
        "moe_status_string": (ctypes.c_char_p, [S]),
        "moe_version": (I, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def plan_desc(hidden=2048, inter=512, num_experts=256, top_k=8, group_size=64, has_shared=1,
              max_tokens=4096, block_m=128, gemm_path=0, small_m_max_tokens=0,
              wait_limit_ms=0) -> MoePlanDesc:
    return MoePlanDesc(hidden, inter, num_experts, top_k, group_size, int(has_shared),
                       max_tokens, block_m, gemm_path, small_m_max_tokens, wait_limit_ms)


def moe_plan_scratch_bytes(desc: MoePlanDesc) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().moe_plan_scratch_bytes(ctypes.byref(desc), ctypes.byref(out)),
           "moe_plan_scratch_bytes")
    return out.value


def moe_plan_create(desc: MoePlanDesc, device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load_library().moe_plan_create(ctypes.byref(desc), device, ctypes.byref(h)),
           "moe_plan_create")
    return h.value


def moe_plan_destroy(plan: int) -> None:
    _check(load_library().moe_plan_destroy(plan), "moe_plan_destroy")


def experts(gate, up, down) -> MoeExperts:
    """``MoeExperts`` from three ``(qweight, scales, biases)`` tensor triples."""
    def w(m):
        return MoeW4(_ptr(m[0]), _ptr(m[1]), _ptr(m[2]))
    return MoeExperts(w(gate), w(up), w(down))


def moe_route(plan: int, x, T: int, router_w, router_bias=None, stream=None) -> MoeRouting:
    out = MoeRouting()
    _check(load_library().moe_route(plan, _ptr(x), T, _ptr(router_w), _ptr(router_bias),
                                    ctypes.byref(out), _stream(stream)), "moe_route")
    return out


def moe_grouped_w4_ffn(plan: int, x, T: int, routing: MoeRouting, routed: MoeExperts,
                       shared: Optional[MoeExperts], y, stream=None) -> None:
    _check(load_library().moe_grouped_w4_ffn(
        plan, _ptr(x), T, ctypes.byref(routing), ctypes.byref(routed),
        ctypes.byref(shared) if shared is not None else None, _ptr(y), _stream(stream)),
        "moe_grouped_w4_ffn")


def moe_forward_layer(plan: int, x, T: int, router_w, router_bias, routed: MoeExperts,
                      shared: Optional[MoeExperts], y, stream=None) -> None:
    _check(load_library().moe_forward_layer(
        plan, _ptr(x), T, _ptr(router_w), _ptr(router_bias), ctypes.byref(routed),
        ctypes.byref(shared) if shared is not None else None, _ptr(y), _stream(stream)),
        "moe_forward_layer")


def moe_forward_layer_residual(plan: int, xn, T: int, router_w, router_bias, routed: MoeExperts,
                               shared: Optional[MoeExperts], alpha: float, x, xn_out,
                               stream=None) -> None:
    _check(load_library().moe_forward_layer_residual(
        plan, _ptr(xn), T, _ptr(router_w), _ptr(router_bias), ctypes.byref(routed),
        ctypes.byref(shared) if shared is not None else None, float(alpha), _ptr(x),
        _ptr(xn_out), _stream(stream)), "moe_forward_layer_residual")


def moe_layers(layers) -> ctypes.Array:
    """A ctypes array of MoeLayer from objects with router_w, router_bias,
    routed_c and shared_c (the tensors must outlive its use)."""
    arr = (MoeLayer * len(layers))()
    for i, L in enumerate(layers):
        arr[i].router_w = _ptr(L.router_w)
        arr[i].router_bias = _ptr(L.router_bias)
        arr[i].routed = L.routed_c
        if L.shared_c is not None:
            arr[i].shared = L.shared_c
    return arr


def moe_forward_stack(plan: int, x, xn, T: int, layers: ctypes.Array, alpha: float,
                      stream=None) -> None:
    _check(load_library().moe_forward_stack(plan, _ptr(x), _ptr(xn), T, layers, len(layers),
                                            float(alpha), _stream(stream)), "moe_forward_stack")


def moe_route_noalloc(x, T: int, hidden: int, router_w, router_bias, num_experts: int,
                      top_k: int, out: MoeRouting, stream=None) -> None:
    """Routing into caller-owned buffers with no device allocation (see header)."""
    _check(load_library().moe_route_noalloc(_ptr(x), T, hidden, _ptr(router_w),
                                            _ptr(router_bias), num_experts, top_k,
                                            ctypes.byref(out), _stream(stream)),
           "moe_route_noalloc")


def moe_route_noalloc_get_error() -> int:
    """Status of moe_route_noalloc's device error word on the current device
    (read and cleared; synchronises the device)."""
    return load_library().moe_route_noalloc_get_error()


def moe_route_noalloc_debug_wait_timeout(limit_us: int, stream=None) -> None:
    _check(load_library().moe_route_noalloc_debug_wait_timeout(int(limit_us), _stream(stream)),
           "moe_route_noalloc_debug_wait_timeout")


def moe_residual_add(plan: int, x, y, T: int, alpha: float, x_out=None, xn_out=None,
                     stream=None) -> None:
    _check(load_library().moe_residual_add(plan, _ptr(x), _ptr(y), T, float(alpha), _ptr(x_out),
                                           _ptr(xn_out), _stream(stream)), "moe_residual_add")


def moe_get_error(plan: int) -> int:
    """Status code of the plan's device error word (read and cleared)."""
    return load_library().moe_get_error(plan)


def moe_debug_wait_timeout(plan: int, limit_us: int, stream=None) -> None:
    _check(load_library().moe_debug_wait_timeout(plan, int(limit_us), _stream(stream)),
           "moe_debug_wait_timeout")


def moe_enable_timing(plan: int, on: bool) -> None:
    _check(load_library().moe_enable_timing(plan, int(bool(on))), "moe_enable_timing")


def moe_read_timing(plan: int) -> dict:
    t = MoeTiming()
    _check(load_library().moe_read_timing(plan, ctypes.byref(t)), "moe_read_timing")
    return {k: (t.ms[i], int(t.launches[i])) for i, k in enumerate(KERNEL_KINDS)}


def moe_set_tail_split(plan: int, on: bool) -> None:
    _check(load_library().moe_set_tail_split(plan, int(bool(on))), "moe_set_tail_split")


def moe_last_gemm_path(plan: int) -> int:
    return load_library().moe_last_gemm_path(plan)


def moe_debug_buffer(plan: int, which: int) -> int:
    """Device address of plan scratch: 0 gathered x, 1 SwiGLU act, 2 expert outputs."""
    return load_library().moe_debug_buffer(plan, which) or 0


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_version() -> int:
    return load_library().moe_version()
