"""Shared helpers of the GPU parity tests: device inputs from the seeded
generator, host copies for the oracle, the layer-0 gap precondition, and the
comparisons."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_grouped_gemm_gb300 import synth

GAP_MIN = 1e-3          # 8th/9th logit gap required for bit-exact routing
Y_TOL = 2e-2            # max|y_gpu - y_oracle| <= Y_TOL * rms(y_oracle)
W_TOL = 1e-5            # top-k weights, absolute


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns (on host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def words(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def bf16_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def host_set(dev_set: dict) -> dict:
    return {m: (words(q), bits(s), bits(b)) for m, (q, s, b) in dev_set.items()}


def enforce_gap(w: synth.Workload, x: torch.Tensor, router_w: torch.Tensor,
                router_bias, k: int, max_attempts: int = 20) -> np.ndarray:
    """Redraw rows of x (in place) until every token's 8th/9th logit gap in
    the oracle's fp64 logits is at least GAP_MIN. Returns the final gaps."""
    orc = oracle.get()
    wr = bits(router_w)
    rb = None if router_bias is None else router_bias.cpu().numpy()
    for attempt in range(1, max_attempts + 1):
        logits = orc.router_logits(bits(x), wr, rb)
        _, _, gap = orc.topk(logits, k)
        bad = np.nonzero(gap < GAP_MIN)[0]
        if bad.size == 0:
            return gap
        synth.redraw_rows(w, x, bad.tolist(), attempt)
    raise AssertionError("could not meet the logit-gap precondition")


class _DevArray:
    """Exposes a raw device address through __cuda_array_interface__."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 2}


def device_view(ptr: int, n: int, dtype) -> torch.Tensor:
    """Zero-copy torch view of n elements at a device address."""
    typestr = {torch.int32: "<i4", torch.float32: "<f4"}[dtype]
    return torch.as_tensor(_DevArray(ptr, n, typestr), device="cuda")


def routing_to_numpy(r, T: int, k: int, E: int) -> dict:
    """Copy a MoeRouting's device arrays to host numpy arrays."""
    torch.cuda.synchronize()

    def get(ptr, n, dtype=torch.int32):
        return device_view(ptr, n, dtype).cpu().numpy()

    nt = int(get(r.num_tiles, 1)[0])
    out = dict(
        topk_idx=get(r.topk_idx, T * k).reshape(T, k),
        topk_w=get(r.topk_w, T * k, torch.float32).reshape(T, k),
        counts=get(r.counts, E),
        offsets=get(r.offsets, E + 1),
        tile_offsets=get(r.tile_offsets, E + 1),
        perm=get(r.perm, T * k),
        inv=get(r.inv, T * k),
        block_map=get(r.block_map, nt * 3).reshape(nt, 3),
        num_tiles=nt,
    )
    if r.logits:
        out["logits"] = get(r.logits, T * E, torch.float32).reshape(T, E)
    return out


def check_y(y_gpu: np.ndarray, y_orc: np.ndarray, tol: float = Y_TOL):
    """max|gpu - oracle| <= tol * rms(oracle); returns the ratio."""
    rms = float(np.sqrt(np.mean(y_orc ** 2)))
    err = float(np.max(np.abs(y_gpu - y_orc)))
    ratio = err / rms
    assert ratio <= tol, f"max|dy| = {err:.3e}, rms(y) = {rms:.3e}, ratio {ratio:.3e} > {tol}"
    return ratio
