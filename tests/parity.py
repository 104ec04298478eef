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


def router_logits_mt(orc, x_bits: np.ndarray, wr_bits: np.ndarray, rb) -> np.ndarray:
    """The oracle's router logits of many rows, the rows split over host
    threads (each thread one call of the oracle on a contiguous slice)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    T = x_bits.shape[0]
    n = max(1, min(os.cpu_count() or 1, (T + 63) // 64))
    cuts = np.linspace(0, T, n + 1).astype(int)
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda i: orc.router_logits(x_bits[cuts[i]:cuts[i + 1]], wr_bits, rb),
                            range(n)))
    return np.concatenate(parts, axis=0)


def enforce_gap(w: synth.Workload, x: torch.Tensor, router_w: torch.Tensor,
                router_bias, k: int, max_attempts: int = 20) -> np.ndarray:
    """Redraw rows of x (in place) until every token's 8th/9th logit gap in
    the oracle's fp64 logits is at least GAP_MIN. Returns the final gaps."""
    orc = oracle.get()
    wr = bits(router_w)
    rb = None if router_bias is None else router_bias.cpu().numpy()
    _, _, gap = orc.topk(router_logits_mt(orc, bits(x), wr, rb), k)
    for attempt in range(1, max_attempts + 1):
        bad = np.nonzero(gap < GAP_MIN)[0]
        if bad.size == 0:
            return gap
        synth.redraw_rows(w, x, bad.tolist(), attempt)
        _, _, gap[bad] = orc.topk(orc.router_logits(bits(x[torch.from_numpy(bad).to(x.device)]),
                                                    wr, rb), k)
    raise AssertionError("could not meet the logit-gap precondition")


class _DevArray:
    """Exposes a raw device address through __cuda_array_interface__."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 2}


def device_view(ptr: int, n: int, dtype) -> torch.Tensor:
    """Zero-copy torch view of n elements at a device address."""
    typestr = {torch.int32: "<i4", torch.float32: "<f4", torch.int16: "<i2"}[dtype]
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


def caller_routing_buffers(T: int, k: int, E: int):
    """Zeroed device buffers for every routing output (layouts of
    moe_routing) and the MoeRouting struct pointing at them."""
    from bit_grouped_gemm_gb300 import binding as bg
    max_tiles = (T * k + 127) // 128 + E
    z = lambda n, dt=torch.int32: torch.zeros(n, dtype=dt, device="cuda")
    bufs = dict(topk_idx=z(T * k), topk_w=z(T * k, torch.float32), counts=z(E),
                offsets=z(E + 1), tile_offsets=z(E + 1), perm=z(T * k), inv=z(T * k),
                block_map=z(max_tiles * 3), num_tiles=z(4), logits=z(T * E, torch.float32))
    r = bg.MoeRouting(**{n: t.data_ptr() for n, t in bufs.items()})
    return bufs, r


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits; normal range)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def layer_output_from_scratch(plan: int, inv: np.ndarray, rows: np.ndarray, T: int, k: int,
                              H: int, has_shared: bool) -> np.ndarray:
    """The block output y of the plan's last layer call for the given token
    rows, rebuilt from the plan's scratch exactly as the combine adds it: the
    shared expert's FP32 row, then the k weighted bf16 routed rows in slot
    order, each addition rounded to FP32 (the fused combine never stores y)."""
    from bit_grouped_gemm_gb300 import binding as bg
    d = device_view(bg.moe_debug_buffer(plan, 2), T * k * H, torch.int16).view(T * k, H)
    pos = torch.from_numpy(inv.reshape(T, k)[rows].astype(np.int64)).cuda()
    dr = d[pos.reshape(-1)].cpu().numpy().reshape(len(rows), k, H)
    dr = (dr.view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    if has_shared:
        dsh = device_view(bg.moe_debug_buffer(plan, 3), T * H, torch.float32).view(T, H)
        acc = dsh[torch.from_numpy(np.asarray(rows, np.int64)).cuda()].cpu().numpy().copy()
    else:
        acc = np.zeros((len(rows), H), np.float32)
    for j in range(k):
        acc = (acc + dr[:, j]).astype(np.float32)
    return acc
