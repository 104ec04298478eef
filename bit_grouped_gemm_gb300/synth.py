"""Seeded synthetic inputs for the W4A16 mixture-of-experts block.

This module only draws numbers. It holds none of the block's arithmetic (no
routing, no dequantisation, no matrix products), so the CUDA path and the CPU
oracle can both consume what it produces without sharing any method code.

Generator
---------
Every tensor is a pure function of ``(seed, tag, layer, element index)``. A
64-bit key is derived from ``(seed, tag, layer)`` with the SplitMix64
finaliser, and element ``i`` of the stream is ``mix64(key + (i + 1) * GAMMA)``
(the SplitMix64 output function evaluated at counter ``i``; Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014). The
integer work runs in torch ``int64`` arithmetic (wrap-around multiply, masked
logical shifts), so it gives the same bits on any device.

Derived draws:

* uniform in [0, 1): top 53 bits of a stream word times 2**-53;
* standard normal: Box-Muller on two uniforms of the same stream
  (elements ``2i`` and ``2i+1``);
* bf16 values are ``bf16(float32(v))`` with round-to-nearest-even at both
  steps, as torch converts.

Workload recipe (shapes of the Qwen3.6-35B-A3B mixture-of-experts block the
pages describe: 256 routed experts scored per token, 8 selected, one shared
expert, 4-bit affine weights in groups of 64 with one bf16 scale and one bf16
bias per group; hidden 2048 and expert width 512 are this build's choice):

* ``x ~ N(0, 1)`` bf16 ``[T, H]``;
* router ``W ~ N(0, 0.02)`` bf16 ``[H, E]``;
* router bias: 0 for uniform routing; for skewed routing a random expert
  permutation ``pi`` is drawn (argsort of stream words) and
  ``b[e] = -s * ln(pi(e) + 1)`` with ``s = 1.1``, the log of the unnormalised
  Zipf(s) mass at the expert's rank;
* packed weights: one uniform 32-bit word per 8 weights (each nibble uniform
  in 0..15), ``scale ~ U[0.005, 0.02]`` bf16, ``bias = -8 * scale + N(0, 1e-3)``
  bf16 (computed from the bf16 scale).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# stream tags
TAG_X = 1
TAG_X_REDRAW = 2
TAG_X_POOL = 3
TAG_ROUTER_W = 10
TAG_ROUTER_PERM = 11
TAG_Q = 100      # + 10 * matrix + expert set
TAG_SCALE = 200
TAG_BIASN = 300

MATRICES = ("gate", "up", "down")
BASE_SEED = 20261202


def _s64(v: int) -> int:
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int, layer: int = 0) -> int:
    """64-bit key of the stream for ``(seed, tag, layer)``."""
    k = _mix64_int(seed + GAMMA)
    k = _mix64_int(k ^ ((tag * 0x100000001B3) & MASK64))
    return _mix64_int(k ^ ((layer * 0xC2B2AE3D27D4EB4F) & MASK64))


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = z ^ _lsr(z, 30)
    z = z * _s64(_M1)
    z = z ^ _lsr(z, 27)
    z = z * _s64(_M2)
    return z ^ _lsr(z, 31)


def stream_u64(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Stream words at counters ``idx`` (int64 tensor), as int64 bit patterns."""
    return _mix64(idx.to(torch.int64) * _s64(GAMMA) + _s64(key + GAMMA))


def _uniform(key: int, idx: torch.Tensor) -> torch.Tensor:
    return _lsr(stream_u64(key, idx), 11).to(torch.float64) * (2.0 ** -53)


def _normal(key: int, idx: torch.Tensor) -> torch.Tensor:
    idx = idx.to(torch.int64)
    u1 = 1.0 - _uniform(key, 2 * idx)          # (0, 1]
    u2 = _uniform(key, 2 * idx + 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def _to_bf16(v: torch.Tensor) -> torch.Tensor:
    return v.to(torch.float32).to(torch.bfloat16)


def _arange(n: int, device, start: int = 0) -> torch.Tensor:
    return torch.arange(start, start + n, dtype=torch.int64, device=device)


def normal_bf16(seed: int, tag: int, layer: int, shape, std: float = 1.0,
                device="cpu", offset: int = 0) -> torch.Tensor:
    n = math.prod(shape)
    v = _normal(stream_key(seed, tag, layer), _arange(n, device, offset))
    return _to_bf16(v * std).reshape(shape)


def uniform_words(seed: int, tag: int, layer: int, shape, device="cpu") -> torch.Tensor:
    """Uniform 32-bit words (int32 bit patterns) of the given shape."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.int32, device=device)
    key = stream_key(seed, tag, layer)
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        w = stream_u64(key, _arange(e - s, device, s)) & 0xFFFFFFFF
        out[s:e] = (w - ((w >= (1 << 31)).to(torch.int64) << 32)).to(torch.int32)
    return out.reshape(shape)


# --------------------------------------------------------------------------
# workload configuration


@dataclasses.dataclass(frozen=True)
class MoEShape:
    hidden: int = 2048
    inter: int = 512
    num_experts: int = 256
    top_k: int = 8
    group_size: int = 64
    has_shared: bool = True


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: ``tokens`` rows through ``layers`` layers."""
    name: str
    tokens: int
    layers: int = 1
    routing: str = "uniform"        # "uniform" | "zipf"
    zipf_s: float = 1.1
    seed: int = BASE_SEED
    shape: MoEShape = MoEShape()


def standard_workloads() -> Dict[str, Workload]:
    """The five synthetic workloads (decode is one entry per batch size)."""
    s = BASE_SEED
    return {
        "t128_uniform": Workload("t128_uniform", 128, 1, "uniform", seed=s + 0),
        "t512_zipf": Workload("t512_zipf", 512, 1, "zipf", seed=s + 1),
        "t2048_uniform": Workload("t2048_uniform", 2048, 1, "uniform", seed=s + 2),
        "t2048_zipf": Workload("t2048_zipf", 2048, 1, "zipf", seed=s + 2),
        "prefill_t4096_l40_zipf": Workload("prefill_t4096_l40_zipf", 4096, 40, "zipf", seed=s + 3),
        "decode_t1_l40": Workload("decode_t1_l40", 1, 40, "zipf", seed=s + 3),
        "decode_t4_l40": Workload("decode_t4_l40", 4, 40, "zipf", seed=s + 3),
        "decode_t8_l40": Workload("decode_t8_l40", 8, 40, "zipf", seed=s + 3),
    }


# --------------------------------------------------------------------------
# tensors


def tokens_x(w: Workload, device="cpu") -> torch.Tensor:
    """Layer-0 activations ``x`` bf16 ``[T, H]``."""
    H = w.shape.hidden
    return normal_bf16(w.seed, TAG_X, 0, (w.tokens, H), 1.0, device)


def redraw_rows(w: Workload, x: torch.Tensor, rows, attempt: int) -> None:
    """Replace ``x[rows]`` in place with fresh N(0,1) rows (attempt >= 1)."""
    H = x.shape[1]
    key = stream_key(w.seed, TAG_X_REDRAW, attempt)
    for r in rows:
        idx = _arange(H, x.device, (int(r) * H))
        x[int(r)] = _to_bf16(_normal(key, idx))


def decode_pool(w: Workload, batches: int, device="cpu") -> torch.Tensor:
    """A pool of fresh decode batches, bf16 ``[batches, T, H]``."""
    H = w.shape.hidden
    return normal_bf16(w.seed, TAG_X_POOL, 0, (batches, w.tokens, H), 1.0, device)


def router_weight(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    sh = w.shape
    return normal_bf16(w.seed, TAG_ROUTER_W, layer, (sh.hidden, sh.num_experts), 0.02, device)


def router_bias(w: Workload, layer: int, device="cpu") -> Optional[torch.Tensor]:
    """fp32 ``[E]`` logit bias, or ``None`` for uniform routing."""
    E = w.shape.num_experts
    if w.routing == "uniform":
        return None
    key = stream_key(w.seed, TAG_ROUTER_PERM, layer)
    words = stream_u64(key, _arange(E, device))
    order = torch.argsort(words, stable=True)          # expert at rank r
    rank = torch.empty_like(order)
    rank[order] = _arange(E, device)
    b = -w.zipf_s * torch.log(rank.to(torch.float64) + 1.0)
    return b.to(torch.float32)


def w4_matrix(w: Workload, layer: int, matrix: str, shared: bool, device="cpu"):
    """Packed 4-bit affine weights of one matrix for all experts of a set.

    Returns ``(qweight int32 [E, N, K/8], scales bf16 [E, N, K/G],
    biases bf16 [E, N, K/G])`` with ``E = 1`` for the shared expert. gate and
    up are ``N = inter, K = hidden``; down is ``N = hidden, K = inter``.
    """
    sh = w.shape
    m = MATRICES.index(matrix)
    E = 1 if shared else sh.num_experts
    N, K = (sh.inter, sh.hidden) if matrix in ("gate", "up") else (sh.hidden, sh.inter)
    G = sh.group_size
    sub = 10 * m + (1 if shared else 0)
    q = uniform_words(w.seed, TAG_Q + sub, layer, (E, N, K // 8), device)
    n_groups = E * N * (K // G)
    u = _uniform(stream_key(w.seed, TAG_SCALE + sub, layer), _arange(n_groups, device))
    s = _to_bf16(0.005 + 0.015 * u)
    noise = _normal(stream_key(w.seed, TAG_BIASN + sub, layer), _arange(n_groups, device))
    b = _to_bf16(-8.0 * s.to(torch.float64) + 1e-3 * noise)
    return q, s.reshape(E, N, K // G), b.reshape(E, N, K // G)


def layer_params(w: Workload, layer: int, device="cpu") -> dict:
    """All tensors of one layer: router, routed experts and shared expert."""
    p = {
        "router_w": router_weight(w, layer, device),
        "router_bias": router_bias(w, layer, device),
        "routed": {m: w4_matrix(w, layer, m, False, device) for m in MATRICES},
        "shared": ({m: w4_matrix(w, layer, m, True, device) for m in MATRICES}
                   if w.shape.has_shared else None),
    }
    return p


def packed_bytes_per_expert(shape: MoEShape) -> int:
    """Bytes of one expert's packed weights plus scales and biases."""
    n_w = 3 * shape.hidden * shape.inter
    return n_w // 2 + 2 * 2 * (n_w // shape.group_size)
