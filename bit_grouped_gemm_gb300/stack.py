"""Device-resident synthetic layers and the stacked-layer driver.

``make_layer`` materialises one layer's tensors (router, routed experts,
shared expert) on a device from the seeded generator in ``synth`` and keeps
the ``MoeExperts`` structs the C ABI takes. ``run_stack`` chains layers with
the residual update ``x <- bf16(x + alpha * moe(rmsnorm(x)))``, every step
through the C ABI.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

from . import binding, synth


@dataclasses.dataclass
class DeviceLayer:
    router_w: torch.Tensor
    router_bias: Optional[torch.Tensor]
    routed: dict            # name -> (q, s, b)
    shared: Optional[dict]
    routed_c: binding.MoeExperts = None
    shared_c: Optional[binding.MoeExperts] = None

    def __post_init__(self):
        r = self.routed
        self.routed_c = binding.experts(r["gate"], r["up"], r["down"])
        if self.shared is not None:
            s = self.shared
            self.shared_c = binding.experts(s["gate"], s["up"], s["down"])

    def nbytes(self) -> int:
        n = self.router_w.numel() * 2
        for d in (self.routed, self.shared or {}):
            for m in d.values():
                n += sum(t.numel() * t.element_size() for t in m)
        return n


def make_layer(w: synth.Workload, layer: int, device="cuda") -> DeviceLayer:
    p = synth.layer_params(w, layer, device)
    return DeviceLayer(p["router_w"], p["router_bias"], p["routed"], p["shared"])


def make_layers(w: synth.Workload, device="cuda") -> List[DeviceLayer]:
    return [make_layer(w, l, device) for l in range(w.layers)]


def residual_alpha(num_layers: int) -> float:
    """Scale of each layer's output in the residual stream (1/sqrt(L))."""
    return 1.0 / math.sqrt(num_layers)


def run_stack(plan: int, x: torch.Tensor, xn: torch.Tensor, layers: List[DeviceLayer], T: int,
              y_buf: torch.Tensor, alpha: float, stream=None, fused: bool = True) -> torch.Tensor:
    """Run the layers in order on the residual stream ``x`` (bf16, updated in
    place) and return it. Every layer sees the RMS-normalised stream ``xn``
    (bf16 scratch of x's shape); ``y_buf`` is the fp32 [T, H] layer output
    (written only when ``fused`` is False).

        xn = rmsnorm(x)
        for each layer: y = moe(xn); x = bf16(x + alpha * y); xn = rmsnorm(x)

    ``fused`` takes each layer and its update in one call
    (moe_forward_layer_residual, y never written); otherwise
    moe_forward_layer then moe_residual_add. Both give identical bits.
    """
    binding.moe_residual_add(plan, x, None, T, 0.0, x, xn, stream)
    for L in layers:
        if fused:
            binding.moe_forward_layer_residual(plan, xn, T, L.router_w, L.router_bias,
                                               L.routed_c, L.shared_c, alpha, x, xn, stream)
        else:
            binding.moe_forward_layer(plan, xn, T, L.router_w, L.router_bias, L.routed_c,
                                      L.shared_c, y_buf, stream)
            binding.moe_residual_add(plan, x, y_buf, T, alpha, x, xn, stream)
    return x
