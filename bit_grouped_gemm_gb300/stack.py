"""Device-resident synthetic layers and the stacked-layer driver.

``make_layer`` materialises one layer's tensors (router, routed experts,
shared expert) on a device from the seeded generator in ``synth`` and keeps
the ``MoeExperts`` structs the C ABI takes. ``run_stack`` chains layers with
the residual update ``x <- bf16(x + alpha * moe(x))``, every step through the
C ABI.
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


def run_stack(plan: int, x: torch.Tensor, layers: List[DeviceLayer], T: int,
              y_buf: torch.Tensor, alpha: float, stream=None,
              y_per_layer: Optional[List[torch.Tensor]] = None,
              x_per_layer: Optional[List[torch.Tensor]] = None) -> torch.Tensor:
    """Run the layers in order on ``x`` (updated in place) and return it.

    When ``y_per_layer`` / ``x_per_layer`` are given, each layer's output and
    input are copied there (for parity checks)."""
    for i, L in enumerate(layers):
        if x_per_layer is not None:
            x_per_layer[i].copy_(x[:T])
        binding.moe_forward_layer(plan, x, T, L.router_w, L.router_bias, L.routed_c, L.shared_c,
                                  y_buf, stream)
        if y_per_layer is not None:
            y_per_layer[i].copy_(y_buf[:T])
        binding.moe_residual_add(plan, x, y_buf, T, alpha, x, stream)
    return x
