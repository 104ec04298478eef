"""GPU parity of the stacked layers:
    xn = rmsnorm(x); y = moe(xn); x <- bf16(x + y/sqrt(L))

The full-size prefill stack (T=4096, 40 layers, Zipf routing, ~18 GB of packed
weights) runs on the GPU in the launch configuration the benchmark times. The
oracle follows a sample of tokens through all 40 layers on its own, in fp64,
from the generator's inputs; no oracle input ever comes from the GPU. At each
layer the GPU also runs the layer on a copy of its own batch in which the
sampled rows are replaced by the oracle's normalised inputs (same T, same
grid, the rest of the batch keeps the GPU's routing context). On those rows:
  * routing indices must equal the oracle's wherever the oracle's 8th/9th
    logit gap is >= 1e-3;
  * outputs must satisfy max|y_gpu - y_oracle| <= 2e-2 * rms(y_oracle) over
    the compared rows of the layer.
The GPU's own chain is checked at every layer for the invariants any correct
routing map has.

The decode stack (T = 8, 40 layers) is checked the same way on all 8 rows.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from bit_grouped_gemm_gb300 import binding as bg
from bit_grouped_gemm_gb300 import stack, synth
from tests import parity
from tests.oracle_pins import check_route_invariants

pytestmark = pytest.mark.gpu
NTHREADS = os.cpu_count() or 4


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_grouped_gemm_gb300 import build
    build.build()
    bg.load_library()


def oracle_layer_for_rows(L: stack.DeviceLayer, xn_bits: np.ndarray, sh: synth.MoEShape):
    """Oracle on the given normalised rows of one layer, copying to the host
    only the experts the oracle's own routing selects (plus router and shared)."""
    orc = oracle.get()
    wr = parity.bits(L.router_w)
    rb = None if L.router_bias is None else L.router_bias.cpu().numpy()
    logits = orc.router_logits(xn_bits, wr, rb)
    idx, _, _ = orc.topk(logits, sh.top_k)
    need = sorted(set(idx.reshape(-1).tolist()))
    routed = {}
    for m, (q, s, b) in L.routed.items():
        qh = np.zeros(tuple(q.shape), np.uint32)
        shh = np.zeros(tuple(s.shape), np.uint16)
        bh = np.zeros(tuple(b.shape), np.uint16)
        for e in need:
            qh[e] = parity.words(q[e])
            shh[e] = parity.bits(s[e])
            bh[e] = parity.bits(b[e])
        routed[m] = (qh, shh, bh)
    shared = parity.host_set(L.shared) if L.shared is not None else None
    return orc.moe_rows(xn_bits, wr, rb, routed, shared, sh.top_k, sh.group_size,
                        nthreads=NTHREADS)


def to_dev_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(b.view(np.int16).copy()).cuda().view(torch.bfloat16)


def run_chain_check(w: synth.Workload, rows: np.ndarray):
    sh = w.shape
    T = w.tokens
    layers = stack.make_layers(w, "cuda")
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    alpha = stack.residual_alpha(w.layers)
    orc = oracle.get()
    stats = []
    try:
        x = synth.tokens_x(w, "cuda")
        xn = torch.empty_like(x)
        y = torch.empty(x.shape, dtype=torch.float32, device="cuda")
        y_chk = torch.empty_like(y)
        xo = parity.bits(x)[rows]                    # oracle's own chain
        bg.moe_residual_add(plan, x, None, T, 0.0, x, xn)
        rows_t = torch.from_numpy(rows.astype(np.int64)).cuda()
        for li, L in enumerate(layers):
            # the GPU chain
            r = bg.moe_route(plan, xn, T, L.router_w, L.router_bias)
            g = parity.routing_to_numpy(r, T, sh.top_k, sh.num_experts)
            check_route_invariants(g, g["topk_idx"], sh.num_experts, 128)
            bg.moe_forward_layer(plan, xn, T, L.router_w, L.router_bias, L.routed_c,
                                 L.shared_c, y)
            # the same layer on the oracle's inputs for the sampled rows
            xon = orc.rmsnorm(xo)
            xin = xn.clone()
            xin[rows_t] = to_dev_bits(xon)
            rc = bg.moe_route(plan, xin, T, L.router_w, L.router_bias)
            gidx = parity.routing_to_numpy(rc, T, sh.top_k, sh.num_experts)["topk_idx"][rows]
            bg.moe_forward_layer(plan, xin, T, L.router_w, L.router_bias, L.routed_c,
                                 L.shared_c, y_chk)
            o = oracle_layer_for_rows(L, xon, sh)
            ok = o["gap"] >= parity.GAP_MIN
            assert np.array_equal(gidx[ok], o["topk_idx"][ok]), li
            yg = y_chk.double().cpu().numpy()[rows]
            ratio = parity.check_y(yg[ok], o["y"][ok])
            stats.append((li, int(ok.sum()), ratio))
            # advance both chains
            bg.moe_residual_add(plan, x, y, T, alpha, x, xn)
            xo = orc.residual(xo, o["y"], alpha)
        assert bg.moe_get_error(plan) == 0
        assert np.isfinite(x.float().cpu().numpy()).all()
        return stats
    finally:
        bg.moe_plan_destroy(plan)


def test_prefill_stack_t4096_l40_sampled():
    w = synth.standard_workloads()["prefill_t4096_l40_zipf"]
    rows = np.array([0, 1, 777, 2048, 3333, 4095], np.int32)
    stats = run_chain_check(w, rows)
    assert sum(n for _, n, _ in stats) >= 0.9 * len(rows) * w.layers, stats


def test_decode_stack_t8_l40():
    w = synth.standard_workloads()["decode_t8_l40"]
    stats = run_chain_check(w, np.arange(8, dtype=np.int32))
    assert sum(n for _, n, _ in stats) >= 0.9 * 8 * w.layers, stats


@pytest.mark.gpu
@pytest.mark.parametrize("T", [8, 512])
def test_fused_layer_update_bit_identical(T):
    """moe_forward_layer_residual (combine and stack update in one pass, y never
    written) gives the same bits as moe_forward_layer + moe_residual_add, on
    the small-M path (T=8) and the tensor-core path (T=512), over 3 layers."""
    from bit_grouped_gemm_gb300 import stack
    w = dataclasses.replace(synth.standard_workloads()["prefill_t4096_l40_zipf"], tokens=T, layers=3)
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    try:
        x0 = synth.tokens_x(w, "cuda")
        y = torch.empty(x0.shape, dtype=torch.float32, device="cuda")
        outs = []
        for fused in (False, True):
            x, xn = x0.clone(), torch.empty_like(x0)
            stack.run_stack(plan, x, xn, layers, T, y, stack.residual_alpha(40), fused=fused)
            torch.cuda.synchronize()
            assert bg.moe_get_error(plan) == 0
            outs.append((x.view(torch.int16).cpu().numpy(), xn.view(torch.int16).cpu().numpy()))
        assert np.array_equal(outs[0][0], outs[1][0])
        assert np.array_equal(outs[0][1], outs[1][1])
        # argument errors of the fused call: x may alias neither the layer's
        # input nor xn_out (status 1 = MOE_ERR_INVALID_ARG)
        L = layers[0]
        for x_arg, xn_out in ((xn, x), (x, x)):
            with pytest.raises(bg.MoeError) as ei:
                bg.moe_forward_layer_residual(plan, xn, T, L.router_w, L.router_bias, L.routed_c,
                                              L.shared_c, 0.1, x_arg, xn_out)
            assert ei.value.status == 1
    finally:
        bg.moe_plan_destroy(plan)


def _stack_bits(plan, w, layers, T, driver, x0):
    x, xn = x0.clone(), torch.empty_like(x0)
    alpha = stack.residual_alpha(40)
    if driver:
        arr = bg.moe_layers(layers)
        bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
    else:
        y = torch.empty(x0.shape, dtype=torch.float32, device="cuda")
        stack.run_stack(plan, x, xn, layers, T, y, alpha, fused=True)
    torch.cuda.synchronize()
    assert bg.moe_get_error(plan) == 0
    return x.view(torch.int16).cpu().numpy()


def test_stack_driver_matches_layer_calls():
    """moe_forward_stack (the native layer loop) gives the bits of the
    per-layer calls, here for one chunk (T <= max_tokens), 3 layers."""
    T = 512
    w = dataclasses.replace(synth.standard_workloads()["prefill_t4096_l40_zipf"], tokens=T, layers=3)
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    try:
        x0 = synth.tokens_x(w, "cuda")
        a = _stack_bits(plan, w, layers, T, True, x0)
        b = _stack_bits(plan, w, layers, T, False, x0)
        assert np.array_equal(a, b)
        # argument errors: no layers, xn overlapping x (status 1)
        x, xn = x0.clone(), torch.empty_like(x0)
        arr = bg.moe_layers(layers)
        assert bg.load_library().moe_forward_stack(plan, x.data_ptr(), xn.data_ptr(), T, arr, 0,
                                                   0.1, None) == 1
        assert bg.load_library().moe_forward_stack(plan, x.data_ptr(), x[1:].data_ptr(), T, arr,
                                                   3, 0.1, None) == 1
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("chunk", [256, 224])
def test_chunked_prefill_matches_one_pass(chunk):
    """A 600-token prompt through 3 layers in chunks of `chunk` rows (the
    plan's capacity; ragged last chunk) gives the bits of one 600-token pass:
    the block treats every token on its own, and every chunk here takes the
    tensor-core path like the whole prompt."""
    T = 600
    w = dataclasses.replace(synth.standard_workloads()["prefill_t4096_l40_zipf"], tokens=T, layers=3)
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    mk = lambda m: bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                                   sh.group_size, int(sh.has_shared), m), 0)
    whole, chunked = mk(T), mk(chunk)
    try:
        x0 = synth.tokens_x(w, "cuda")
        a = _stack_bits(whole, w, layers, T, True, x0)
        b = _stack_bits(chunked, w, layers, T, True, x0)
        assert np.array_equal(a, b)
    finally:
        bg.moe_plan_destroy(whole)
        bg.moe_plan_destroy(chunked)
